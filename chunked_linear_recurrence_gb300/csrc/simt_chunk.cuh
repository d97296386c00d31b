// simt_chunk.cuh -- parameters and launchers of the FP32 CUDA-core chunk kernels.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace sfg {

enum { MODE_FWD = 0, MODE_SUMMARY = 1, MODE_REPLAY = 2 };

// One parameter block for every chain kernel; unused members are NULL.
struct ChainParams {
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  const float* beta;
  const float* s0;        // [N,H,V,K] or NULL
  const int32_t* cu;      // [N+1] or NULL
  const int32_t* bounds;  // [R,2] (summary)
  void* out;              // [B,T,H,V]
  float* final_state;     // [N,H,V,K] or NULL
  float* P;               // [R,H,K,K] (summary)
  float* E;               // [R,H,V,K] (summary)
  float* ckpt;            // [slots,H] chunk-entry states (replay / backward): FP32 [V,K], or
                          // for BF16 with K = V = 128 BF16 swizzled [128][128] tiles (32 KB)
  float* tape;            // [slots,H] chunk-exit cotangents (backward), laid out as ckpt
  const void* dout;       // [B,T,H,V] (backward)
  const float* dsf;       // [N,H,V,K] or NULL (backward)
  void* dq;
  void* dk;
  void* dv;
  float* dg;
  float* dbeta;
  float* ds0;             // [N,H,V,K] or NULL
  float* fac;             // [slots,H] per-chunk backward factors (BF16 backward)
  int fac_ready;          // BF16, K = 128: the state replay has written the chunk records to
                          // fac (chunk_record.cuh), so the factor kernel is not run
  // paged state cache (forward): sequence n starts from pool[state_idx[n]] (zeros when
  // has_init[n] == 0) and leaves its final state there; state_idx[n] <= 0 marks padding:
  // zero output, the pool untouched.  p.s0 / p.final_state are then unused.
  float* pool;            // [num_slots,H,V,K] or NULL
  const int32_t* state_idx;
  const uint8_t* has_init;  // or NULL (every slot is loaded)
  int num_slots;          // slot indices >= num_slots are treated as padding as well
  int dqk_f32;            // backward: dq, dk are FP32 [B,T,H,K] per value head (grouped
                          // heads, summed into the caller's tensors afterwards)
  int B, T, H, N;
  int HK;                 // query/key heads (divides H): value head h reads h / (H / HK)
  float scale;
  int* status;            // the workspace's status words (kernels with bounded waits), or NULL
  uint32_t* sync;         // BF16, K = 128, dense: scratch of N*H + 1 128-byte lines (the
                          // reverse chain's written-tile counts and a work counter when it
                          // runs beside the gradients), or NULL
};

// Query/key head of value head h.
__host__ __device__ inline int qk_head(int h, int H, int HK) { return h / (H / HK); }

// CTAs along the slot axis of the per-chunk backward kernels (which walk slots with a
// grid stride and stop at the first empty one): one per slot for dense inputs, where every
// slot holds a chunk; for packed inputs, whose offsets may end long before T, about eight
// waves of (slot, head) CTAs at most, so that empty slots cost no launches.
inline int64_t slot_grid(const ChainParams& p, int64_t slots) {
  if (!p.cu) return slots;
  int dev = 0, nsm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || nsm < 1)
    nsm = 1;
  const int64_t cap = (8LL * nsm + p.H - 1) / p.H;
  return slots < cap ? slots : cap;
}

// Forward / summary / replay chain kernel: `items` = N (fwd, replay) or R (summary).
cudaError_t launch_simt_chain(const ChainParams& p, int mode, bool bf16, int D, int items,
                              cudaStream_t st);
// Backward after a replay: reverse cotangent chain then per-chunk token gradients.
// chain_only: only the reverse cotangent chain (and, for BF16, its per-chunk factors) --
// the segments' cotangent maps need p.ds0 alone, no state replay and no token gradients.
cudaError_t launch_simt_bwd(const ChainParams& p, bool bf16, int D, int64_t slots,
                            cudaStream_t st, bool chain_only = false);
// Grouped heads: out[r, hk, c] = sum over j < H / HK of acc[r, hk (H / HK) + j, c] for the
// active rows r (r < cu[N] when cu != NULL, else all B*T), in the q/k/v dtype.
cudaError_t launch_group_sum(const float* acc, void* out, bool bf16, int64_t rows, int H, int HK,
                             int D, const int32_t* cu, int N, cudaStream_t st);
// BF16 backward's reverse cotangent chain on the warp-level tensor cores
// (bwd_chain_mma.cu): per-chunk factors into p.fac, then the chain (tape, ds0).
size_t mma_bwd_fac_bytes(int D);
cudaError_t launch_mma_bwd_chain(const ChainParams& p, float* fac, int D, int64_t slots,
                                 cudaStream_t st);
// Per-chunk token gradients on the warp-level tensor cores (bwd_grad_mma.cu): BF16 or FP32
// inputs with head size 64, FP32 [V,K] checkpoints and tape.
cudaError_t launch_mma_bwd_grad(const ChainParams& p, bool bf16, int D, int64_t slots,
                                cudaStream_t st);
// Per-chunk token gradients on tcgen05 (bwd_grad_tc.cu): BF16, K = V = 128, checkpoints and
// tape as BF16 swizzled tiles.
cudaError_t launch_tc_bwd_grad(const ChainParams& p, int64_t slots, cudaStream_t st);
// Whether the reverse chain can run in the gradients' launch (dense inputs, p.sync set, at
// most 64 chains and at least 32 SMs left for the gradients), and that launch: the chain
// over the chunk records `fac` (with Qg) on CTAs [0, N*H), the gradients on the rest, each
// chunk-head taken once its exit cotangent is written.
bool tc_bwd_fusable(const ChainParams& p);
cudaError_t launch_tc_bwd_fused(const ChainParams& p, const float* fac, cudaStream_t st);

}  // namespace sfg
