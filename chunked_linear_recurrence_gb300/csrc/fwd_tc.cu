// fwd_tc.cu -- tensor-core forward of the chunked gated delta rule for BF16
// q/k/v with K = V = 128 on sm_103a: TMA tile loads, tcgen05.mma with FP32
// accumulators in TMEM, the FP32 state carried in TMEM across chunks.
//
// One CTA per (sequence, head) chain walks its 64-token chunks in order
// (StateFlow section 2.2, Eq. 2: Pre -> ST -> Out per chunk; section 3.1,
// Eq. 4-5: the chunk's output state is the next chunk's input state).  Every
// product is arranged so that its M dimension is 128 (the full TMEM lane
// count): the state-side products run "transposed", with the value index v
// (or the key index k) on the M axis and the 64 chunk tokens on N:
//
//   KQ   = [K; Q] K^T                       M=128 (64 key rows, 64 query rows), N=64, K=128
//   W^T  = K^T T''^T,  T'' = T diag(beta e^gamma)                   M=128, N=64, K=64
//   U^T  = V^T T'^T,   T'  = T diag(beta)     (into the Delta^T accumulator)
//   Delta^T += -S W^T                                              M=128, N=64, K=128
//   SQ   = S Q^T                                                   M=128, N=64, K=128
//   S   <- e^{gamma_C} S + (Delta^T diag(dec)) K                   M=128, N=128, K=64
//   OA   = Delta^T Ahat^T,  Ahat = M o Gamma o Q K^T               M=128, N=64, K=64
//   out[i][v] = scale (e^{gamma_i} SQ[v][i] + OA[v][i])
//
// The 64x64 triangular solve T = (I + A)^{-1} runs on the CUDA cores in FP32
// (hierarchical 16x16 blocks); its BF16 copies T', T'' are tensor-core
// operands, as are the BF16 copies of the state, W and Delta (the state itself
// stays FP32 in TMEM; the pages stage chunk-entry states in the Q/K/V dtype in
// the same way).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "fwd_tc.cuh"
#include "solve_tc.cuh"
#include "tc_ptx.cuh"

namespace sfg {
namespace {

using namespace tc;

constexpr int D = 128;
constexpr int NTHR = 256;

// Shared-memory map (bytes from a 1024-aligned base).  Panel layout, see tc_ptx.cuh.
constexpr uint32_t OFF_KQ = 0;          // 2 stages x 32 KB; a stage is 2 panels x 16 KB:
constexpr uint32_t KQ_STAGE = 32768;    //   rows 0-63 K, rows 64-127 Q of one chunk
constexpr uint32_t KQ_PANEL = 16384;
constexpr uint32_t OFF_V = 65536;       // 2 panels x 8 KB: V [64 tokens][128]
constexpr uint32_t V_PANEL = 8192;
constexpr uint32_t OFF_S = 81920;       // 2 panels x 16 KB: S (BF16) [128 v][128 k]
constexpr uint32_t S_PANEL = 16384;
constexpr uint32_t OFF_WT = 114688;     // 16 KB: W^T [128 k][64 i]
constexpr uint32_t OFF_DT = 131072;     // 16 KB: Delta^T [128 v][64 j]; solve scratch before
constexpr uint32_t OFF_DDT = 147456;    // 16 KB: (Delta^T diag(dec)) [128 v][64 j]
constexpr uint32_t OFF_T1 = 163840;     // 8 KB: T'  [64 i][64 j]   } output staging
constexpr uint32_t OFF_T2 = 172032;     // 8 KB: T'' [64 i][64 j]   } [64][128] BF16 after
constexpr uint32_t OFF_AH = 180224;     // 8 KB: Ahat [64 i][64 j]
constexpr uint32_t OFF_A32 = 188416;    // FP32 A [64][SOLVE_LD]
constexpr uint32_t OFF_T32 = 205824;    // FP32 T [64][SOLVE_LD]
constexpr uint32_t OFF_VEC = 223232;    // FP32 vectors: g, beta, gamma, e^gamma, dec, e^+, e^- (7 x 64)
constexpr uint32_t OFF_BAR = 225024;    // mbarriers + TMEM address
constexpr uint32_t SMEM_USED = OFF_BAR + 64;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;   // slack to align the base to 1024
static_assert(OFF_A32 + 64 * SOLVE_LD * 4 <= OFF_T32, "A32");
static_assert(OFF_T32 + 64 * SOLVE_LD * 4 <= OFF_VEC, "T32");
static_assert(32 * SOLVE_LD * 4 <= 16384, "solve scratch fits the Delta^T tile");

// TMEM columns (FP32 accumulators, 128 lanes each).
constexpr uint32_t TM_S = 0;      // S [v][k]        128 cols
constexpr uint32_t TM_KQ = 128;   // [K;Q] K^T       64 cols
constexpr uint32_t TM_WT = 192;   // W^T [k][i]      64 cols
constexpr uint32_t TM_DT = 256;   // U^T / Delta^T   64 cols
constexpr uint32_t TM_SQ = 320;   // S Q^T [v][i]    64 cols
constexpr uint32_t TM_OA = 384;   // Delta^T Ahat^T  64 cols
constexpr uint32_t TM_COLS = 512;

constexpr uint32_t ID_KQ = idesc_bf16(128, 64, false, false);
constexpr uint32_t ID_WT = idesc_bf16(128, 64, true, false);        // A = K^T (MN-major)
constexpr uint32_t ID_DT = idesc_bf16(128, 64, false, true, true);  // A = -S, B = W^T (MN-major)
constexpr uint32_t ID_SQ = idesc_bf16(128, 64, false, false);
constexpr uint32_t ID_SU = idesc_bf16(128, 128, false, true);       // B = K (MN-major)
constexpr uint32_t ID_OA = idesc_bf16(128, 64, false, false);

struct TcParams {
  const float* g;
  const float* beta;
  const float* s0;
  const int32_t* cu;
  __nv_bfloat16* out;
  float* final_state;
  int* status;
  int B, T, H, N;
  float scale;
};

struct CtaBar {
  __device__ __forceinline__ void operator()() const { __syncthreads(); }
};

// All threads agree on the outcome of a bounded wait.
__device__ __forceinline__ bool cta_wait(uint64_t* bar, uint32_t parity, int* status) {
  const bool ok = mbar_wait(bar, parity);
  const bool all = __syncthreads_and(ok) != 0;
  if (!all && threadIdx.x == 0) atomicExch(status, 5 /* SF_ERR_TIMEOUT */);
  return all;
}

__global__ void __launch_bounds__(NTHR, 1)
    gdn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(sm);
  float* sA = reinterpret_cast<float*>(sm + OFF_A32);
  float* sT = reinterpret_cast<float*>(sm + OFF_T32);
  float* sX = reinterpret_cast<float*>(sm + OFF_DT);       // solve scratch (Delta^T tile is free then)
  float* sg = reinterpret_cast<float*>(sm + OFF_VEC);
  float* sbeta = sg + 64;
  float* sgam = sbeta + 64;
  float* seg = sgam + 64;      // e^{gamma_i}
  float* sdec = seg + 64;      // e^{gamma_C - gamma_i}
  float* sep = sdec + 64;      // e^{gamma_i - mid}   (factorised decay, see below)
  float* sem = sep + 64;       // e^{mid - gamma_j}
  uint64_t* bar_kq = reinterpret_cast<uint64_t*>(sm + OFF_BAR);   // [2] K/Q stage loaded
  uint64_t* bar_v = bar_kq + 2;                                    // V loaded
  uint64_t* bar_mma = bar_kq + 3;                                  // MMA batch done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_kq + 4);
  int* flag = reinterpret_cast<int*>(tmem_slot + 1);               // per-chunk decay path

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = p.H;
  const int n = blockIdx.x / H, h = blockIdx.x % H;
  const int q4 = warp & 3;                 // TMEM lane quarter of this warp
  const int half = warp >> 2;              // which half of the columns this warp handles
  const int row = q4 * 32 + lane;          // accumulator row (TMEM lane) of this thread
  const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;

  int64_t bos, eos;
  seq_span(n, p.B, p.T, p.cu, bos, eos);
  const int nchunks = (int)((eos - bos + CHUNK - 1) / CHUNK);
  const size_t state_off = ((size_t)n * H + h) * D * D;

  if (tid == 0) {
    mbar_init(bar_kq, 1);
    mbar_init(bar_kq + 1, 1);
    mbar_init(bar_v, 1);
    mbar_init(bar_mma, 1);
    fence_mbar_init();
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    if (nchunks > 0) {        // prologue: chunk 0's K, Q and V
      mbar_arrive_expect_tx(bar_kq, 4 * 8192);
      mbar_arrive_expect_tx(bar_v, 2 * 8192);
#pragma unroll
      for (int pnl = 0; pnl < 2; ++pnl) {
        tma_load_3d(sm + OFF_KQ + pnl * KQ_PANEL, &tmK, bar_kq, 64 * pnl, h, (int)bos);
        tma_load_3d(sm + OFF_KQ + pnl * KQ_PANEL + 8192, &tmQ, bar_kq, 64 * pnl, h, (int)bos);
        tma_load_3d(sm + OFF_V + pnl * V_PANEL, &tmV, bar_v, 64 * pnl, h, (int)bos);
      }
    }
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tmem_slot;
  const uint32_t tl = tm + lane_off;       // this warp's lane base

  // initial state -> TMEM (FP32) and the BF16 operand copy
#pragma unroll
  for (int cc = 0; cc < 2; ++cc) {
    const int c0 = 64 * half + 32 * cc;
    float x[32];
    if (p.s0) {
      const float4* src = reinterpret_cast<const float4*>(p.s0 + state_off + (size_t)row * D + c0);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float4 t = src[e];
        x[4 * e] = t.x; x[4 * e + 1] = t.y; x[4 * e + 2] = t.z; x[4 * e + 3] = t.w;
      }
    } else {
#pragma unroll
      for (int e = 0; e < 32; ++e) x[e] = 0.f;
    }
    tmem_st32(tl + TM_S + c0, x);
#pragma unroll
    for (int e = 0; e < 4; ++e) st_row8_bf16(sm + OFF_S, row, c0 + 8 * e, S_PANEL, x + 8 * e);
  }
  tmem_st_wait();
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  uint32_t ph_mma = 0;
  bool ok = true;
  for (int c = 0; c < nchunks && ok; ++c) {
    const int64_t c0 = bos + (int64_t)c * CHUNK;
    const int L = (int)((eos - c0) < CHUNK ? (eos - c0) : CHUNK);
    const int st = c & 1;
    uint8_t* kq = sm + OFF_KQ + st * KQ_STAGE;
    const uint32_t kqa = sb + OFF_KQ + st * KQ_STAGE;
    // ---- load the chunk: prefetch the next chunk's K/Q into the other stage
    //      (its previous chunk is finished); gate and beta by plain loads
    if (tid == 0 && c + 1 < nchunks) {
      uint64_t* bn = bar_kq + (st ^ 1);
      uint8_t* kqn = sm + OFF_KQ + (st ^ 1) * KQ_STAGE;
      mbar_arrive_expect_tx(bn, 4 * 8192);
#pragma unroll
      for (int pnl = 0; pnl < 2; ++pnl) {
        tma_load_3d(kqn + pnl * KQ_PANEL, &tmK, bn, 64 * pnl, h, (int)(c0 + CHUNK));
        tma_load_3d(kqn + pnl * KQ_PANEL + 8192, &tmQ, bn, 64 * pnl, h, (int)(c0 + CHUNK));
      }
    }
    if (tid < 64) {
      const size_t off = (size_t)(c0 + tid) * H + h;
      sg[tid] = (tid < L) ? p.g[off] : 0.f;
      sbeta[tid] = (tid < L) ? p.beta[off] : 0.f;
    }
    if (!(ok = cta_wait(bar_kq + st, (uint32_t)(c >> 1) & 1u, p.status))) break;
    if (!(ok = cta_wait(bar_v, (uint32_t)c & 1u, p.status))) break;
    if (L < CHUNK) {
      // rows past the sequence end belong to the next sequence (or are past
      // the tensor): zero them so they contribute nothing to any product
      const int rows = CHUNK - L;
      for (int idx = tid; idx < 6 * rows * 8; idx += NTHR) {
        const int t6 = idx / (rows * 8), rem = idx % (rows * 8);
        const int r = L + rem / 8, ch = rem % 8;
        const int pnl = t6 & 1, which = t6 >> 1;
        uint8_t* base = (which == 2) ? sm + OFF_V + pnl * V_PANEL
                                     : kq + pnl * KQ_PANEL + (which == 1 ? 8192u : 0u);
        *reinterpret_cast<uint4*>(base + r * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
      }
    }
    __syncthreads();
    if (warp == 0) {
      warp_cumsum64(sg, sgam, lane);
      __syncwarp();
      // decay factors: e^{gamma_i - gamma_j} = e^{gamma_i - mid} e^{mid - gamma_j} when the
      // chunk's gamma range keeps both factors inside e^{+-40} (no overflow, no
      // denormals); otherwise every entry takes its own exponential
      const float a0 = sgam[2 * lane], a1 = sgam[2 * lane + 1];
      float mx = fmaxf(a0, a1), mn = fminf(a0, a1);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
      }
      const bool fact = (mx - mn) <= 80.f;
      const float mid = 0.5f * (mx + mn);
      if (lane == 0) *flag = fact ? 1 : 0;
      const float gC = sgam[63];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int i = 2 * lane + e;
        const float gi = sgam[i];
        seg[i] = expf(gi);
        sdec[i] = expf(gC - gi);
        sep[i] = fact ? expf(gi - mid) : 0.f;
        sem[i] = fact ? expf(mid - gi) : 0.f;
      }
    }
    fence_proxy_async_smem();
    __syncthreads();

    // ---- Pre: KQ = [K; Q] K^T
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t a = kqa + (kk >> 2) * KQ_PANEL + (kk & 3) * 32;
        mma_bf16(tm + TM_KQ, sdesc_sw128(a, 0, 1024), sdesc_sw128(a, 0, 1024), ID_KQ, kk > 0);
      }
      mma_commit(bar_mma);
    }
    if (!(ok = cta_wait(bar_mma, ph_mma, p.status))) break;
    ph_mma ^= 1;
    tc_fence_after();
    {
      float x[32];
      tmem_ld32(tl + TM_KQ + 32 * half, x);
      tmem_ld_wait();
      const bool fact = *flag != 0;
      const int i = row & 63;
      const float gi = sgam[i], epi = sep[i];
      const float bi = (row < 64) ? sbeta[i] : 1.f;
#pragma unroll
      for (int jj = 0; jj < 32; ++jj) {
        const int j = 32 * half + jj;
        const float dcy = fact ? epi * sem[j] : expf(j <= i ? gi - sgam[j] : 0.f);
        x[jj] *= bi * dcy;
      }
      if (row < 64) {          // A_ij = beta_i Gamma_ij (k_i . k_j), j < i
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
          const int j = 32 * half + jj;
          sA[i * SOLVE_LD + j] = (j < i) ? x[jj] : 0.f;
        }
      } else {                 // Ahat_ij = Gamma_ij (q_i . k_j), j <= i
#pragma unroll
        for (int jj = 0; jj < 32; ++jj)
          if (32 * half + jj > i) x[jj] = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) st_row8_bf16(sm + OFF_AH, i, 32 * half + 8 * e, 8192, x + 8 * e);
      }
    }
    __syncthreads();
    // ---- Pre: T = (I + A)^{-1} (FP32), then T' = T diag(beta), T'' = T diag(beta e^gamma)
    solve64_tc(sA, sT, sX, tid, NTHR, CtaBar());
    for (int idx = tid; idx < 64 * 8; idx += NTHR) {
      const int i = idx >> 3, cg = (idx & 7) * 8;
      float t1[8], t2[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int j = cg + e;
        const float t = sT[i * SOLVE_LD + j] * sbeta[j];
        t1[e] = t;
        t2[e] = t * seg[j];
      }
      st_row8_bf16(sm + OFF_T1, i, cg, 8192, t1);
      st_row8_bf16(sm + OFF_T2, i, cg, 8192, t2);
    }
    fence_proxy_async_smem();
    __syncthreads();
    // ---- W^T = K^T T''^T ; U^T = V^T T'^T (into the Delta^T accumulator)
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        mma_bf16(tm + TM_WT, sdesc_sw128(kqa + kk * 2048, KQ_PANEL, 1024),
                 sdesc_sw128(sb + OFF_T2 + kk * 32, 0, 1024), ID_WT, kk > 0);
      }
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        mma_bf16(tm + TM_DT, sdesc_sw128(sb + OFF_V + kk * 2048, V_PANEL, 1024),
                 sdesc_sw128(sb + OFF_T1 + kk * 32, 0, 1024), ID_WT, kk > 0);
      }
      mma_commit(bar_mma);
    }
    if (!(ok = cta_wait(bar_mma, ph_mma, p.status))) break;
    ph_mma ^= 1;
    tc_fence_after();
    if (tid == 0 && c + 1 < nchunks) {      // V is free: load the next chunk's
      mbar_arrive_expect_tx(bar_v, 2 * 8192);
#pragma unroll
      for (int pnl = 0; pnl < 2; ++pnl)
        tma_load_3d(sm + OFF_V + pnl * V_PANEL, &tmV, bar_v, 64 * pnl, h, (int)(c0 + CHUNK));
    }
    {
      float x[32];
      tmem_ld32(tl + TM_WT + 32 * half, x);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 4; ++e) st_row8_bf16(sm + OFF_WT, row, 32 * half + 8 * e, 16384, x + 8 * e);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    // ---- ST: Delta^T += -S W^T ; Out: SQ = S Q^T
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t a = sb + OFF_S + (kk >> 2) * S_PANEL + (kk & 3) * 32;
        mma_bf16(tm + TM_DT, sdesc_sw128(a, 0, 1024),
                 sdesc_sw128(sb + OFF_WT + kk * 2048, 16384, 1024), ID_DT, 1);
      }
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t a = sb + OFF_S + (kk >> 2) * S_PANEL + (kk & 3) * 32;
        const uint32_t b = kqa + (kk >> 2) * KQ_PANEL + 8192 + (kk & 3) * 32;
        mma_bf16(tm + TM_SQ, sdesc_sw128(a, 0, 1024), sdesc_sw128(b, 0, 1024), ID_SQ, kk > 0);
      }
      mma_commit(bar_mma);
    }
    if (!(ok = cta_wait(bar_mma, ph_mma, p.status))) break;
    ph_mma ^= 1;
    tc_fence_after();
    {
      float x[32];
      tmem_ld32(tl + TM_DT + 32 * half, x);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 4; ++e) st_row8_bf16(sm + OFF_DT, row, 32 * half + 8 * e, 16384, x + 8 * e);
#pragma unroll
      for (int jj = 0; jj < 32; ++jj) x[jj] *= sdec[32 * half + jj];
#pragma unroll
      for (int e = 0; e < 4; ++e) st_row8_bf16(sm + OFF_DDT, row, 32 * half + 8 * e, 16384, x + 8 * e);
      // S <- e^{gamma_C} S in TMEM before the update accumulates on top of it
      const float gC = seg[63];
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const uint32_t col = TM_S + 64 * half + 32 * cc;
        tmem_ld32(tl + col, x);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) x[e] *= gC;
        tmem_st32(tl + col, x);
      }
      tmem_st_wait();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    // ---- ST: S += (Delta^T diag(dec)) K ; Out: OA = Delta^T Ahat^T
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        mma_bf16(tm + TM_S, sdesc_sw128(sb + OFF_DDT + kk * 32, 0, 1024),
                 sdesc_sw128(kqa + kk * 2048, KQ_PANEL, 1024), ID_SU, 1);
      }
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        mma_bf16(tm + TM_OA, sdesc_sw128(sb + OFF_DT + kk * 32, 0, 1024),
                 sdesc_sw128(sb + OFF_AH + kk * 32, 0, 1024), ID_OA, kk > 0);
      }
      mma_commit(bar_mma);
    }
    if (!(ok = cta_wait(bar_mma, ph_mma, p.status))) break;
    ph_mma ^= 1;
    tc_fence_after();
    {
      // out[i][v] = scale (e^{gamma_i} SQ[v][i] + OA[v][i]), staged as a [64][128]
      // BF16 row-major tile in the (now free) T'/T'' region, then stored 16 B at a time
      float sq[32], oa[32];
      tmem_ld32(tl + TM_SQ + 32 * half, sq);
      tmem_ld32(tl + TM_OA + 32 * half, oa);
      tmem_ld_wait();
      __nv_bfloat16* stage = reinterpret_cast<__nv_bfloat16*>(sm + OFF_T1);
#pragma unroll
      for (int jj = 0; jj < 32; ++jj) {
        const int i = 32 * half + jj;
        stage[i * D + row] = __float2bfloat16_rn(p.scale * (seg[i] * sq[jj] + oa[jj]));
      }
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int col = 64 * half + 32 * cc;
        tmem_ld32(tl + TM_S + col, sq);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 4; ++e) st_row8_bf16(sm + OFF_S, row, col + 8 * e, S_PANEL, sq + 8 * e);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    {
      const uint4* stage = reinterpret_cast<const uint4*>(sm + OFF_T1);
      for (int idx = tid; idx < 64 * 16; idx += NTHR) {
        const int i = idx >> 4, ch = idx & 15;
        if (i < L)
          *reinterpret_cast<uint4*>(p.out + ((size_t)(c0 + i) * H + h) * D + ch * 8) = stage[idx];
      }
    }
    __syncthreads();
    tc_fence_after();
  }

  if (ok && p.final_state) {
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      const int c0 = 64 * half + 32 * cc;
      float x[32];
      tmem_ld32(tl + TM_S + c0, x);
      tmem_ld_wait();
      float4* dst = reinterpret_cast<float4*>(p.final_state + state_off + (size_t)row * D + c0);
#pragma unroll
      for (int e = 0; e < 8; ++e) dst[e] = make_float4(x[4 * e], x[4 * e + 1], x[4 * e + 2], x[4 * e + 3]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tm, TM_COLS);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// [rows, H, 128] BF16 viewed as a 3-D tensor (128, H, rows); box = 64 x 1 x 64.
bool make_map(CUtensorMap* m, const void* base, int rows, int H) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
  cuuint32_t box[3] = {64, 1, 64};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool tc_fwd_available() { return encode_fn() != nullptr; }

cudaError_t launch_tc_fwd(const ChainParams& cp, int* status, cudaStream_t st) {
  const int rows = cp.B * cp.T;
  if (rows <= 0) return cudaErrorInvalidValue;
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, cp.q, rows, cp.H) || !make_map(&mk, cp.k, rows, cp.H) ||
      !make_map(&mv, cp.v, rows, cp.H))
    return cudaErrorInvalidValue;
  TcParams p;
  p.g = cp.g;
  p.beta = cp.beta;
  p.s0 = cp.s0;
  p.cu = cp.cu;
  p.out = reinterpret_cast<__nv_bfloat16*>(cp.out);
  p.final_state = cp.final_state;
  p.status = status;
  p.B = cp.B;
  p.T = cp.T;
  p.H = cp.H;
  p.N = cp.N;
  p.scale = cp.scale;
  cudaError_t e = cudaFuncSetAttribute(gdn_fwd_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  gdn_fwd_tc_kernel<<<cp.N * cp.H, NTHR, SMEM_ALLOC, st>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace sfg
