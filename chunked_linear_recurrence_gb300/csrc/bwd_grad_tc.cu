// bwd_grad_tc.cu -- token gradients of one chunk of the chunked gated delta rule on the
// sm_103a tensor cores: tcgen05 products with BF16 operands in shared memory and FP32
// accumulators in TMEM, for BF16 inputs with K = V = 128.
//
// StateFlow section 3.4.2, Eq. 18 ("OutputGrad" and "PrepGrad"): given the chunk's entry
// state S (state replay) and the cotangent dSn of its exit state (reverse state chain),
// the chunk's factors are recomputed and the gradient is pushed back through Out, ST and
// Pre -- the chunk algebra differentiated term by term (the same steps as the warp-level
// kernel in bwd_grad_mma.cu):
//
//   Ak = Gamma o K K^T (strict), Aqk = Gamma o Q K^T (incl. diagonal), T = (I + diag(beta) Ak)^-1
//   W = T diag(beta e^gamma) K, U = T diag(beta) V, Delta = U - W S^T
//   dDelta = scale Aqk^T dO + diag(dec) K dSn^T
//   G = (scale dO Delta^T) o Gamma,  dq = scale diag(e^gamma) dO S + G K
//   dW = -dDelta S,  X = T^T dDelta (dv = diag(beta) X),  Y = T^T dW,  Z = Delta dSn
//   dT = dDelta (beta V)^T + dW (beta e^gamma K)^T,  dA = -(T^T dT T^T) strictly lower
//   dKK = dA o (beta Gamma),  dk = G^T Q + diag(dec) Z + diag(beta e^gamma) Y + dKK K + dKK^T K
//   dgate = reverse cumulative sum of dgamma (collected from every decay factor), dbeta.
//
// One CTA (512 threads, one per SM) per chunk-head.  Products whose output feeds a
// contraction over the feature axis, or is a gradient row, are computed transposed --
// features on the 128 TMEM lanes, the 64 tokens on the columns -- so every product has
// M = 128: dq^T, dk^T, Z^T, Y^T, X^T, Delta^T, dDelta^T, dW^T, W^T.  The 64 x 64 token
// products (Q K^T stacked over K K^T as one M = 128 product; dO Delta^T, dT, T^T dT T^T)
// fill half of the lanes; each is placed on the lane half where the factor it combines
// with sits (dO Delta^T beside Q K^T, T^T X1 beside K K^T), so the combination stays in
// one thread.  Operand tiles are BF16 in the 128-byte-swizzled panel layout of
// tc_ptx.cuh; one tile serves as a K-major or an MN-major operand as the product needs,
// so no tile is ever transposed.  The triangular solve is the FP32 one of the forward
// (solve_tc.cuh).  Row sums over the feature axis (q . dq-part, k . Z, k . Y, v . X) are
// warp-shuffle reductions over the lanes that hold the features.
//
// S and dSn arrive as BF16 tiles in that same layout (the state replay and the reverse
// chain write them so), one bulk copy each.  The CTAs are persistent: the next chunk's S,
// dSn and dO are fetched as soon as the current chunk's last product reading them has
// completed, and its Q one step later, so that only K and V (read until the last step)
// load in the open.
//
// Each step is: one thread issues the products and commits them to an mbarrier; all
// threads wait for it, read the accumulators, write the next operand tiles; a CTA
// barrier hands the tiles to the next step.  Every wait is bounded; a CTA that gives up
// writes SF_ERR_TIMEOUT to the status word, drains its products and copies and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "api_internal.cuh"
#include "chain_tc.cuh"
#include "common.cuh"
#include "simt_chunk.cuh"
#include "solve_tc.cuh"
#include "tc_ptx.cuh"
#include "tmap.cuh"

namespace sfg {
namespace {

using namespace tc;

constexpr int D = 128;
constexpr int NT = 512;

// ---- shared memory (bytes from a 1024-aligned base) ----
constexpr uint32_t QK_PANEL = 16384;  // [Q;K]: 128 rows (Q 0-63, K 64-127) per 64-column panel
constexpr uint32_t X_PANEL = 8192;    // 64-row tiles
constexpr uint32_t F_PANEL = 16384;   // 128-row tiles
constexpr uint32_t O_QK = 0;          // [Q;K] [128][128]
constexpr uint32_t O_K = O_QK + 8192; //   its K rows
constexpr uint32_t O_V = 32768;       // V [64 tok][128 v]
constexpr uint32_t O_DO = 49152;      // dO [64 tok][128 v]
constexpr uint32_t O_S = 65536;       // S [128 v][128 k]
constexpr uint32_t O_DSN = 98304;     // dSn [128 v][128 k]
constexpr uint32_t O_DDT = 131072;    // dDelta^T [128 v][64 i]
constexpr uint32_t O_TT = 147456;     // T [64 i][64 j]
constexpr uint32_t O_DWT = 155648;    // dW^T [128 k][64 j]
constexpr uint32_t O_NWT = 172032;    // -W^T [128 k][64 i], then Delta^T [128 v][64 i]
constexpr uint32_t O_UN = 188416;     // area shared by steps that do not overlap in time:
constexpr uint32_t U_AQK = 0;         //   scale Aqk [64 j][64 i]      (until dDelta^T)
constexpr uint32_t U_AT = 8192;       //   FP32 A, then T [64][SOLVE_LD] (the solve)
constexpr uint32_t U_X = 25600;       //   FP32 solve scratch [32][SOLVE_LD]
constexpr uint32_t U_T1 = 0;          //   T' = T diag(beta)          (after dDelta^T)
constexpr uint32_t U_T2 = 25600;      //   T'' = T diag(beta e^gamma) (after the solve)
constexpr uint32_t U_DT = 8192;       //   dT [64 i][64 j]             (after the T tiles)
constexpr uint32_t U_X1 = 16384;      //   X1 = dT T^T [64 i][64 l]
constexpr uint32_t U_G = 0;           //   G [64 i][64 j]              (after W^T, U^T)
constexpr uint32_t U_DKK = 25600;     //   dKK [64 i][64 j]
constexpr uint32_t UN_BYTES = U_X + 32 * SOLVE_LD * 4;
constexpr uint32_t O_VEC = O_UN + UN_BYTES;
enum { V_G = 0, V_B, V_GAM, V_EG, V_DEC, V_BEG, V_SC, V_DG, V_DB, V_Z, V_KT, V_COUNT };
constexpr uint32_t O_BAR = O_VEC + V_COUNT * 64 * 4;
constexpr uint32_t SMEM_USED = O_BAR + 64;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;
static_assert(U_AT + 64 * SOLVE_LD * 4 <= U_X && U_T2 + 8192 <= UN_BYTES, "union area");
static_assert(U_X1 + 8192 <= U_T2 && U_DT + 8192 <= U_X1, "union area");
static_assert((O_UN + U_T2) % 1024 == 0 && O_UN % 1024 == 0, "tile alignment");
static_assert(SMEM_ALLOC <= 232448, "shared memory");
// products whose M = 128 operand reads 64 rows past a 64-row tile read these neighbours:
static_assert(O_DO + 2 * X_PANEL == O_S, "dO Delta^T: the rows past dO's second panel");
static_assert(O_UN + U_DT + X_PANEL == O_UN + U_X1, "dT T^T: the rows past dT");
static_assert(O_DDT + F_PANEL == O_TT && O_DWT + F_PANEL == O_NWT, "MN-major padding groups");
static_assert(O_TT - X_PANEL == O_DDT + X_PANEL, "T^T X1 on the upper lanes: the group before T");
// (the next chunk's S, dSn, dO and Q land while the last steps run: no product of those
// steps reads them, padding groups included)

// TMEM columns (512 allocated): accumulators of 64 FP32 columns each
constexpr uint32_t TM_KQ = 0;     // [Q;K] K^T (lanes 0-63: Q K^T, 64-127: K K^T)
constexpr uint32_t TM_DQ = 64;    // S^T dO^T, scaled in place, then += K^T G^T  (dq^T)
constexpr uint32_t TM_DK = 128;   // Q^T G + K^T dKK^T + K^T dKK
constexpr uint32_t TM_Z = 192;    // U^T - S W^T (Delta^T), then dSn^T Delta^T (Z^T)
constexpr uint32_t TM_Y = 256;    // dW^T T (Y^T)
constexpr uint32_t TM_X = 320;    // dDelta^T T (X^T)
constexpr uint32_t TM_A = 384;    // transient: dO^T Aqk, S^T dDelta^T, dW K^T, dO Delta^T, T^T X1
constexpr uint32_t TM_B = 448;    // transient: dSn K^T, K^T T''^T, dDelta V^T, dT T^T

// instruction descriptors (M = 128, N = 64)
constexpr uint32_t ID_KK = idesc_bf16(128, 64, false, false);
constexpr uint32_t ID_MK = idesc_bf16(128, 64, true, false);   // A MN-major
constexpr uint32_t ID_KM = idesc_bf16(128, 64, false, true);   // B MN-major
constexpr uint32_t ID_MM = idesc_bf16(128, 64, true, true);

constexpr unsigned long long WAIT_NS = 2000000000ull;

// TMEM -> registers: 32 lanes x 16 consecutive 32-bit columns (one lane per thread).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&r)[16]) {
  uint32_t* u = reinterpret_cast<uint32_t*>(r);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15}, [%16];"
      : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]),
        "=r"(u[7]), "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]), "=r"(u[13]),
        "=r"(u[14]), "=r"(u[15])
      : "r"(taddr));
}

// Descriptor start offsets (in 16-byte units) of the 16-wide K step kk.
__device__ __forceinline__ uint64_t kstep_k(int kk, uint32_t panel) {   // K-major
  return (uint64_t)(((uint32_t)(kk >> 2) * panel + (uint32_t)(kk & 3) * 32u) >> 4);
}
__device__ __forceinline__ uint64_t kstep_mn(int kk) { return (uint64_t)(kk * 2048 >> 4); }

__device__ __forceinline__ float bf_at(const uint8_t* tile, int row, int col, uint32_t panel) {
  return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(tile + sw128_off(row, col, panel)));
}

// Sums each of v[0..15] over the 32 lanes of the warp.  Lane l ends with the total of
// column colsum_col(l) (lanes l and l ^ 1 hold the same one).
__device__ __forceinline__ float warp_colsum16(float (&v)[16], int lane) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const bool hi = lane & 16;
    const float send = hi ? v[j] : v[j + 8];
    v[j] = (hi ? v[j + 8] : v[j]) + __shfl_xor_sync(0xffffffffu, send, 16);
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const bool hi = lane & 8;
    const float send = hi ? v[j] : v[j + 4];
    v[j] = (hi ? v[j + 4] : v[j]) + __shfl_xor_sync(0xffffffffu, send, 8);
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const bool hi = lane & 4;
    const float send = hi ? v[j] : v[j + 2];
    v[j] = (hi ? v[j + 2] : v[j]) + __shfl_xor_sync(0xffffffffu, send, 4);
  }
  {
    const bool hi = lane & 2;
    const float send = hi ? v[0] : v[1];
    v[0] = (hi ? v[1] : v[0]) + __shfl_xor_sync(0xffffffffu, send, 2);
  }
  return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 1);
}
__device__ __forceinline__ int colsum_col(int lane) {
  return ((lane >> 4) & 1) * 8 + ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1);
}

// mbarriers
enum { B_SDO = 0, B_MMA, B_DRAIN, B_Q, B_K, B_V, B_COUNT };
constexpr uint32_t TILE_BYTES = 32768;   // one BF16 [128][128] S or dSn tile

// The launch that runs the reverse chain beside the gradients (dense inputs): CTAs
// [0, nchain) run one (sequence, head) chain x each, then join the others in taking
// chunk-heads, claimed one at a time from the counter tape[nchain * FLAG_STRIDE] in the
// order the chains write their exit-cotangent tiles (chain x's count of written tiles at
// tape[x * FLAG_STRIDE]).  nchain = 0: the gradients' own launch (a fixed grid stride).
struct Fuse {
  int nchain;
  uint32_t* tape;
};
constexpr int FLAG_STRIDE = 32;   // one 128-byte line per chain

// One chunk-head: backward slot, value head, query/key head, first row, length; fused
// launch: its chain x and the tape count its exit cotangent needs (x = -1 otherwise).
struct Item {
  int64_t slot, c0;
  int h, hk, L, x;
  uint32_t need;
  bool valid;
};

__device__ __forceinline__ Item locate_item(const ChainParams& p, int64_t item, const Fuse& f) {
  Item it{};
  it.valid = false;
  it.x = -1;
  if (f.nchain > 0) {
    // the chains write chunk nc - 1 first: item = (step, chain), step-major
    const int64_t nc = n_chunks(p.T), s = item / f.nchain;
    if (s >= nc) return it;
    const int x = (int)(item % f.nchain), n = x / p.H;
    const int64_t ci = nc - 1 - s;
    it.slot = (int64_t)n * nc + ci;
    it.h = x % p.H;
    it.hk = qk_head(it.h, p.H, p.HK);
    it.c0 = (int64_t)n * p.T + ci * CHUNK;
    it.L = (int)((p.T - ci * CHUNK) < CHUNK ? (p.T - ci * CHUNK) : CHUNK);
    it.x = x;
    it.need = (uint32_t)(s + 1);
    it.valid = true;
    return it;
  }
  const int64_t slot = item / p.H;
  int n = -1;
  int64_t bos = 0, eos = 0, ci = 0;
  if (!locate_chunk(slot, p.B, p.T, p.cu, p.N, n, bos, eos, ci)) return it;
  it.slot = slot;
  it.h = (int)(item % p.H);
  it.hk = qk_head(it.h, p.H, p.HK);
  it.c0 = bos + ci * CHUNK;
  it.L = (int)((eos - it.c0) < CHUNK ? (eos - it.c0) : CHUNK);
  it.valid = true;
  return it;
}

struct Maps {
  const CUtensorMap *q, *k, *v, *dout;
};

struct Ctx {
  uint8_t* sm;
  uint32_t sb;       // shared address of sm
  uint32_t tm;       // TMEM base
  uint64_t* bars;
  float* vec;
  int tid, warp, lane, q4, wg;
  uint32_t lph, mph;   // completed phases of the per-chunk load barriers / of B_MMA
  uint32_t pend;       // thread 0: copies issued and not yet waited for (1 << B_SDO | ...)
  float ng, nb;        // threads 0-63: the next chunk's gate and beta at this thread's row
  int* status;
  const uint32_t* tape;  // fused launch: the chains' written-tile counts (FLAG_STRIDE apart)
  __device__ float* v(int which) const { return vec + which * 64; }
  // TMEM address of this warp's lane quarter at column `col`
  __device__ uint32_t ta(uint32_t col) const { return tm + ((uint32_t)(32 * q4) << 16) + col; }
};

__device__ __forceinline__ void note_timeout(const Ctx& c, uint32_t what) {
  if (!c.status) return;
  atomicCAS(c.status, 0, (int)SF_ERR_TIMEOUT);
  atomicCAS(c.status + 1, 0,
            (int)(0x40000000u | (blockIdx.x << 12) | ((threadIdx.x >> 5) << 6) | (what & 63u)));
}

// Products committed by thread 0 -> every thread waits (bounded), then orders its TMEM
// reads after them.
__device__ __forceinline__ bool wait_products(Ctx& c) {
  const bool ok = mbar_wait(&c.bars[B_MMA], c.mph & 1, WAIT_NS);
  if (!ok) note_timeout(c, 1);
  ++c.mph;
  tc_fence_after();
  return ok;
}

// Hands this step's operand tiles (generic-proxy smem writes) and TMEM reads to the next
// products; all threads agree on whether every wait so far succeeded.
__device__ __forceinline__ bool step_barrier(bool ok) {
  fence_proxy_async_smem();
  tc_fence_before();
  ok = __syncthreads_and(ok);
  tc_fence_after();
  return ok;
}

// Writes 16 values as BF16 into columns [c0, c0 + 16) of `row` of a 64-column tile.
__device__ __forceinline__ void st_row16(uint8_t* tile, int row, int c0, const float* x) {
  st_row8_bf16(tile, row, c0, X_PANEL, x);
  st_row8_bf16(tile, row, c0 + 8, X_PANEL, x + 8);
}

// Thread 0: the chunk's S and dSn tiles (bulk copies) and its dO tile (TMA).  In the fused
// launch, first the chain's tile count (bounded wait); false when that wait expired.
__device__ __forceinline__ bool fetch_sdo(Ctx& c, const ChainParams& p, const Maps& m,
                                          const Item& it) {
  if (it.x >= 0) {
    const uint32_t* flag = c.tape + (size_t)it.x * FLAG_STRIDE;
    if (ld_acquire_u32(flag) < it.need) {
      const uint64_t t0 = globaltimer_ns();
      while (ld_acquire_u32(flag) < it.need) {
        __nanosleep(200);
        if (globaltimer_ns() - t0 > WAIT_NS) {
          note_timeout(c, 6);
          return false;
        }
      }
    }
    fence_proxy_async_global();   // the chain's generic stores, then our bulk read
  }
  const uint8_t* ck = reinterpret_cast<const uint8_t*>(p.ckpt);
  const uint8_t* tp = reinterpret_cast<const uint8_t*>(p.tape);
  const size_t off = ((size_t)it.slot * p.H + it.h) * TILE_BYTES;
  c.pend |= 1u << B_SDO;
  mbar_arrive_expect_tx(&c.bars[B_SDO], 2 * TILE_BYTES + 2 * X_PANEL);
  bulk_g2s(c.sm + O_S, ck + off, TILE_BYTES, &c.bars[B_SDO]);
  bulk_g2s(c.sm + O_DSN, tp + off, TILE_BYTES, &c.bars[B_SDO]);
#pragma unroll
  for (int pp = 0; pp < 2; ++pp)
    tma_load_3d(c.sm + O_DO + pp * X_PANEL, m.dout, &c.bars[B_SDO], 64 * pp, it.h, (int)it.c0);
  return true;
}
// Thread 0: the chunk's Q tile.
__device__ __forceinline__ void fetch_q(Ctx& c, const Maps& m, const Item& it) {
  c.pend |= 1u << B_Q;
  mbar_arrive_expect_tx(&c.bars[B_Q], 2 * X_PANEL);
#pragma unroll
  for (int pp = 0; pp < 2; ++pp)
    tma_load_3d(c.sm + O_QK + pp * QK_PANEL, m.q, &c.bars[B_Q], 64 * pp, it.hk, (int)it.c0);
}
// Thread 0: the chunk's K tile.
__device__ __forceinline__ void fetch_k(Ctx& c, const Maps& m, const Item& it) {
  c.pend |= 1u << B_K;
  mbar_arrive_expect_tx(&c.bars[B_K], 2 * X_PANEL);
#pragma unroll
  for (int pp = 0; pp < 2; ++pp)
    tma_load_3d(c.sm + O_K + pp * QK_PANEL, m.k, &c.bars[B_K], 64 * pp, it.hk, (int)it.c0);
}
// Thread 0: the chunk's V tile.
__device__ __forceinline__ void fetch_v(Ctx& c, const Maps& m, const Item& it) {
  c.pend |= 1u << B_V;
  mbar_arrive_expect_tx(&c.bars[B_V], 2 * X_PANEL);
#pragma unroll
  for (int pp = 0; pp < 2; ++pp)
    tma_load_3d(c.sm + O_V + pp * X_PANEL, m.v, &c.bars[B_V], 64 * pp, it.h, (int)it.c0);
}
// Threads 0-63: the chunk's gate and beta values (registers, stored at the chunk's start).
__device__ __forceinline__ void fetch_gb(Ctx& c, const ChainParams& p, const Item& it) {
  const size_t off = (size_t)(it.c0 + c.tid) * p.H + it.h;
  c.ng = (c.tid < it.L) ? p.g[off] : 0.f;
  c.nb = (c.tid < it.L) ? p.beta[off] : 0.f;
}

// One chunk.  Its copies (S, dSn, dO, Q, K, V; gate and beta into registers) were issued
// before; this chunk issues those of the next chunk `nx` as its own tiles fall free.  False
// when a wait expired (the status word then says where).
__device__ bool grad_chunk(Ctx& c, const ChainParams& p, const Maps& m, const Item& it,
                           const Item& nx) {
  uint8_t* sm = c.sm;
  const uint32_t sb = c.sb;
  const int tid = c.tid, lane = c.lane, q4 = c.q4, wg = c.wg;
  const int h = it.h, H = p.H, L = it.L;
  const int64_t c0 = it.c0;
  const float scale = p.scale;
  float* vg = c.v(V_G);
  float* vb = c.v(V_B);
  float* vgam = c.v(V_GAM);
  float* veg = c.v(V_EG);
  float* vdec = c.v(V_DEC);
  float* vbeg = c.v(V_BEG);
  float* vsc = c.v(V_SC);
  float* vdg = c.v(V_DG);
  float* vdb = c.v(V_DB);
  float* vz = c.v(V_Z);
  float* vkt = c.v(V_KT);

  // ---- inputs: every copy is in flight already ----
  if (tid < 64) {
    vg[tid] = c.ng;
    vb[tid] = c.nb;
    vdg[tid] = 0.f;
    vdb[tid] = 0.f;
    vz[tid] = 0.f;
    vkt[tid] = 0.f;
  }
  __syncthreads();
  if (tid < 32) warp_cumsum64(vg, vgam, lane);
  __syncthreads();
  if (tid < 64) {
    const float eg = expf(vgam[tid]);
    veg[tid] = eg;
    vdec[tid] = expf(vgam[63] - vgam[tid]);
    vbeg[tid] = vb[tid] * eg;
    vsc[tid] = scale * eg;
  }
  const uint32_t par = c.lph & 1;
  bool ok = mbar_wait(&c.bars[B_SDO], par, WAIT_NS);
  if (!ok) note_timeout(c, 0);
  float sdot = 0.f;   // <dSn, S>: both tiles share one layout, so position by position
  {
    const uint4* a4 = reinterpret_cast<const uint4*>(sm + O_S);
    const uint4* b4 = reinterpret_cast<const uint4*>(sm + O_DSN);
#pragma unroll
    for (int mm = 0; mm < 4; ++mm) {
      const uint4 x = a4[tid + NT * mm], y = b4[tid + NT * mm];
      const uint32_t xa[4] = {x.x, x.y, x.z, x.w}, ya[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 fx = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xa[e]));
        const float2 fy = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ya[e]));
        sdot += fx.x * fy.x + fx.y * fy.y;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sdot += __shfl_xor_sync(0xffffffffu, sdot, o);
  if (ok && !(ok = mbar_wait(&c.bars[B_Q], par, WAIT_NS))) note_timeout(c, 3);
  if (ok && !(ok = mbar_wait(&c.bars[B_K], par, WAIT_NS))) note_timeout(c, 4);
  if (ok && !(ok = mbar_wait(&c.bars[B_V], par, WAIT_NS))) note_timeout(c, 5);
  if (ok) {
    c.pend = 0;
    ++c.lph;
  }
  if (L < 64) {
    // rows past the chunk's end read other tokens (or the fill): zero them in every tile
    for (int idx = tid; idx < (64 - L) * 8 * 8; idx += NT) {
      const int r = L + (idx >> 6), t = (idx >> 3) & 7, w = idx & 7;   // row, tile panel, 16 B
      const uint32_t base = t < 2   ? O_QK + t * QK_PANEL
                            : t < 4 ? O_K + (t - 2) * QK_PANEL
                            : t < 6 ? O_V + (t - 4) * X_PANEL
                                    : O_DO + (t - 6) * X_PANEL;
      *reinterpret_cast<uint4*>(sm + base + r * 128 + w * 16) = make_uint4(0, 0, 0, 0);
    }
  }
  if (!step_barrier(ok)) return false;
  if (lane == 0) atomicAdd(&vdg[63], veg[63] * sdot);

  // ---- [Q;K] K^T, S^T dO^T, dSn K^T ----
  if (tid == 0) {
    const uint64_t aqk = sdesc_sw128(sb + O_QK, 0, 1024), bk = sdesc_sw128(sb + O_K, 0, 1024);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      mma_bf16(c.tm + TM_KQ, aqk + kstep_k(kk, QK_PANEL), bk + kstep_k(kk, QK_PANEL), ID_KK,
               kk > 0);
    const uint64_t as = sdesc_sw128(sb + O_S, F_PANEL, 1024), bdo = sdesc_sw128(sb + O_DO, 0, 1024);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      mma_bf16(c.tm + TM_DQ, as + kstep_mn(kk), bdo + kstep_k(kk, X_PANEL), ID_MK, kk > 0);
    const uint64_t ad = sdesc_sw128(sb + O_DSN, 0, 1024);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      mma_bf16(c.tm + TM_B, ad + kstep_k(kk, F_PANEL), bk + kstep_k(kk, QK_PANEL), ID_KK, kk > 0);
    mma_commit(&c.bars[B_MMA]);
  }
  ok = wait_products(c);
  {
    // Aqk (lanes 0-63) -> scale Aqk tile; A = beta Ak (lanes 64-127) -> the solve's input
    float x[16];
    tmem_ld16(c.ta(TM_KQ + 16 * wg), x);
    tmem_ld_wait();
    const int i = 32 * (q4 & 1) + lane, j0 = 16 * wg;
    const float gi = vgam[i];
    if (q4 < 2) {
      float y[16];
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) {
        const int j = j0 + jj;
        y[jj] = (j <= i) ? scale * expf(gi - vgam[j]) * x[jj] : 0.f;
      }
      st_row16(sm + O_UN + U_AQK, i, j0, y);
    } else {
      float* at = reinterpret_cast<float*>(sm + O_UN + U_AT) + i * SOLVE_LD + j0;
      const float bi = vb[i];
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) {
        const int j = j0 + jj;
        at[jj] = (j < i) ? bi * expf(gi - vgam[j]) * x[jj] : 0.f;
      }
    }
  }
  if (!step_barrier(ok)) return false;

  // ---- dDelta^T's first part dO^T (scale Aqk); meanwhile warps 0-7 solve for T and warps
  // 8-15 finish dq's first part and form dDelta^T ----
  if (tid == 0) {
    const uint64_t a = sdesc_sw128(sb + O_DO, X_PANEL, 1024);
    const uint64_t b = sdesc_sw128(sb + O_UN + U_AQK, X_PANEL, 1024);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_bf16(c.tm + TM_A, a + kstep_mn(kk), b + kstep_mn(kk), ID_MM, kk > 0);
    mma_commit(&c.bars[B_MMA]);
  }
  if (c.warp < 8) {
    float* AT = reinterpret_cast<float*>(sm + O_UN + U_AT);
    solve64_tc_inplace(AT, reinterpret_cast<float*>(sm + O_UN + U_X), tid, 256,
                       [] { named_bar(1, 256); });
    ok = wait_products(c);   // T' overwrites the Aqk tile that dO^T (scale Aqk) reads
    // T, T' = T diag(beta), T'' = T diag(beta e^gamma) as BF16 tiles [i][j]
    for (int idx = tid; idx < 64 * 8; idx += 256) {
      const int i = idx >> 3, j0 = 8 * (idx & 7);
      const float* at = AT + i * SOLVE_LD + j0;
      float t[8], t1[8], t2[8];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        t[jj] = at[jj];
        t1[jj] = t[jj] * vb[j0 + jj];
        t2[jj] = t[jj] * vbeg[j0 + jj];
      }
      st_row8_bf16(sm + O_TT, i, j0, X_PANEL, t);
      st_row8_bf16(sm + O_UN + U_T1, i, j0, X_PANEL, t1);
      st_row8_bf16(sm + O_UN + U_T2, i, j0, X_PANEL, t2);
    }
  } else {
    // two warps per lane quarter, 32 columns each
    const int r = 32 * q4 + lane, cbase = 32 * ((c.warp - 8) >> 2);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      // S^T dO^T (features k on the lanes): scale column i by scale e^{gamma_i}, add
      // q_i . (that column) to dgamma_i, and leave the scaled values for G K to accumulate on
      const int i0 = cbase + 16 * hh;
      float x[16], pr[16];
      tmem_ld16(c.ta(TM_DQ + i0), x);
      tmem_ld_wait();
#pragma unroll
      for (int ii = 0; ii < 16; ++ii) {
        x[ii] *= vsc[i0 + ii];
        pr[ii] = x[ii] * bf_at(sm + O_QK, i0 + ii, r, QK_PANEL);
      }
      uint32_t u[16];
#pragma unroll
      for (int ii = 0; ii < 16; ++ii) u[ii] = __float_as_uint(x[ii]);
      tmem_st16(c.ta(TM_DQ + i0), u);
      const float sum = warp_colsum16(pr, lane);
      if (!(lane & 1)) atomicAdd(&vdg[i0 + colsum_col(lane)], sum);
    }
    tmem_st_wait();
    ok = wait_products(c);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      // dDelta^T = dO^T (scale Aqk) + (dSn K^T) diag(dec)
      const int i0 = cbase + 16 * hh;
      float x1[16], x2[16];
      tmem_ld16(c.ta(TM_A + i0), x1);
      tmem_ld16(c.ta(TM_B + i0), x2);
      tmem_ld_wait();
#pragma unroll
      for (int ii = 0; ii < 16; ++ii) x1[ii] += vdec[i0 + ii] * x2[ii];
      st_row16(sm + O_DDT, r, i0, x1);
    }
  }
  if (!step_barrier(ok)) return false;

  // ---- S^T dDelta^T (-> dW^T), K^T T''^T (W^T), V^T T'^T (U^T), dDelta^T T (X^T) ----
  if (tid == 0) {
    const uint64_t as = sdesc_sw128(sb + O_S, F_PANEL, 1024);
    const uint64_t bdd = sdesc_sw128(sb + O_DDT, F_PANEL, 1024);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      mma_bf16(c.tm + TM_A, as + kstep_mn(kk), bdd + kstep_mn(kk), ID_MM, kk > 0);
    const uint64_t akt = sdesc_sw128(sb + O_K, QK_PANEL, 1024);
    const uint64_t bt2 = sdesc_sw128(sb + O_UN + U_T2, 0, 1024);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_bf16(c.tm + TM_B, akt + kstep_mn(kk), bt2 + kstep_k(kk, X_PANEL), ID_MK, kk > 0);
    const uint64_t avt = sdesc_sw128(sb + O_V, X_PANEL, 1024);
    const uint64_t bt1 = sdesc_sw128(sb + O_UN + U_T1, 0, 1024);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_bf16(c.tm + TM_Z, avt + kstep_mn(kk), bt1 + kstep_k(kk, X_PANEL), ID_MK, kk > 0);
    const uint64_t add = sdesc_sw128(sb + O_DDT, 0, 1024);
    const uint64_t btt = sdesc_sw128(sb + O_TT, X_PANEL, 1024);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_bf16(c.tm + TM_X, add + kstep_k(kk, F_PANEL), btt + kstep_mn(kk), ID_KM, kk > 0);
    mma_commit(&c.bars[B_MMA]);
  }
  ok = wait_products(c);
  {
    // dW^T = -(S^T dDelta^T) and -W^T as BF16 tiles (features on the rows)
    float x[16];
    const int r = 32 * q4 + lane, i0 = 16 * wg;
    tmem_ld16(c.ta(TM_A + 16 * wg), x);
    tmem_ld_wait();
#pragma unroll
    for (int ii = 0; ii < 16; ++ii) x[ii] = -x[ii];
    st_row16(sm + O_DWT, r, i0, x);
    tmem_ld16(c.ta(TM_B + 16 * wg), x);
    tmem_ld_wait();
#pragma unroll
    for (int ii = 0; ii < 16; ++ii) x[ii] = -x[ii];
    st_row16(sm + O_NWT, r, i0, x);
  }
  if (!step_barrier(ok)) return false;

  // ---- Delta^T = U^T + S (-W^T); Y^T = dW^T T; dT's two parts dW K^T, dDelta V^T ----
  if (tid == 0) {
    const uint64_t as = sdesc_sw128(sb + O_S, 0, 1024);
    const uint64_t bnw = sdesc_sw128(sb + O_NWT, F_PANEL, 1024);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      mma_bf16(c.tm + TM_Z, as + kstep_k(kk, F_PANEL), bnw + kstep_mn(kk), ID_KM, 1u);
    const uint64_t adw = sdesc_sw128(sb + O_DWT, 0, 1024);
    const uint64_t btt = sdesc_sw128(sb + O_TT, X_PANEL, 1024);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_bf16(c.tm + TM_Y, adw + kstep_k(kk, F_PANEL), btt + kstep_mn(kk), ID_KM, kk > 0);
    // token products on lanes 0-63 (the MN-major A's second group of 64 columns reads the
    // next tile and fills lanes 64-127, which nothing reads)
    const uint64_t adwm = sdesc_sw128(sb + O_DWT, F_PANEL, 1024);
    const uint64_t bk = sdesc_sw128(sb + O_K, 0, 1024);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      mma_bf16(c.tm + TM_A, adwm + kstep_mn(kk), bk + kstep_k(kk, QK_PANEL), ID_MK, kk > 0);
    const uint64_t addm = sdesc_sw128(sb + O_DDT, F_PANEL, 1024);
    const uint64_t bv = sdesc_sw128(sb + O_V, 0, 1024);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      mma_bf16(c.tm + TM_B, addm + kstep_mn(kk), bv + kstep_k(kk, X_PANEL), ID_MK, kk > 0);
    mma_commit(&c.bars[B_MMA]);
  }
  {
    // (while those run) X^T = dDelta^T T, features v on the lanes: dv = diag(beta) X;
    // dbeta += v . X
    const int r = 32 * q4 + lane, i0 = 16 * wg;
    float x[16], pv[16];
    tmem_ld16(c.ta(TM_X + 16 * wg), x);
    tmem_ld_wait();
    __nv_bfloat16* dv = reinterpret_cast<__nv_bfloat16*>(p.dv);
    const size_t base = ((size_t)(c0 + i0) * H + h) * D + r;
#pragma unroll
    for (int ii = 0; ii < 16; ++ii) {
      const int i = i0 + ii;
      pv[ii] = bf_at(sm + O_V, i, r, X_PANEL) * x[ii];
      if (i < L) dv[base + (size_t)ii * H * D] = __float2bfloat16_rn(vb[i] * x[ii]);
    }
    const float sum = warp_colsum16(pv, lane);
    if (!(lane & 1)) atomicAdd(&vdb[i0 + colsum_col(lane)], sum);
  }
  ok = wait_products(c) && ok;
  {
    // Delta^T -> BF16 tile (over -W^T, whose product has completed)
    float x[16];
    tmem_ld16(c.ta(TM_Z + 16 * wg), x);
    tmem_ld_wait();
    st_row16(sm + O_NWT, 32 * q4 + lane, 16 * wg, x);
  }
  if (q4 < 2) {
    // dT = (dDelta V^T) diag(beta) + (dW K^T) diag(beta e^gamma), rows i on lanes 0-63
    float x1[16], x2[16];
    tmem_ld16(c.ta(TM_B + 16 * wg), x1);
    tmem_ld16(c.ta(TM_A + 16 * wg), x2);
    tmem_ld_wait();
    const int i = 32 * q4 + lane, j0 = 16 * wg;
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) x1[jj] = vb[j0 + jj] * x1[jj] + vbeg[j0 + jj] * x2[jj];
    st_row16(sm + O_UN + U_DT, i, j0, x1);
  }
  if (!step_barrier(ok)) return false;

  // ---- dO Delta^T (lanes 0-63), Z^T = dSn^T Delta^T, X1 = dT T^T (lanes 0-63) ----
  if (tid == 0) {
    const uint64_t ado = sdesc_sw128(sb + O_DO, 0, 1024);
    const uint64_t bd = sdesc_sw128(sb + O_NWT, F_PANEL, 1024);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      mma_bf16(c.tm + TM_A, ado + kstep_k(kk, X_PANEL), bd + kstep_mn(kk), ID_KM, kk > 0);
    const uint64_t adn = sdesc_sw128(sb + O_DSN, F_PANEL, 1024);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      mma_bf16(c.tm + TM_Z, adn + kstep_mn(kk), bd + kstep_mn(kk), ID_MM, kk > 0);
    const uint64_t adt = sdesc_sw128(sb + O_UN + U_DT, 0, 1024);
    const uint64_t bt = sdesc_sw128(sb + O_TT, 0, 1024);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_bf16(c.tm + TM_B, adt + kstep_k(kk, X_PANEL), bt + kstep_k(kk, X_PANEL), ID_KK, kk > 0);
    mma_commit(&c.bars[B_MMA]);
    if (nx.valid) {
      // the next chunk's V (every read of this chunk's V is behind the barrier above)
      fence_proxy_async_smem();
      fetch_v(c, m, nx);
    }
  }
  {
    // (while those run) Y^T = dW^T T, features k on the lanes: kt_i = k_i . Y_i
    const int r = 32 * q4 + lane, i0 = 16 * wg;
    float x[16];
    tmem_ld16(c.ta(TM_Y + 16 * wg), x);
    tmem_ld_wait();
#pragma unroll
    for (int ii = 0; ii < 16; ++ii) x[ii] *= bf_at(sm + O_K, i0 + ii, r, QK_PANEL);
    const float sum = warp_colsum16(x, lane);
    if (!(lane & 1)) atomicAdd(&vkt[i0 + colsum_col(lane)], sum);
  }
  ok = wait_products(c) && ok;
  if (tid == 0 && nx.valid) {
    // the next chunk's S, dSn and dO (the last products reading this chunk's have completed)
    fence_proxy_async_smem();
    ok = fetch_sdo(c, p, m, nx) && ok;
  }
  if (tid < 64 && nx.valid) fetch_gb(c, p, nx);
  if (q4 < 2) {
    // dAqk = scale dO Delta^T: G = dAqk o Gamma (lower incl. diagonal) -> tile; rho =
    // G o (Q K^T) -> dgamma_i += row sum, dgamma_j -= column sum.  X1 -> tile.
    float x[16], r[16];
    tmem_ld16(c.ta(TM_A + 16 * wg), x);
    tmem_ld16(c.ta(TM_KQ + 16 * wg), r);
    tmem_ld_wait();
    const int i = 32 * q4 + lane, j0 = 16 * wg;
    const float gi = vgam[i];
    float rs = 0.f;
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) {
      const int j = j0 + jj;
      const float gv = (j <= i) ? scale * x[jj] * expf(gi - vgam[j]) : 0.f;
      x[jj] = gv;
      r[jj] *= gv;
      rs += r[jj];
    }
    st_row16(sm + O_UN + U_G, i, j0, x);
    atomicAdd(&vdg[i], rs);
    const float cs = warp_colsum16(r, lane);
    if (!(lane & 1)) atomicAdd(&vdg[j0 + colsum_col(lane)], -cs);
    tmem_ld16(c.ta(TM_B + 16 * wg), x);
    tmem_ld_wait();
    st_row16(sm + O_UN + U_X1, i, j0, x);
  }
  if (!step_barrier(ok)) return false;

  // ---- dq^T += K^T G^T; dk^T = Q^T G; T^T X1 on lanes 64-127 ----
  if (tid == 0) {
    const uint64_t akt = sdesc_sw128(sb + O_K, QK_PANEL, 1024);
    const uint64_t bg = sdesc_sw128(sb + O_UN + U_G, X_PANEL, 1024);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_bf16(c.tm + TM_DQ, akt + kstep_mn(kk), bg + kstep_k(kk, X_PANEL), ID_MK, 1u);
    const uint64_t aqt = sdesc_sw128(sb + O_QK, QK_PANEL, 1024);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_bf16(c.tm + TM_DK, aqt + kstep_mn(kk), bg + kstep_mn(kk), ID_MM, kk > 0);
    // A = T^T as an MN-major operand whose second group of 64 rows (lanes 64-127) is T:
    // the descriptor starts one tile before T
    const uint64_t att = sdesc_sw128(sb + O_TT - X_PANEL, X_PANEL, 1024);
    const uint64_t bx1 = sdesc_sw128(sb + O_UN + U_X1, X_PANEL, 1024);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_bf16(c.tm + TM_A, att + kstep_mn(kk), bx1 + kstep_mn(kk), ID_MM, kk > 0);
    mma_commit(&c.bars[B_MMA]);
  }
  {
    // (while those run) Z^T = dSn^T Delta^T, features k on the lanes: z_i = k_i . Z_i
    const int r = 32 * q4 + lane, i0 = 16 * wg;
    float x[16];
    tmem_ld16(c.ta(TM_Z + 16 * wg), x);
    tmem_ld_wait();
#pragma unroll
    for (int ii = 0; ii < 16; ++ii) x[ii] *= bf_at(sm + O_K, i0 + ii, r, QK_PANEL);
    const float sum = warp_colsum16(x, lane);
    if (!(lane & 1)) atomicAdd(&vz[i0 + colsum_col(lane)], sum);
  }
  ok = wait_products(c) && ok;
  if (tid == 0 && nx.valid) {
    // the next chunk's Q (the last product reading this chunk's Q has completed)
    fence_proxy_async_smem();
    fetch_q(c, m, nx);
  }
  if (q4 >= 2) {
    // dA = -(T^T X1) strictly lower (rows i on lanes 64-127, beside K K^T): dbeta_i +=
    // sum_j dA Ak; rho = dA beta_i Ak -> dgamma; dKK = dA beta_i Gamma -> tile
    float x[16], r[16];
    tmem_ld16(c.ta(TM_A + 16 * wg), x);
    tmem_ld16(c.ta(TM_KQ + 16 * wg), r);
    tmem_ld_wait();
    const int i = 32 * (q4 - 2) + lane, j0 = 16 * wg;
    const float gi = vgam[i], bi = vb[i];
    float r1 = 0.f, rs = 0.f;
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) {
      const int j = j0 + jj;
      float dkk = 0.f, rho = 0.f;
      if (j < i) {
        const float gam = expf(gi - vgam[j]), da = -x[jj], ak = gam * r[jj];
        r1 += da * ak;
        rho = da * bi * ak;
        dkk = da * bi * gam;
      }
      x[jj] = dkk;
      r[jj] = rho;
      rs += rho;
    }
    st_row16(sm + O_UN + U_DKK, i, j0, x);
    atomicAdd(&vdb[i], r1);
    atomicAdd(&vdg[i], rs);
    const float cs = warp_colsum16(r, lane);
    if (!(lane & 1)) atomicAdd(&vdg[j0 + colsum_col(lane)], -cs);
  }
  if (!step_barrier(ok)) return false;

  // ---- dk^T += K^T dKK^T + K^T dKK ----
  if (tid == 0) {
    const uint64_t akt = sdesc_sw128(sb + O_K, QK_PANEL, 1024);
    const uint64_t bkk = sdesc_sw128(sb + O_UN + U_DKK, X_PANEL, 1024);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_bf16(c.tm + TM_DK, akt + kstep_mn(kk), bkk + kstep_k(kk, X_PANEL), ID_MK, 1u);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_bf16(c.tm + TM_DK, akt + kstep_mn(kk), bkk + kstep_mn(kk), ID_MM, 1u);
    mma_commit(&c.bars[B_MMA]);
  }
  ok = wait_products(c);
  if (tid == 0 && nx.valid) {
    // the next chunk's K (the last product reading this chunk's K has completed)
    fence_proxy_async_smem();
    fetch_k(c, m, nx);
  }
  if (tid < 32) {
    // dgate and dbeta (every contribution is in by now): the exit-state decay (dk gained
    // dec o Z, so dgamma_i -= dec_i z_i and the chunk's last position collects their sum),
    // Y (dbeta += e^gamma kt, dgamma += beta e^gamma kt); dgate = reverse cumulative sum of
    // dgamma.  Lane l holds rows 2l and 2l + 1.
    float d[2], db[2], tz = 0.f;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int i = 2 * lane + e;
      const float t = vdec[i] * vz[i];
      tz += t;
      d[e] = vdg[i] - t + vbeg[i] * vkt[i];
      db[e] = vdb[i] + veg[i] * vkt[i];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tz += __shfl_xor_sync(0xffffffffu, tz, o);
    if (lane == 31) d[1] += tz;
    float suf = d[0] + d[1];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float t = __shfl_down_sync(0xffffffffu, suf, o);
      if (lane + o < 32) suf += t;
    }
    const float r[2] = {suf, suf - d[0]};
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int i = 2 * lane + e;
      if (i < L) {
        const size_t off = (size_t)(c0 + i) * H + h;
        p.dg[off] = r[e];
        p.dbeta[off] = db[e];
      }
    }
  }

  // ---- dq and dk rows (features on the lanes, tokens on the columns) ----
  {
    const int r = 32 * q4 + lane, i0 = 16 * wg;
    const size_t row_stride = (size_t)H * D;
    const size_t base = ((size_t)(c0 + i0) * H + h) * D + r;
    float x[16], y[16], z[16];
    tmem_ld16(c.ta(TM_DQ + 16 * wg), x);
    tmem_ld_wait();
    if (p.dqk_f32) {
      float* dq = reinterpret_cast<float*>(p.dq);
#pragma unroll
      for (int ii = 0; ii < 16; ++ii)
        if (i0 + ii < L) dq[base + ii * row_stride] = x[ii];
    } else {
      __nv_bfloat16* dq = reinterpret_cast<__nv_bfloat16*>(p.dq);
#pragma unroll
      for (int ii = 0; ii < 16; ++ii)
        if (i0 + ii < L) dq[base + ii * row_stride] = __float2bfloat16_rn(x[ii]);
    }
    // dk = Q^T G + K^T (dKK + dKK^T) + Z^T diag(dec) + Y^T diag(beta e^gamma)
    tmem_ld16(c.ta(TM_DK + 16 * wg), x);
    tmem_ld16(c.ta(TM_Z + 16 * wg), z);
    tmem_ld16(c.ta(TM_Y + 16 * wg), y);
    tmem_ld_wait();
#pragma unroll
    for (int ii = 0; ii < 16; ++ii) x[ii] += vdec[i0 + ii] * z[ii] + vbeg[i0 + ii] * y[ii];
    if (p.dqk_f32) {
      float* dk = reinterpret_cast<float*>(p.dk);
#pragma unroll
      for (int ii = 0; ii < 16; ++ii)
        if (i0 + ii < L) dk[base + ii * row_stride] = x[ii];
    } else {
      __nv_bfloat16* dk = reinterpret_cast<__nv_bfloat16*>(p.dk);
#pragma unroll
      for (int ii = 0; ii < 16; ++ii)
        if (i0 + ii < L) dk[base + ii * row_stride] = __float2bfloat16_rn(x[ii]);
    }
  }
  tc_fence_before();
  return ok;
}

// kFused: the CTAs below f.nchain run the reverse chain (chain_tc.cuh) over the records
// `fac`; the others take the chunk-heads as their exit cotangents arrive.
template <bool kFused>
__global__ void __launch_bounds__(NT, 1)
    tc_bwd_grad_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                       const __grid_constant__ CUtensorMap mv,
                       const __grid_constant__ CUtensorMap mdo, const ChainParams p,
                       const float* fac, const Fuse f) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Ctx c;
  c.sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  if constexpr (kFused) {
    if ((int)blockIdx.x < f.nchain)
      chaintc::chain_cta<true>(&mk, &mdo, p, fac, (int)blockIdx.x,
                               f.tape + (size_t)blockIdx.x * FLAG_STRIDE, c.sm);
  }
  c.sb = smem_u32(c.sm);
  c.bars = reinterpret_cast<uint64_t*>(c.sm + O_BAR);
  c.vec = reinterpret_cast<float*>(c.sm + O_VEC);
  c.tid = threadIdx.x;
  c.warp = c.tid >> 5;
  c.lane = c.tid & 31;
  c.q4 = c.warp & 3;
  c.wg = c.warp >> 2;
  c.lph = 0;
  c.mph = 0;
  c.pend = 0;
  c.ng = c.nb = 0.f;
  c.status = p.status;
  c.tape = f.tape;
  const Maps m{&mq, &mk, &mv, &mdo};
  uint32_t* tslot = reinterpret_cast<uint32_t*>(c.sm + O_BAR + 8 * B_COUNT);
  uint32_t* claim = tslot + 1;   // fused: the chunk-head claimed last
  uint32_t* counter = f.tape + (size_t)f.nchain * FLAG_STRIDE;
  if (c.tid == 0) {
    if constexpr (kFused) *claim = atomicAdd(counter, 2u);   // this chunk-head and the next
    for (int b = 0; b < B_COUNT; ++b) mbar_init(&c.bars[b], 1);
    fence_mbar_init();
    prefetch_tmap(&mq);
    prefetch_tmap(&mk);
    prefetch_tmap(&mv);
    prefetch_tmap(&mdo);
  }
  if (c.warp == 0) tmem_alloc(tslot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  c.tm = *tslot;
  // chunk-heads blockIdx.x, + gridDim.x, ... in the order (slot, head) until the first empty
  // one; fused: claimed in the order (chain step, chain)
  int64_t next = kFused ? (int64_t)*claim + 1 : (int64_t)blockIdx.x + gridDim.x;
  Item it = locate_item(p, kFused ? (int64_t)*claim : (int64_t)blockIdx.x, f);
  bool ok = true;
  if (c.tid == 0 && it.valid) {
    ok = fetch_sdo(c, p, m, it);
    if (ok) {
      fetch_q(c, m, it);
      fetch_k(c, m, it);
      fetch_v(c, m, it);
    }
  }
  if (c.tid < 64 && it.valid) fetch_gb(c, p, it);
  ok = __syncthreads_and(ok);
  while (it.valid && ok) {
    const Item nx = locate_item(p, next, f);
    ok = grad_chunk(c, p, m, it, nx);
    if (!ok) break;
    // (every thread read *claim before grad_chunk's first CTA barrier)
    if (kFused && c.tid == 0) *claim = atomicAdd(counter, 1u);
    __syncthreads();   // the next chunk's vectors overwrite those read above
    next = kFused ? (int64_t)*claim : next + gridDim.x;
    it = nx;
  }
  if (!ok && c.tid == 0) {
    // leave no product running into the TMEM freed below, and no copy landing after exit
    mma_commit(&c.bars[B_DRAIN]);
    mbar_wait(&c.bars[B_DRAIN], 0, WAIT_NS);
    for (int b = 0; b < B_COUNT; ++b)
      if (c.pend & (1u << b)) mbar_wait(&c.bars[b], c.lph & 1, WAIT_NS);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (c.warp == 0) tmem_dealloc(c.tm, 512);
}

}  // namespace

size_t tc_bwd_grad_smem() { return SMEM_ALLOC; }

cudaError_t launch_tc_bwd_grad(const ChainParams& p, int64_t slots, cudaStream_t st) {
  if (slots <= 0 || (int64_t)p.B * p.T == 0) return cudaSuccess;   // no chunk
  CUtensorMap mq, mk, mv, mdo;
  const int rows = p.B * p.T;
  if (!make_bf16_map(&mq, p.q, rows, p.HK) || !make_bf16_map(&mk, p.k, rows, p.HK) ||
      !make_bf16_map(&mv, p.v, rows, p.H) || !make_bf16_map(&mdo, p.dout, rows, p.H))
    return cudaErrorInvalidValue;
  auto kern = tc_bwd_grad_kernel<false>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  int dev = 0, nsm = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  // one persistent CTA per SM (the shared memory allows no second), at most one per item
  const int64_t items = slots * p.H;
  const int grid = (int)(items < nsm ? items : nsm);
  const Fuse f{0, nullptr};
  const float* fac = nullptr;
  if (grid > 0) kern<<<grid, NT, SMEM_ALLOC, st>>>(mq, mk, mv, mdo, p, fac, f);
  return cudaGetLastError();
}

bool tc_bwd_fusable(const ChainParams& p) {
  int dev = 0, nsm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return false;
  const int chains = p.N * p.H;
  return !p.cu && p.sync && p.B == p.N && chains >= 1 && chains <= 64 && nsm - chains >= 32 &&
         (int64_t)p.B * p.T > 0;
}

cudaError_t launch_tc_bwd_fused(const ChainParams& p, const float* fac, cudaStream_t st) {
  CUtensorMap mq, mk, mv, mdo;
  const int rows = p.B * p.T;
  if (!make_bf16_map(&mq, p.q, rows, p.HK) || !make_bf16_map(&mk, p.k, rows, p.HK) ||
      !make_bf16_map(&mv, p.v, rows, p.H) || !make_bf16_map(&mdo, p.dout, rows, p.H))
    return cudaErrorInvalidValue;
  static_assert(chaintc::SMEM_ALLOC <= SMEM_ALLOC, "the chain CTAs fit the launch's smem");
  const void* kern = reinterpret_cast<const void*>(tc_bwd_grad_kernel<true>);
  cudaError_t e = cudaFuncSetAttribute(tc_bwd_grad_kernel<true>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  int dev = 0, nsm = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  Fuse f{p.N * p.H, p.sync};
  // the chains' tile counts and the claim counter
  e = cudaMemsetAsync(p.sync, 0, (size_t)(f.nchain + 1) * FLAG_STRIDE * sizeof(uint32_t), st);
  if (e != cudaSuccess) return e;
  // cooperative: every chain CTA is resident with the gradient CTAs that wait for it
  ChainParams pc = p;
  void* args[] = {&mq, &mk, &mv, &mdo, &pc, const_cast<float**>(&fac), &f};
  return cudaLaunchCooperativeKernel(kern, dim3(nsm), dim3(NT), args, SMEM_ALLOC, st);
}

}  // namespace sfg
