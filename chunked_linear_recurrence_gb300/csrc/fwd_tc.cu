// fwd_tc.cu -- tensor-core forward of the chunked gated delta rule for BF16
// q/k/v with K = V = 128 on sm_103a: TMA tile loads, tcgen05.mma with FP32
// accumulators in TMEM, the FP32 state carried in TMEM across chunks.
//
// One CTA per (sequence, head) chain walks its 64-token chunks in order
// (StateFlow section 2.2, Eq. 2: Pre -> ST -> Out per chunk; section 3.1,
// Eq. 4-5: a chunk's output state is the next chunk's input state).  The CTA
// is warp-specialised so that the next chunk's preparation overlaps the
// current chunk's state transition (the on-chip form of StateFlow's
// split-and-overlap schedule, section 3.4.2, Eq. 17):
//
//   warp 0      loader: TMA of K/Q (3-stage ring) and V (2-stage ring), gate/beta
//   warp 1      MMA issuer: one thread issues tcgen05.mma from a non-blocking
//               priority loop (state-transition products first)
//   warps 4-7   state: the serial chain -- Delta^T and the state S between MMAs
//   warps 8-11  prep:  decays, A and Ahat, e^gamma-scaled Q, the triangular
//               solve, T' and T'', the W^T tile -- for the chunk ahead
//   warps 12-15 out:   reads the output accumulator and stores BF16 rows
//
// Products (every M is 128, the full TMEM lane count; "A@tmem" = the A
// operand is read from TMEM as BF16 pairs):
//   KQ   = [K; Q] K^T                                      N=64,  K=128
//   W^T  = K^T T''^T,   T'' = T diag(beta e^gamma)         N=64,  K=64
//   U^T  = V^T T'^T,    T'  = T diag(beta)  -> Delta^T acc N=64,  K=64
//   Delta^T += -S W^T                      (S A@tmem)      N=64,  K=128
//   O    = S (diag(e^gamma) Q)^T           (S A@tmem)      N=64,  K=128
//   S   <- e^{gamma_C} S + (Delta^T diag(dec)) K  (A@tmem) N=128, K=64
//   O   += Delta^T Ahat^T,  Ahat = M o Gamma o Q K^T (A@tmem) N=64, K=64
//   out[i][v] = scale O[v][i]
// The 64x64 solve T = (I + A)^{-1} is FP32 (solve_tc.cuh).  BF16 copies of
// S, W, Delta, T', T'' are the tensor-core operands; S itself stays FP32 in
// TMEM (the pages stage chunk-entry states in the Q/K/V dtype the same way).
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
constexpr int NTHR = 512;
constexpr int BAR_STATE = 1, BAR_PREP = 2;   // named barriers: state (128 threads), prep (256)

// Shared-memory map (bytes from a 1024-aligned base); tiles use the panel layout of tc_ptx.cuh.
constexpr uint32_t KQ_STAGES = 3, V_STAGES = 2;
constexpr uint32_t OFF_KQ = 0;           // 3 x 32 KB; stage = 2 panels x 16 KB (rows 0-63 K, 64-127 Q)
constexpr uint32_t KQ_STAGE = 32768;
constexpr uint32_t KQ_PANEL = 16384;
constexpr uint32_t OFF_V = 98304;        // 2 x 16 KB; stage = 2 panels x 8 KB: V [64][128]
constexpr uint32_t V_STAGE = 16384;
constexpr uint32_t V_PANEL = 8192;
constexpr uint32_t OFF_WT = 131072;      // 16 KB: W^T [128 k][64 i]
constexpr uint32_t OFF_T1 = 147456;      // 8 KB: T'  [64 i][64 j]
constexpr uint32_t OFF_T2 = 155648;      // 8 KB: T'' [64 i][64 j]
constexpr uint32_t OFF_AH = 163840;      // 2 x 8 KB: Ahat [64 i][64 j]
constexpr uint32_t OFF_AT = 180224;      // FP32 [64][SOLVE_LD]: A, then T (in place)
constexpr uint32_t OFF_X = 197632;       // FP32 [32][SOLVE_LD]: solve scratch
constexpr uint32_t OFF_VEC = 206336;     // 3 stages x 512 floats (see VEC_*)
constexpr uint32_t OFF_BAR = 212480;     // mbarriers, TMEM address, abort flag
constexpr uint32_t SMEM_USED = OFF_BAR + 256;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;
static_assert(OFF_AT + 64 * SOLVE_LD * 4 <= OFF_X, "AT");
static_assert(OFF_X + 32 * SOLVE_LD * 4 <= OFF_VEC, "X");
static_assert(OFF_VEC + KQ_STAGES * 512 * 4 <= OFF_BAR, "VEC");
static_assert(SMEM_ALLOC <= 232448, "shared memory");

// Per-chunk vectors (ring stage = chunk % 3): gate, beta (loader); the rest (prep).
constexpr int VEC_G = 0, VEC_BETA = 64, VEC_GAM = 128, VEC_EG = 192, VEC_DEC = 256,
              VEC_EP = 320, VEC_EM = 384, VEC_FLAG = 448;

// TMEM columns.
constexpr uint32_t TM_S = 0;      // S FP32 [v][k]                  128
constexpr uint32_t TM_KQ = 128;   // [K;Q] K^T                      64
constexpr uint32_t TM_WT = 192;   // W^T [k][i]                     64
constexpr uint32_t TM_DT = 256;   // U^T / Delta^T FP32 [v][j]      64
constexpr uint32_t TM_O = 320;    // O [v][i]                       64
constexpr uint32_t TM_SB = 384;   // S BF16 pairs (A operand)       64
constexpr uint32_t TM_DB = 448;   // Delta^T BF16 pairs             32
constexpr uint32_t TM_DDB = 480;  // (Delta^T diag(dec)) BF16 pairs 32
constexpr uint32_t TM_COLS = 512;

constexpr uint32_t ID_KQ = idesc_bf16(128, 64, false, false);
constexpr uint32_t ID_WT = idesc_bf16(128, 64, true, false);        // A = K^T / V^T (MN-major)
constexpr uint32_t ID_DT = idesc_bf16(128, 64, false, true, true);  // -S W^T, B MN-major
constexpr uint32_t ID_SQ = idesc_bf16(128, 64, false, false);
constexpr uint32_t ID_SU = idesc_bf16(128, 128, false, true);       // B = K (MN-major)
constexpr uint32_t ID_OA = idesc_bf16(128, 64, false, false);

// mbarrier indices
enum {
  B_KQFULL = 0,    // [3] K/Q tiles + gate/beta of a stage landed (33 arrivals + tx)
  B_KQEMPTY = 3,   // [3] stage free again (MMA commit after the chunk's state update)
  B_VFULL = 6,     // [2]
  B_VEMPTY = 8,    // [2] (MMA commit after U^T)
  B_KQREADY = 10,  // prep: padded rows zeroed, decay vectors written
  B_KQDONE = 11,   // MMA: KQ complete
  B_KQFREE = 12,   // prep: KQ accumulator read
  B_QG = 13,       // [3] prep: Q rows of a stage scaled by e^gamma
  B_TTREADY = 16,  // prep: T', T'', Ahat written
  B_WTDONE = 17,   // MMA: W^T and U^T complete
  B_WTREADY = 18,  // prep: W^T tile written
  B_DTDONE = 19,   // MMA: Delta^T complete
  B_DREADY = 20,   // state: Delta BF16 operands in TMEM
  B_SUDONE = 21,   // MMA: state update complete
  B_SREADY = 22,   // state: S BF16 operand and e^{gamma_C}-scaled S in TMEM
  B_ODONE = 23,    // MMA: O complete
  B_OFREE = 24,    // out: O read
  B_AHFREE = 25,   // [2] MMA: Ahat buffer free (commit after O += Delta^T Ahat^T)
  B_VEC = 27,      // [3] prep: decay vectors of a stage written
  B_COUNT = 30
};
static_assert(B_COUNT * 8 + 8 <= 256, "barrier area");

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
  int mode;                 // TC_MODE_*
  const int32_t* bounds;    // summary: [R,2] token ranges
  float* P;                 // summary: [R,H,K,K]
  float* E;                 // summary: [R,H,V,K]
  float* ckpt;              // replay: [slots,H,V,K] chunk-entry states
  int R;
};

// Wait limit in SM clock cycles (about 2 s at the GB300's clocks).  The cycle
// counter is read instead of the global timer: it costs a few cycles, so the
// issuer's polling loop stays responsive.
constexpr long long kWaitLimitCycles = 4000000000ll;

__device__ __forceinline__ void raise_abort(volatile int* abort_flag, int* status) {
  *abort_flag = 1;
  atomicExch(status, 5 /* SF_ERR_TIMEOUT */);
}

// Bounded wait that also gives up when another role has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity,
                                              volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > kWaitLimitCycles) return false;
  }
}

// Every thread of a role (nthr threads on named barrier bar_id) waits, then they
// agree on the outcome.
__device__ __forceinline__ bool wg_wait(uint64_t* bar, uint32_t parity, int bar_id,
                                        volatile int* abort_flag, int* status, int nthr = 128) {
  const bool ok = named_bar_and(bar_id, nthr, wait_or_abort(bar, parity, abort_flag));
  if (!ok && (threadIdx.x & (nthr - 1)) == 0) raise_abort(abort_flag, status);
  return ok;
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          int* status) {
  const bool ok = __all_sync(0xffffffffu, wait_or_abort(bar, parity, abort_flag)) != 0;
  if (!ok && (threadIdx.x & 31) == 0) raise_abort(abort_flag, status);
  return ok;
}

constexpr int PREP_THREADS = 256;   // warps 8-15
struct PrepBar {
  __device__ __forceinline__ void operator()() const { named_bar(BAR_PREP, PREP_THREADS); }
};

__device__ __forceinline__ int chunk_len(int64_t bos, int64_t eos, int c) {
  const int64_t r = eos - (bos + (int64_t)c * CHUNK);
  return (int)(r < CHUNK ? r : CHUNK);
}

__global__ void __launch_bounds__(NTHR, 1)
    gdn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(sm);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_BAR + B_COUNT * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* vecs = reinterpret_cast<float*>(sm + OFF_VEC);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = p.H;
  // Work item.  FWD / REPLAY: one (sequence, head) chain.  SUMMARY: one (range,
  // head) pair; the first R*H CTAs build S_ext (zero entry state, value term on),
  // the next R*H build P (identity entry state, value term off) -- the probing
  // construction of the Attention Gym "Context Parallelism" section.
  int n, h;
  int64_t bos = 0, eos = 0;
  bool valid = true, value_on = true;
  const bool has_out = (p.mode == TC_MODE_FWD);
  int init_kind = p.s0 ? 1 : 0;              // 0: zero, 1: initial state, 2: identity
  float* final_dst = (p.mode == TC_MODE_FWD) ? p.final_state : nullptr;
  if (p.mode == TC_MODE_SUMMARY) {
    const int per = p.R * H;
    const bool second = (int)blockIdx.x >= per;
    const int bx = (int)blockIdx.x - (second ? per : 0);
    n = bx / H;
    h = bx % H;
    const int64_t total = (int64_t)p.B * p.T;
    const int64_t r0 = p.bounds[2 * n], r1 = p.bounds[2 * n + 1];
    valid = (r0 >= 0 && r1 >= r0 && r1 <= total && (r1 == r0 || r0 / p.T == (r1 - 1) / p.T));
    if (valid) {
      bos = r0;
      eos = r1;
    }
    value_on = !second;
    init_kind = second ? 2 : 0;
    final_dst = second ? p.P : p.E;
  } else {
    n = blockIdx.x / H;
    h = blockIdx.x % H;
    seq_span(n, p.B, p.T, p.cu, bos, eos);
  }
  const int nc = (int)((eos - bos + CHUNK - 1) / CHUNK);
  const size_t state_off = ((size_t)n * H + h) * D * D;

  if (tid == 0) {
    for (int i = 0; i < B_COUNT; ++i) mbar_init(&bars[i], 1);
    for (int s = 0; s < (int)KQ_STAGES; ++s) mbar_init(&bars[B_KQFULL + s], 33);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tmem_slot;

  // Roles, each with its own register budget (launch: 128 per thread = the whole
  // register file; budgets sum to 512 x 128 threads = 65536):
  // loader/issuer 56, state (+ output stores) 136, prep (two warpgroups) 160.
  if (warp < 4) {
   reg_dealloc<56>();
   if (warp == 0) {
    // ------------------------------------------------------------- loader
    int last_kq[KQ_STAGES] = {-1, -1, -1}, last_v[V_STAGES] = {-1, -1};
    for (int c = 0; c < nc; ++c) {
      const int s = c % KQ_STAGES, sv = c & 1;
      const int64_t c0 = bos + (int64_t)c * CHUNK;
      const int L = chunk_len(bos, eos, c);
      if (c >= (int)KQ_STAGES &&
          !warp_wait(&bars[B_KQEMPTY + s], (uint32_t)((c - KQ_STAGES) / KQ_STAGES) & 1u, abort_flag,
                     p.status))
        break;
      if (lane == 0) {
        uint8_t* kq = sm + OFF_KQ + s * KQ_STAGE;
        mbar_arrive_expect_tx(&bars[B_KQFULL + s], (has_out ? 4 : 2) * 8192);
#pragma unroll
        for (int pnl = 0; pnl < 2; ++pnl) {
          tma_load_3d(kq + pnl * KQ_PANEL, &tmK, &bars[B_KQFULL + s], 64 * pnl, h, (int)c0);
          if (has_out)
            tma_load_3d(kq + pnl * KQ_PANEL + 8192, &tmQ, &bars[B_KQFULL + s], 64 * pnl, h,
                        (int)c0);
        }
      }
      last_kq[s] = c;
      float* vs = vecs + s * 512;
#pragma unroll
      for (int e = lane; e < 64; e += 32) {
        const size_t off = (size_t)(c0 + e) * H + h;
        vs[VEC_G + e] = (e < L) ? p.g[off] : 0.f;
        vs[VEC_BETA + e] = (e < L) ? p.beta[off] : 0.f;
      }
      mbar_arrive(&bars[B_KQFULL + s]);
      if (!value_on) continue;
      if (c >= (int)V_STAGES &&
          !warp_wait(&bars[B_VEMPTY + sv], (uint32_t)((c - V_STAGES) >> 1) & 1u, abort_flag,
                     p.status))
        break;
      if (lane == 0) {
        uint8_t* vt = sm + OFF_V + sv * V_STAGE;
        mbar_arrive_expect_tx(&bars[B_VFULL + sv], 2 * 8192);
#pragma unroll
        for (int pnl = 0; pnl < 2; ++pnl)
          tma_load_3d(vt + pnl * V_PANEL, &tmV, &bars[B_VFULL + sv], 64 * pnl, h, (int)c0);
      }
      last_v[sv] = c;
    }
    // never leave with a tile copy in flight
    for (int s = 0; s < (int)KQ_STAGES; ++s)
      if (last_kq[s] >= 0)
        mbar_wait(&bars[B_KQFULL + s], (uint32_t)(last_kq[s] / KQ_STAGES) & 1u, 100000000ull);
    for (int s = 0; s < (int)V_STAGES; ++s)
      if (last_v[s] >= 0) mbar_wait(&bars[B_VFULL + s], (uint32_t)(last_v[s] >> 1) & 1u, 100000000ull);
    __syncwarp();
   } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0 && nc > 0) {
      int nKQ = 0, nWU = 0, nDT = 0, nSQ = 0, nSU = 0;
      long long t_prog = clock64();
      while (nSU < nc) {
        bool prog = false;
        // state transition: Delta^T += -S W^T
        if (nDT < nWU && mbar_test(&bars[B_WTREADY], nDT & 1) &&
            mbar_test(&bars[B_SREADY], nDT & 1)) {
          tc_fence_after();
          const uint64_t bd = sdesc_sw128(sb + OFF_WT, 16384, 1024);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_bf16_ta(tm + TM_DT, tm + TM_SB + kk * 8, bd + (uint64_t)(kk * 2048 >> 4), ID_DT,
                        (value_on || kk > 0) ? 1u : 0u);
          mma_commit(&bars[B_DTDONE]);
          ++nDT;
          prog = true;
        }
        // output, state part: O = S Qg^T
        if (has_out && nSQ < nDT && mbar_test(&bars[B_QG + nSQ % KQ_STAGES], (nSQ / KQ_STAGES) & 1) &&
            (nSQ == 0 || mbar_test(&bars[B_OFREE], (nSQ - 1) & 1))) {
          tc_fence_after();
          const uint32_t kqa = sb + OFF_KQ + (nSQ % KQ_STAGES) * KQ_STAGE;
          const uint64_t bd = sdesc_sw128(kqa + 8192, 0, 1024);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_bf16_ta(tm + TM_O, tm + TM_SB + kk * 8,
                        bd + (uint64_t)(((kk >> 2) * KQ_PANEL + (kk & 3) * 32) >> 4), ID_SQ, kk > 0);
          ++nSQ;
          prog = true;
        }
        // state update S += (Delta^T diag(dec)) K, then O += Delta^T Ahat^T
        if (nSU < (has_out ? nSQ : nDT) && mbar_test(&bars[B_DREADY], nSU & 1)) {
          tc_fence_after();
          const int s = nSU % KQ_STAGES;
          const uint32_t kqa = sb + OFF_KQ + s * KQ_STAGE;
          const uint64_t bk = sdesc_sw128(kqa, KQ_PANEL, 1024);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16_ta(tm + TM_S, tm + TM_DDB + kk * 8, bk + (uint64_t)(kk * 2048 >> 4), ID_SU, 1);
          mma_commit(&bars[B_SUDONE]);
          mma_commit(&bars[B_KQEMPTY + s]);
          if (has_out) {
            const uint32_t ah = sb + OFF_AH + (nSU & 1) * 8192;
            const uint64_t ba = sdesc_sw128(ah, 0, 1024);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_bf16_ta(tm + TM_O, tm + TM_DB + kk * 8, ba + (uint64_t)(kk * 2), ID_OA, 1);
            mma_commit(&bars[B_ODONE]);
            mma_commit(&bars[B_AHFREE + (nSU & 1)]);
          }
          ++nSU;
          prog = true;
        }
        // prep products of chunk nWU: W^T and U^T (U^T needs the Delta^T accumulator free)
        if (nWU < nKQ && nSU >= nWU && mbar_test(&bars[B_TTREADY], nWU & 1)) {
          tc_fence_after();
          const uint32_t kqa = sb + OFF_KQ + (nWU % KQ_STAGES) * KQ_STAGE;
          const uint32_t va = sb + OFF_V + (nWU & 1) * V_STAGE;
          const uint64_t ak = sdesc_sw128(kqa, KQ_PANEL, 1024), b2 = sdesc_sw128(sb + OFF_T2, 0, 1024);
          const uint64_t av = sdesc_sw128(va, V_PANEL, 1024), b1 = sdesc_sw128(sb + OFF_T1, 0, 1024);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16(tm + TM_WT, ak + (uint64_t)(kk * 2048 >> 4), b2 + (uint64_t)(kk * 2), ID_WT, kk > 0);
          if (value_on) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_bf16(tm + TM_DT, av + (uint64_t)(kk * 2048 >> 4), b1 + (uint64_t)(kk * 2), ID_WT,
                       kk > 0);
          }
          mma_commit(&bars[B_WTDONE]);
          if (value_on) mma_commit(&bars[B_VEMPTY + (nWU & 1)]);
          ++nWU;
          prog = true;
        }
        // prep product of chunk nKQ: [K; Q] K^T
        if (nKQ < nc && mbar_test(&bars[B_KQREADY], nKQ & 1) &&
            (nKQ == 0 || mbar_test(&bars[B_KQFREE], (nKQ - 1) & 1))) {
          tc_fence_after();
          const uint32_t kqa = sb + OFF_KQ + (nKQ % KQ_STAGES) * KQ_STAGE;
          const uint64_t bq = sdesc_sw128(kqa, 0, 1024);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t d = bq + (uint64_t)(((kk >> 2) * KQ_PANEL + (kk & 3) * 32) >> 4);
            mma_bf16(tm + TM_KQ, d, d, ID_KQ, kk > 0);
          }
          mma_commit(&bars[B_KQDONE]);
          ++nKQ;
          prog = true;
        }
        if (prog) {
          t_prog = clock64();
        } else if (*abort_flag || clock64() - t_prog > kWaitLimitCycles) {
          raise_abort(abort_flag, p.status);
          break;
        }
      }
    }
    __syncwarp();
   }
  } else if (warp < 8) {
    reg_alloc<136>();
    // --------------------------------------------------------------- state
    const int v = tid - 128;                         // TMEM lane = state row
    const uint32_t tl = tm + ((uint32_t)((warp & 3) * 32) << 16);
    bool ok = true;
    // entry state row v, 4 consecutive columns starting at c
    auto init4 = [&](int c) -> float4 {
      if (init_kind == 1)
        return *reinterpret_cast<const float4*>(p.s0 + state_off + (size_t)v * D + c);
      if (init_kind == 2)
        return make_float4(v == c ? 1.f : 0.f, v == c + 1 ? 1.f : 0.f, v == c + 2 ? 1.f : 0.f,
                           v == c + 3 ? 1.f : 0.f);
      return make_float4(0.f, 0.f, 0.f, 0.f);
    };
    // replay: chunk-entry states go to ckpt[slot][h] (unscaled FP32)
    float* ckpt = (p.mode == TC_MODE_REPLAY)
                      ? p.ckpt + ((size_t)chunk_slot_base(n, p.B, p.T, p.cu) * H + h) * D * D +
                            (size_t)v * D
                      : nullptr;
    const size_t ckpt_stride = (size_t)H * D * D;
    if (nc == 0) {
      if (final_dst) {
        const float nanv = __int_as_float(0x7fc00000);
        for (int c = 0; c < D; c += 4)
          *reinterpret_cast<float4*>(final_dst + state_off + (size_t)v * D + c) =
              valid ? init4(c) : make_float4(nanv, nanv, nanv, nanv);
      }
    } else {
      ok = wg_wait(&bars[B_VEC + 0], 0, BAR_STATE, abort_flag, p.status);
      if (ok) {
        const float g0 = vecs[VEC_EG + 63];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          float x[32];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float4 t = init4(32 * cc + 4 * e);
            x[4 * e] = t.x; x[4 * e + 1] = t.y; x[4 * e + 2] = t.z; x[4 * e + 3] = t.w;
          }
          if (ckpt) {
            float4* dst = reinterpret_cast<float4*>(ckpt + 32 * cc);
#pragma unroll
            for (int e = 0; e < 8; ++e)
              dst[e] = make_float4(x[4 * e], x[4 * e + 1], x[4 * e + 2], x[4 * e + 3]);
          }
          uint32_t u[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) u[e] = pack_bf16x2(x[2 * e], x[2 * e + 1]);
          tmem_st16(tl + TM_SB + 16 * cc, u);
#pragma unroll
          for (int e = 0; e < 32; ++e) x[e] *= g0;
          tmem_st32(tl + TM_S + 32 * cc, x);
        }
        tmem_st_wait();
        tc_fence_before();
        named_bar(BAR_STATE, 128);
        if (v == 0) mbar_arrive(&bars[B_SREADY]);
      }
      for (int c = 0; c < nc && ok; ++c) {
        const float* vs = vecs + (c % KQ_STAGES) * 512;
        if (!(ok = wg_wait(&bars[B_DTDONE], c & 1, BAR_STATE, abort_flag, p.status))) break;
        tc_fence_after();
        {
          float x[64];
          tmem_ld32(tl + TM_DT, *reinterpret_cast<float(*)[32]>(x));
          tmem_ld32(tl + TM_DT + 32, *reinterpret_cast<float(*)[32]>(x + 32));
          tmem_ld_wait();
          uint32_t u[16];
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
            for (int e = 0; e < 16; ++e) u[e] = pack_bf16x2(x[32 * hh + 2 * e], x[32 * hh + 2 * e + 1]);
            tmem_st16(tl + TM_DB + 16 * hh, u);
          }
          const float4* dec4 = reinterpret_cast<const float4*>(vs + VEC_DEC);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float4 d4 = dec4[8 * hh + e];
              u[2 * e] = pack_bf16x2(x[32 * hh + 4 * e] * d4.x, x[32 * hh + 4 * e + 1] * d4.y);
              u[2 * e + 1] = pack_bf16x2(x[32 * hh + 4 * e + 2] * d4.z, x[32 * hh + 4 * e + 3] * d4.w);
            }
            tmem_st16(tl + TM_DDB + 16 * hh, u);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        named_bar(BAR_STATE, 128);
        if (v == 0) mbar_arrive(&bars[B_DREADY]);
        if (!(ok = wg_wait(&bars[B_SUDONE], c & 1, BAR_STATE, abort_flag, p.status))) break;
        tc_fence_after();
        const bool last = (c + 1 == nc);
        float gn = 0.f;
        if (!last) {
          if (!(ok = wg_wait(&bars[B_VEC + (c + 1) % KQ_STAGES], ((c + 1) / KQ_STAGES) & 1,
                             BAR_STATE, abort_flag, p.status)))
            break;
          gn = vecs[((c + 1) % KQ_STAGES) * 512 + VEC_EG + 63];
        }
#pragma unroll
        for (int cp = 0; cp < 2; ++cp) {
          float x[64];
          tmem_ld32(tl + TM_S + 64 * cp, *reinterpret_cast<float(*)[32]>(x));
          tmem_ld32(tl + TM_S + 64 * cp + 32, *reinterpret_cast<float(*)[32]>(x + 32));
          tmem_ld_wait();
          if (!last) {
            if (ckpt) {
              float4* dst = reinterpret_cast<float4*>(ckpt + (size_t)(c + 1) * ckpt_stride + 64 * cp);
#pragma unroll
              for (int e = 0; e < 16; ++e)
                dst[e] = make_float4(x[4 * e], x[4 * e + 1], x[4 * e + 2], x[4 * e + 3]);
            }
            uint32_t u[16];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
              for (int e = 0; e < 16; ++e) u[e] = pack_bf16x2(x[32 * hh + 2 * e], x[32 * hh + 2 * e + 1]);
              tmem_st16(tl + TM_SB + 32 * cp + 16 * hh, u);
            }
#pragma unroll
            for (int e = 0; e < 64; ++e) x[e] *= gn;
            tmem_st32(tl + TM_S + 64 * cp, *reinterpret_cast<float(*)[32]>(x));
            tmem_st32(tl + TM_S + 64 * cp + 32, *reinterpret_cast<float(*)[32]>(x + 32));
          } else if (final_dst) {
            float4* dst =
                reinterpret_cast<float4*>(final_dst + state_off + (size_t)v * D + 64 * cp);
#pragma unroll
            for (int e = 0; e < 16; ++e)
              dst[e] = make_float4(x[4 * e], x[4 * e + 1], x[4 * e + 2], x[4 * e + 3]);
          }
        }
        if (!last) {
          tmem_st_wait();
          tc_fence_before();
          named_bar(BAR_STATE, 128);
          if (v == 0) mbar_arrive(&bars[B_SREADY]);
        }
        if (has_out) {
          // out[i][v] = scale O[v][i]: one warp writes 32 consecutive v of a token row
          if (!(ok = wg_wait(&bars[B_ODONE], c & 1, BAR_STATE, abort_flag, p.status))) break;
          tc_fence_after();
          float a[64];
          tmem_ld32(tl + TM_O, *reinterpret_cast<float(*)[32]>(a));
          tmem_ld32(tl + TM_O + 32, *reinterpret_cast<float(*)[32]>(a + 32));
          tmem_ld_wait();
          tc_fence_before();
          named_bar(BAR_STATE, 128);
          if (v == 0) mbar_arrive(&bars[B_OFREE]);
          const int64_t c0 = bos + (int64_t)c * CHUNK;
          const int L = chunk_len(bos, eos, c);
          __nv_bfloat16* orow = p.out + ((size_t)c0 * H + h) * D + v;
          const size_t rs = (size_t)H * D;
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (i < L) orow[i * rs] = __float2bfloat16_rn(p.scale * a[i]);
        }
      }
    }
  } else {
    reg_alloc<160>();
    // ---------------------------------------------------------------- prep
    // Warps 8-15 prepare the chunk ahead.  Order per chunk c: [KQ(c) epilogue ->
    // release KQ] [head of chunk c+1, so its KQ product runs during this chunk's
    // solve] [solve(c), T', T''] [W^T tile].  A thread owns TMEM row `lrow` and the
    // column half `half` of it.
    const int pt = tid - 256;                        // 0..255
    const int half = pt >> 7;
    const int lrow = ((warp & 3) << 5) + lane;
    const uint32_t tl = tm + ((uint32_t)((warp & 3) * 32) << 16);
    float* AT = reinterpret_cast<float*>(sm + OFF_AT);
    float* X = reinterpret_cast<float*>(sm + OFF_X);
    // head: the chunk's tiles have landed -> zero padded rows, gamma and decay vectors
    auto head = [&](int c) -> bool {
      const int s = c % KQ_STAGES, sv = c & 1;
      const int L = chunk_len(bos, eos, c);
      float* vs = vecs + s * 512;
      if (!wg_wait(&bars[B_KQFULL + s], (c / KQ_STAGES) & 1, BAR_PREP, abort_flag, p.status,
                   PREP_THREADS))
        return false;
      if (value_on && !wg_wait(&bars[B_VFULL + sv], (c >> 1) & 1, BAR_PREP, abort_flag, p.status,
                               PREP_THREADS))
        return false;
      if (L < CHUNK) {
        // rows past the sequence end belong to the next sequence (or are past
        // the tensor): zero them so they contribute nothing to any product
        uint8_t* kq = sm + OFF_KQ + s * KQ_STAGE;
        uint8_t* vt = sm + OFF_V + sv * V_STAGE;
        const int rows = CHUNK - L;
        for (int idx = pt; idx < (value_on ? 6 : 4) * rows * 8; idx += PREP_THREADS) {
          const int t6 = idx / (rows * 8), rem = idx % (rows * 8);
          const int r = L + rem / 8, ch = rem % 8;
          const int pnl = t6 & 1, which = t6 >> 1;
          uint8_t* base = (which == 2) ? vt + pnl * V_PANEL
                                       : kq + pnl * KQ_PANEL + (which == 1 ? 8192u : 0u);
          *reinterpret_cast<uint4*>(base + r * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
      }
      if (pt < 32) {
        warp_cumsum64(vs + VEC_G, vs + VEC_GAM, lane);
        __syncwarp();
        const float a0 = vs[VEC_GAM + 2 * lane], a1 = vs[VEC_GAM + 2 * lane + 1];
        float mx = fmaxf(a0, a1), mn = fminf(a0, a1);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
          mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        }
        // decay factors: e^{gamma_i - gamma_j} = e^{gamma_i - mid} e^{mid - gamma_j} when
        // the chunk's gamma range keeps both factors inside e^{+-40}; else one
        // exponential per entry
        if (lane == 0) {
          vs[VEC_FLAG] = (mx - mn) <= 80.f ? 1.f : 0.f;
          vs[VEC_FLAG + 1] = 0.5f * (mx + mn);
        }
      }
      named_bar(BAR_PREP, PREP_THREADS);
      if (pt < 64) {
        const bool fact = vs[VEC_FLAG] != 0.f;
        const float mid = vs[VEC_FLAG + 1], gi = vs[VEC_GAM + pt], gC = vs[VEC_GAM + 63];
        vs[VEC_EG + pt] = expf(gi);
        vs[VEC_DEC + pt] = expf(gC - gi);
        vs[VEC_EP + pt] = fact ? expf(gi - mid) : 0.f;
        vs[VEC_EM + pt] = fact ? expf(mid - gi) : 0.f;
      }
      named_bar(BAR_PREP, PREP_THREADS);
      if (pt == 0) {
        mbar_arrive(&bars[B_KQREADY]);
        mbar_arrive(&bars[B_VEC + s]);
      }
      return true;
    };
    bool ok = nc > 0 ? head(0) : true;
    for (int c = 0; c < nc && ok; ++c) {
      const int s = c % KQ_STAGES;
      float* vs = vecs + s * 512;
      uint8_t* kq = sm + OFF_KQ + s * KQ_STAGE;
      if (has_out && c >= 2 &&
          !(ok = wg_wait(&bars[B_AHFREE + (c & 1)], ((c - 2) >> 1) & 1, BAR_PREP, abort_flag,
                         p.status, PREP_THREADS)))
        break;
      if (!(ok = wg_wait(&bars[B_KQDONE], c & 1, BAR_PREP, abort_flag, p.status, PREP_THREADS)))
        break;
      tc_fence_after();
      {
        const bool fact = vs[VEC_FLAG] != 0.f;
        const int i = lrow & 63, j0 = 32 * half;
        const float gi = vs[VEC_GAM + i], epi = vs[VEC_EP + i];
        const float bi = (lrow < 64) ? vs[VEC_BETA + i] : 1.f;
        float x[32];
        tmem_ld32(tl + TM_KQ + j0, x);
        tmem_ld_wait();
        if (fact) {
          const float f = bi * epi;
          const float4* em4 = reinterpret_cast<const float4*>(vs + VEC_EM + j0);
#pragma unroll
          for (int j4 = 0; j4 < 8; ++j4) {
            const float4 e4 = em4[j4];
            x[4 * j4] *= f * e4.x;
            x[4 * j4 + 1] *= f * e4.y;
            x[4 * j4 + 2] *= f * e4.z;
            x[4 * j4 + 3] *= f * e4.w;
          }
        } else {
#pragma unroll
          for (int jj = 0; jj < 32; ++jj)
            x[jj] *= bi * expf(j0 + jj <= i ? gi - vs[VEC_GAM + j0 + jj] : 0.f);
        }
        if (lrow < 64) {       // A_ij = beta_i Gamma_ij (k_i . k_j), j < i
          float4* row = reinterpret_cast<float4*>(AT + i * SOLVE_LD + j0);
#pragma unroll
          for (int j4 = 0; j4 < 8; ++j4) {
            const int j = j0 + 4 * j4;
            row[j4] = make_float4(j < i ? x[4 * j4] : 0.f, j + 1 < i ? x[4 * j4 + 1] : 0.f,
                                  j + 2 < i ? x[4 * j4 + 2] : 0.f, j + 3 < i ? x[4 * j4 + 3] : 0.f);
          }
        } else if (has_out) {  // Ahat_ij = Gamma_ij (q_i . k_j), j <= i
          uint8_t* ah = sm + OFF_AH + (c & 1) * 8192;
#pragma unroll
          for (int jj = 0; jj < 32; ++jj)
            if (j0 + jj > i) x[jj] = 0.f;
#pragma unroll
          for (int e = 0; e < 4; ++e) st_row8_bf16(ah, i, j0 + 8 * e, 8192, x + 8 * e);
        }
      }
      tc_fence_before();
      // Q rows scaled by e^{gamma_i} in place (the KQ product has consumed them): O's
      // state part S (diag(e^gamma) Q)^T then shares one accumulator with Delta^T Ahat^T
      for (int idx = pt; has_out && idx < 64 * 2 * 8; idx += PREP_THREADS) {
        const int r = idx >> 4, pnl = (idx >> 3) & 1, ch = idx & 7;
        uint4* ptr = reinterpret_cast<uint4*>(kq + pnl * KQ_PANEL + 8192 + r * 128 + ch * 16);
        const float e = vs[VEC_EG + r];
        uint4 w = *ptr;
        uint32_t* wu = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
        for (int q2 = 0; q2 < 4; ++q2) {
          __nv_bfloat162 b2 = *reinterpret_cast<__nv_bfloat162*>(&wu[q2]);
          float2 f = __bfloat1622float2(b2);
          wu[q2] = pack_bf16x2(f.x * e, f.y * e);
        }
        *ptr = w;
      }
      fence_proxy_async_smem();
      named_bar(BAR_PREP, PREP_THREADS);
      if (pt == 0) {
        mbar_arrive(&bars[B_KQFREE]);
        mbar_arrive(&bars[B_QG + s]);
      }
      if (c + 1 < nc && !(ok = head(c + 1))) break;
      // T = (I + A)^{-1}, then T' = T diag(beta), T'' = T diag(beta e^gamma)
      solve64_tc_inplace(AT, X, pt, PREP_THREADS, PrepBar());
      for (int idx = pt; idx < 64 * 8; idx += PREP_THREADS) {
        const int i = idx >> 3, cg = (idx & 7) * 8;
        const float4* tr = reinterpret_cast<const float4*>(AT + i * SOLVE_LD + cg);
        const float4* b4 = reinterpret_cast<const float4*>(vs + VEC_BETA + cg);
        const float4* g4 = reinterpret_cast<const float4*>(vs + VEC_EG + cg);
        float t1[8], t2[8];
#pragma unroll
        for (int h4 = 0; h4 < 2; ++h4) {
          const float4 t = tr[h4], b = b4[h4], g = g4[h4];
          t1[4 * h4] = t.x * b.x; t1[4 * h4 + 1] = t.y * b.y;
          t1[4 * h4 + 2] = t.z * b.z; t1[4 * h4 + 3] = t.w * b.w;
          t2[4 * h4] = t1[4 * h4] * g.x; t2[4 * h4 + 1] = t1[4 * h4 + 1] * g.y;
          t2[4 * h4 + 2] = t1[4 * h4 + 2] * g.z; t2[4 * h4 + 3] = t1[4 * h4 + 3] * g.w;
        }
        st_row8_bf16(sm + OFF_T1, i, cg, 8192, t1);
        st_row8_bf16(sm + OFF_T2, i, cg, 8192, t2);
      }
      fence_proxy_async_smem();
      named_bar(BAR_PREP, PREP_THREADS);
      if (pt == 0) mbar_arrive(&bars[B_TTREADY]);
      if (!(ok = wg_wait(&bars[B_WTDONE], c & 1, BAR_PREP, abort_flag, p.status, PREP_THREADS)))
        break;
      tc_fence_after();
      {
        float x[32];
        tmem_ld32(tl + TM_WT + 32 * half, x);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 4; ++e)
          st_row8_bf16(sm + OFF_WT, lrow, 32 * half + 8 * e, 16384, x + 8 * e);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      named_bar(BAR_PREP, PREP_THREADS);
      if (pt == 0) mbar_arrive(&bars[B_WTREADY]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
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

bool make_bf16_map(CUtensorMap* m, const void* base, int rows, int H) {
  return make_map(m, base, rows, H);
}

cudaError_t launch_tc(const ChainParams& cp, int mode, int* status, cudaStream_t st) {
  const int rows = cp.B * cp.T;
  if (rows <= 0) return cudaErrorInvalidValue;
  CUtensorMap mq, mk, mv;
  // without an output the query tiles are never loaded; the K map stands in
  const void* qsrc = (mode == TC_MODE_FWD) ? cp.q : cp.k;
  if (!make_map(&mq, qsrc, rows, cp.H) || !make_map(&mk, cp.k, rows, cp.H) ||
      !make_map(&mv, cp.v, rows, cp.H))
    return cudaErrorInvalidValue;
  TcParams p{};
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
  p.mode = mode;
  p.bounds = cp.bounds;
  p.P = cp.P;
  p.E = cp.E;
  p.ckpt = cp.ckpt;
  p.R = cp.N;
  cudaError_t e = cudaFuncSetAttribute(gdn_fwd_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  const int ctas = (mode == TC_MODE_SUMMARY ? 2 : 1) * cp.N * cp.H;
  if (ctas > 0) gdn_fwd_tc_kernel<<<ctas, NTHR, SMEM_ALLOC, st>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace sfg
