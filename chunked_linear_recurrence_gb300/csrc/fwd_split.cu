// fwd_split.cu -- forward of the chunked gated delta rule for dense BF16 q/k/v with
// K = V = 128 on sm_103a, split across the GPU by role.
//
// The per-chunk work of the chunk-parallel form (StateFlow section 2.2, Eq. 2) has
// two parts with very different shapes:
//   Pre  (fully parallel over chunks): the decays, [K;Q] K^T, the triangular solve
//        T = (I + A)^{-1}, and the factors W = T diag(beta e^gamma) K,
//        T' = T diag(beta), Ahat = M o Gamma o Q K^T;
//   ST + Out (serial along a chain): Delta = U - W S^T with U = T' V,
//        O = diag(e^gamma) Q S^T + Ahat Delta, S <- e^{gamma_C} S + Delta^T diag(dec) K.
// One cooperative persistent launch gives each kind its own SMs.  The first `nch`
// CTAs are state-chain CTAs, each owning a fixed list of (sequence, head) chains and
// walking their chunks in order; the other CTAs are preparation CTAs that turn
// chunks into "records" (the chunk's factors as ready-made BF16 tensor-core tiles) in
// the order the chains consume them, two chunks in flight per CTA.  Records pass
// through a per-chain-CTA ring of 8 or 16 slots in global memory (small enough to stay
// in L2); a slot's `ready` flag (release/acquire) hands it to the chain CTA, which
// copies it into shared memory with a bulk copy and hands the slot back through its
// `consumed` counter.  This is StateFlow's split of Pre from ST (section 3.4.2,
// Eq. 17: the next chunk's Pre overlaps the current ST) carried across SMs: the
// serial chain no longer waits on the preparation of its own chunks.
//
// Record of one chunk (BF16 tiles in the 128-byte-swizzled panel layout of tc_ptx.cuh):
//   (-W)^T [128 k][64 i]                        (B of D += S (-W)^T)
//   T'     [64 i][64 j]                         (B of U^T = V^T T'^T)
//   Ahat   [64 i][64 j]                         (B of O2 = Delta^T Ahat^T)
//   e^{gamma_C - gamma_j}, e^{gamma_i}, e^{gamma_C}  (FP32)
// The chain CTA loads the chunk's K, Q and V tiles itself (TMA; the preparation warmed
// them in L2) and forms the value and query terms on its own tensor pipe, off the serial
// path.  Chain products per chunk (all M = 128; S, Delta as BF16 A operands in TMEM):
//   D  = V^T T'^T (= U^T), then D += S (-W)^T    N = 64, K = 64 / 128   -> Delta^T
//   O1 = S Q^T                                    N = 64, K = 128  (while Delta is formed)
//   S <- e^{gamma_C} S + (Delta^T diag(dec)) K    N = 128, K = 64
//   O2 = Delta^T Ahat^T                           N = 64,  K = 64
//   out[i][v] = scale (e^{gamma_i} O1[v][i] + O2[v][i])
// Preparation products per chunk: KQ = [K;Q] K^T and (-W)^T = K^T (-T'')^T (N = 64),
// T' = T diag(beta), T'' = T diag(beta e^gamma), the 64x64 solve in FP32 with TF32 merges
// (solve::); the K/Q tiles are double-buffered so that the next chunk's KQ runs during
// the current chunk's solve.
//
// Segment summaries (the affine map S_out = S_in P + E of a token range) run on the same
// kernel: the chain from S0 = 0 with the value term gives E, the chain from S0 = I
// without it gives P (it multiplies S by e^{gamma_C} I - W^T diag(dec) K per chunk).  Each
// chunk's record -- (-W)^T, T' and the decays only -- is prepared once and read by two
// chain CTAs, j for E and nch + j for P; its ring slot is free when both have copied it.
//
// Every wait (mbarrier or global flag) is bounded; a CTA that gives up raises a
// global abort flag that every other CTA polls, writes SF_ERR_TIMEOUT to the status
// word, lets its own copies land, frees its TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "chunk_record.cuh"
#include "common.cuh"
#include "fwd_split.cuh"
#include "tmap.cuh"
#include "solve_tc.cuh"
#include "tc_ptx.cuh"

namespace sfg {
namespace {

using namespace tc;

constexpr int D = 128;
constexpr int NTHR = 512;
// Ring slots per chain CTA: a dense launch with output and one chain per chain CTA (its
// preparation has little slack, and 64 chain CTAs' rings of 8 stay in L2) takes
// NSLOT_OUT; the others (replay, summaries: preparation ahead, a deeper ring hides the
// hand-over latency; packed inputs and several chains per CTA: streams of different
// lengths) NSLOT_MAX, which the workspace always has room for.
constexpr int NSLOT_OUT = 8, NSLOT_MAX = 16;
constexpr int NBUF = 2;           // chunk buffers (record + K, Q, V tiles) of a chain CTA
constexpr int NBUF_NO = 3;        // the same without output (no Q tile): replay, summaries
constexpr int MAX_NCH = 64;       // chain CTAs that own record streams, at most
// Stream-owning chain CTAs of a segment-summary launch, at most (each with a P twin).  The
// summary's chains (two per (range, head), about 2 us per chunk step) and its preparation
// (about 6 us per record on each of a CTA's two pipelines) balance near 44 + 44 chain CTAs
// and 64 preparation CTAs on 152 SMs.
#ifndef SF_SUMMARY_CHAINS
#define SF_SUMMARY_CHAINS 44
#endif
static_assert(SF_SUMMARY_CHAINS >= 1 && SF_SUMMARY_CHAINS <= MAX_NCH, "summary chain CTAs");
constexpr int FLAG_STRIDE = 32;   // words between chain CTAs' flags: one 128-byte line each

// ---- record (global ring slot, and the chain CTA's shared-memory copy): chunk_record.cuh

// ---- state replay checkpoints: one BF16 [128 v][128 k] tile per chunk-head, two 64-column
// panels of 128 rows x 128 bytes, 16-byte chunk c of row v at ((c ^ (v mod 8)) << 4) (the
// layout the tensor-core gradient kernel reads as an operand) ----
constexpr uint32_t CKPT_TILE_BYTES = 32768;

// Row v of one panel of a checkpoint tile from the 64 values' BF16 pairs u.
__device__ __forceinline__ void store_ckpt_row(uint8_t* row, int v, const uint32_t (&u)[32]) {
#pragma unroll
  for (int c = 0; c < 8; ++c)
    *reinterpret_cast<uint4*>(row + ((c ^ (v & 7)) << 4)) =
        make_uint4(u[4 * c], u[4 * c + 1], u[4 * c + 2], u[4 * c + 3]);
}

// ---- chain CTA shared memory: NBUF buffers, each the record then the K, Q, V tiles, and
// two staging tiles of the output.  A launch without output has NBUF_NO buffers of the
// record's (-W)^T, T' and decays (no Ahat), K and V, and the staging of one checkpoint tile.
constexpr uint32_t C_K = 34816;       // K tile [64 tok][128 k]: 2 panels x 8 KB
constexpr uint32_t C_Q = 51200;       // Q tile, same layout
constexpr uint32_t C_V = 67584;       // V tile [64 tok][128 v]
constexpr uint32_t C_T_PANEL = 8192;
constexpr uint32_t C_BUF = 83968;     // buffer stride (1024-aligned)
constexpr uint32_t C_OST = NBUF * C_BUF;   // two staging tiles of the output [64 tok][128 v]
constexpr uint32_t C_VEC_NO = R_AH;   // no output: the decays where Ahat would be
constexpr uint32_t C_K_NO = C_VEC_NO + (REC_BYTES - R_VEC);
constexpr uint32_t C_V_NO = C_K_NO + 2 * C_T_PANEL;
constexpr uint32_t C_BUF_NO = C_V_NO + 2 * C_T_PANEL;
constexpr uint32_t C_CST = NBUF_NO * C_BUF_NO;   // checkpoint staging: 4 KB per state warp
constexpr uint32_t C_BAR_OUT = C_OST + 2 * 16384, C_BAR_NO = C_CST + CKPT_TILE_BYTES;
constexpr uint32_t C_BAR = C_BAR_OUT > C_BAR_NO ? C_BAR_OUT : C_BAR_NO;
static_assert(C_K >= REC_BYTES && C_K % 1024 == 0 && C_BUF % 1024 == 0, "chain smem");
static_assert(C_Q == C_K + 2 * C_T_PANEL && C_V == C_Q + 2 * C_T_PANEL &&
              C_BUF == C_V + 2 * C_T_PANEL, "chain tiles");
static_assert(R_W == 0 && R_T1 == 16384 && R_AH == 24576 && C_K_NO % 1024 == 0 &&
              C_BUF_NO % 1024 == 0, "chain smem without output");

// Buffers of a chain CTA with (kOut) or without output products.
template <bool kOut>
struct ChainBufs {
  static constexpr int NB = kOut ? NBUF : NBUF_NO;
  static constexpr uint32_t STRIDE = kOut ? C_BUF : C_BUF_NO;
  static constexpr uint32_t K = kOut ? C_K : C_K_NO;
  static constexpr uint32_t V = kOut ? C_V : C_V_NO;
  static constexpr uint32_t VEC = kOut ? R_VEC : C_VEC_NO;
};

// ---- preparation CTA shared memory, per pipeline (two pipelines) ----
constexpr uint32_t P_KQ = 0;          // two [K;Q] tile buffers: 2 panels x 16 KB each
constexpr uint32_t P_KQ_PANEL = 16384;  // (rows 0-63 K, 64-127 Q; pipeline 1: [Q;K])
constexpr uint32_t P_KQ_BUF = 32768;
constexpr uint32_t P_T1 = 65536;      // T'  [64 i][64 j]
constexpr uint32_t P_T2 = 73728;      // -T'' [64 i][64 j]
constexpr uint32_t P_AT = 81920;      // FP32 [64][SOLVE_LD]: A, then T
constexpr uint32_t P_X = 99328;       // staging of the Ahat rows (2 warps x 4 KB)
constexpr uint32_t P_VEC = 107520;    // 2 slots x 512 floats (items alternate)
constexpr uint32_t P_VEC_SLOT = 2048;
constexpr uint32_t P_STRIDE = 111616;
constexpr uint32_t P_BAR = 2 * P_STRIDE;
static_assert(P_T1 == P_KQ + 2 * P_KQ_BUF && P_T2 == P_T1 + 8192 && P_AT == P_T2 + 8192,
              "prep smem");
static_assert(P_AT + 64 * SOLVE_LD * 4 <= P_X && P_X + 2 * 4096 <= P_VEC, "prep smem");
static_assert(P_VEC + 2 * P_VEC_SLOT <= P_STRIDE && P_STRIDE % 1024 == 0, "prep smem");
static_assert(64 * SOLVE_LD * 4 >= 4 * 4096, "the A/T area doubles as the store staging area");

// Registers per thread after setmaxnreg, by role.  Each CTA is launched with 128 per
// thread (512 threads, the SM's 64K), and the roles' shares must add up to no more.
constexpr int RC_CTL = 56, RC_STATE = 168, RC_OUT = 120;        // chain: 4, 8, 4 warps
constexpr int RP_CTL = 96, RP_PIPE = 192, RP_AUX = 32;          // preparation: 4, 8, 4 warps
static_assert(4 * RC_CTL + 8 * RC_STATE + 4 * RC_OUT <= 16 * 128, "chain register split");
static_assert(4 * RP_CTL + 8 * RP_PIPE + 4 * RP_AUX <= 16 * 128, "preparation register split");

constexpr uint32_t BAR_BYTES = 512;
// packed inputs: stream lengths and their order (2 x 64 ints), then the production-order
// table (65 stream positions as ints, 65 record counts as long longs)
constexpr uint32_t GEO_BYTES = 2 * 64 * 4 + 65 * 4 + 4 + 65 * 8;
constexpr uint32_t SMEM_USED = (P_BAR > C_BAR ? P_BAR : C_BAR) + BAR_BYTES + GEO_BYTES;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;
static_assert(SMEM_ALLOC <= 232448, "shared memory");

// per-pipeline vectors (floats)
constexpr int VEC_BETA = 64, VEC_GAM = 128, VEC_EG = 192, VEC_DEC = 256,
              VEC_EP = 320, VEC_EM = 384, VEC_FLAG = 448,
              VEC_ITEM = 450;   // the use's item, -1: no more items; then its chain CTA and
                                // stream position (ints)

// ---- TMEM columns ----
// chain: S FP32, S BF16 pairs, Delta^T BF16 pairs, Delta^T diag(dec) BF16 pairs, the
// Delta accumulator (U^T - S W^T), O1 = S Q^T and O2 = Delta^T Ahat^T.
constexpr uint32_t TM_S = 0, TM_SB = 128, TM_DB = 192, TM_DDB = 224, TM_D = 256,
                   TM_O1 = 320, TM_O2 = 384;
// preparation, per pipeline p at 256 p: [K;Q] K^T and (-W)^T
constexpr uint32_t TP_KQ = 0, TP_WT = 64;
constexpr uint32_t TM_COLS = 512;

constexpr uint32_t ID_N64 = idesc_bf16(128, 64, false, false);   // both K-major
constexpr uint32_t ID_AMN = idesc_bf16(128, 64, true, false);    // A MN-major (X^T from a tile)
constexpr uint32_t ID_MG = idesc_bf16(128, 128, false, true);    // A@tmem, B MN-major, N = 128
constexpr uint32_t ID_MG64 = idesc_bf16(128, 64, false, true);   // the same, N = 64

// ---- mbarriers ----
enum {
  // chain CTA
  C_RECFULL = 0,   // [3] the chunk's record and tiles in shared memory (tx, or the
                   //     loader's arrival once a partial chunk's rows are zeroed)
  C_RECFREE = 3,   // [3] the chunk's last product done (MMA commit) + its output tile out
  C_LANDED = 6,    // [3] a partial chunk's copies landed (tx)
  C_MERGED = 9,    // MMA: Delta accumulator U^T - S W^T complete
  C_DREADY = 10,   // state: Delta BF16 operands in TMEM
  C_SUDONE = 11,   // MMA: state update complete (and O1 of the chunk)
  C_SREADY = 12,   // state: S BF16 operand in TMEM
  C_SSCALED = 13,  // state: TMEM S scaled by e^{gamma_C} of the chunk
  C_ODONE = 14,    // MMA: O1 and O2 of the chunk complete
  C_OFREE = 15,    // out: O1 and O2 read
  C_DRAIN = 16,    // MMA issuer, abort path only: every product it issued has completed
  C_COUNT = 17,
  // preparation CTA
  P_FULL = 0,      // [2 pipelines][2 buffers] K and Q tiles landed (tx)
  P_HEAD = 4,      // [2][2 slots] controller: item slot, decay vectors, padding rows zeroed
  P_KQDONE = 8,    // [2]
  P_WDONE = 12,    // [2] (-W)^T complete
  P_ITEMFREE = 14, // [2][2 buffers] the tile buffer's last product, (-W)^T, done
  P_PUB = 18,      // [2] item's record landed (one arrival per warp): it may be released
  P_SLOTOK = 20,   // [2] publisher: the item's ring slot has been copied out by its chain CTA
  P_KQFREE = 22,   // [2] KQ accumulator of a pipeline read out (one arrival per warp)
  P_VECFREE = 24,  // [2][2] vector slot (pipeline, use % 2) free: its item finished
  P_DRAIN = 28,    // [2][2] MMA issuers (KQ, the pipeline's W), abort path only: their
                   //        products completed
  P_COUNT = 32
};
static_assert(P_COUNT * 8 <= 256 && C_COUNT * 8 <= 256, "barrier area (TMEM address at +256)");
static_assert(NBUF <= 3 && NBUF_NO <= 3 && C_RECFREE == C_RECFULL + 3 &&
              C_LANDED == C_RECFREE + 3 && C_MERGED == C_LANDED + 3, "chain barriers");

// named barriers
constexpr int BAR_STATE = 1, BAR_OUT = 2;       // chain: 256, 128 threads
constexpr int BAR_PREP0 = 1;                    // preparation pipeline p: BAR_PREP0 + p
constexpr int BAR_SOLVE0 = 3;                   // its solve's phase 2: BAR_SOLVE0 + p

struct SplitParams {
  const float* g;
  const float* beta;
  const float* s0;           // [N,H,V,K] or NULL
  __nv_bfloat16* out;        // or NULL (state replay: no output)
  float* final_state;        // or NULL
  float* ckpt;               // state replay: [slots,H] BF16 chunk-entry state tiles, else NULL
  uint8_t* fac;              // state replay: [slots,H] copies of the chunk records (strided
                             // REC2_BYTES; the backward's reverse chain reads Ahat, (-W)^T and
                             // the decays, and Qg, which its own small kernel adds)
  int* status;               // workspace status word
  int* abort_g;              // global abort flag
  uint32_t* next_item;       // items claimed so far by the preparation CTAs
  uint32_t* consumed;        // [nch] records consumed (copied out), one line per chain CTA
  uint32_t* ready;           // [nch] lines: [nslot] stream position + 1 of the slot's record
  uint8_t* ring;             // [nch][nslot][REC_BYTES]
  int nslot;                 // ring slots per chain CTA (a power of two)
  const int32_t* cu;         // packed sequences: cu_seqlens [N+1], else NULL
  int* sstart;               // packed: [N*H] first stream position of each chain in its CTA
  int* slot0;                // packed: [N] first backward slot of each sequence
  int* lenj;                 // packed: [nch] stream length of each chain CTA
  int* sortj;                // packed: [nch] chain CTAs by stream length, longest first
  // segment summaries (twin != 0): chain x = n H + h is token range n of `bounds`; chain
  // CTA j < nch runs it from S0 = 0 with the value term (-> sumE), chain CTA nch + j runs
  // the same records from S0 = I without it (-> sumP)
  const int32_t* bounds;     // [N,2] token ranges, else NULL
  // paged state cache: sequence n reads and advances slot state_idx[n] of pool (zeros in
  // when has_init[n] == 0); state_idx[n] <= 0: zero output, the pool untouched
  float* pool;               // [num_slots,H,V,K] or NULL
  const int32_t* state_idx;
  const uint8_t* has_init;   // or NULL
  int num_slots;             // indices >= num_slots: padding as well
  float* sumP;               // [N,H,K,K]
  float* sumE;               // [N,H,V,K]
  int twin;
  int B, T, H, N;
  int HK;                    // query/key heads: value head h reads head h / (H / HK)
  int qk_group;              // H / HK
  int nch, nprep;
  float scale;
  long long wait_limit;      // clock cycles a bounded wait may take before it gives up
  long long drop_item;       // failure-detection tests only: this record is never published
};

// Query/key head of value head h (no division in the common case HK = H).
__device__ __forceinline__ int qk_of(const SplitParams& p, int h) {
  return p.qk_group == 1 ? h : h / p.qk_group;
}

// Token rows [bos, eos) of chain x = n H + h: sequence n (dense rows or cu_seqlens), or
// token range n of `bounds`.  A range out of [0, B T], reversed or crossing a batch row is
// empty here and returns false.
__device__ __forceinline__ bool chain_span(const SplitParams& p, int x, int64_t& bos,
                                           int64_t& eos) {
  const int n = x / p.H;
  if (!p.bounds) {
    seq_span(n, p.B, p.T, p.cu, bos, eos);
    return true;
  }
  const int64_t total = (int64_t)p.B * p.T;
  const int64_t r0 = p.bounds[2 * n], r1 = p.bounds[2 * n + 1];
  const bool ok = r0 >= 0 && r1 >= r0 && r1 <= total && (r1 == r0 || r0 / p.T == (r1 - 1) / p.T);
  bos = ok ? r0 : 0;
  eos = ok ? r1 : 0;
  return ok;
}

// About 2 s at the GB300's clocks.
constexpr long long kWaitLimitCycles = 4000000000ll;

// Failure-detection tests: the next split launch on this host thread never publishes one
// record and uses a short wait limit, so that a bounded wait runs out (one shot).
struct InjectedTimeout {
  long long item = -1;
  long long wait_limit = 0;
};
thread_local InjectedTimeout g_inject;

struct Ctx {
  volatile int* abort_l;     // CTA-local abort flag (shared memory)
  const SplitParams* p;
};

__device__ __forceinline__ void raise_abort(const Ctx& cx) {
  *cx.abort_l = 1;
  atomicExch(cx.p->abort_g, 1);
  atomicExch(cx.p->status, 5 /* SF_ERR_TIMEOUT */);
}

// The CTA's own flag is read every time; the global flag, on a line that every polling
// thread of the grid would otherwise keep hot, only on every 64th call of a wait loop.
__device__ __forceinline__ bool aborted(const Ctx& cx, uint32_t n) {
  return *cx.abort_l || ((n & 63) == 0 && ld_volatile_s32(cx.p->abort_g));
}

// The first wait that runs out records where it was in the word after the status word
// (kept, like the status, until the caller clears it): bit 30 set, the CTA in bits 12-29,
// the warp in bits 6-11, and what it waited on in bits 0-5 (an mbarrier's index in its
// CTA, or 63 for a flag in global memory).
__device__ __forceinline__ void note_timeout(const Ctx& cx, uint32_t what) {
  atomicCAS(cx.p->status + 1, 0,
            (int)(0x40000000u | (blockIdx.x << 12) | ((threadIdx.x >> 5) << 6) | (what & 63u)));
}

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, const Ctx& cx) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if (*cx.abort_l) return false;
    if (clock64() - t0 > cx.p->wait_limit) {
      note_timeout(cx, (smem_u32(bar) & 255u) >> 3);
      return false;
    }
  }
}

// All `nthr` threads on named barrier `id` wait; they agree on the outcome.
__device__ __forceinline__ bool group_wait(uint64_t* bar, uint32_t parity, int id, int nthr,
                                           const Ctx& cx) {
  const bool ok = named_bar_and(id, nthr, wait_bar(bar, parity, cx));
  if (!ok && (threadIdx.x & (nthr - 1)) == 0) raise_abort(cx);
  return ok;
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const Ctx& cx) {
  const bool ok = __all_sync(0xffffffffu, wait_bar(bar, parity, cx)) != 0;
  if (!ok && (threadIdx.x & 31) == 0) raise_abort(cx);
  return ok;
}

// One thread waits until the global counter reaches `target`.
__device__ __forceinline__ bool poll_ge(const uint32_t* f, uint32_t target, const Ctx& cx) {
  if (ld_acquire_u32(f) >= target) return true;
  const long long t0 = clock64();
  for (uint32_t n = 1;; ++n) {
    __nanosleep(32);
    if (ld_acquire_u32(f) >= target) return true;
    if (aborted(cx, n)) return false;
    if (clock64() - t0 > cx.p->wait_limit) {
      note_timeout(cx, 63);
      return false;
    }
  }
}

__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&x)[64]) {
  tmem_ld32(taddr, *reinterpret_cast<float(*)[32]>(x));
  tmem_ld32(taddr + 32, *reinterpret_cast<float(*)[32]>(x + 32));
  tmem_ld_wait();
}

// Geometry.  Chain CTA j owns the chains x = j + nch t (t = 0, 1, ...; x = n H + h) and
// walks their chunks in order: its stream position s is chunk c of one of them.  Records
// are produced in the order (s, j): every chain CTA's position s before any s + 1, the
// CTAs with the longer streams first.  Dense inputs have closed forms; packed inputs and
// token ranges use the per-chain stream starts and per-CTA stream lengths built by
// split_setup_kernel.
struct Geo {
  const SplitParams* p;
  int H, NH, nch, ncd, q, r;
  bool packed;
  const int* lenj;           // packed: shared-memory copy
  const int* sortj;
  long long full, total;
  // packed: production order in intervals of stream positions with a constant number of
  // active chain CTAs -- interval m (m = 0 .. nch-1) has nch - m of them, starts at
  // position seg_s(m) and at record seg_w(m); the table follows sortj in shared memory
  __device__ const int* seg_s() const { return sortj + 64; }
  __device__ const long long* seg_w() const { return reinterpret_cast<const long long*>(sortj + 64 + 66); }
  __device__ void init(const SplitParams& pr, const int* len_s, const int* sort_s) {
    p = &pr;
    H = pr.H;
    NH = pr.N * pr.H;
    nch = pr.nch;
    packed = pr.cu != nullptr || pr.bounds != nullptr;
    ncd = (pr.T + CHUNK - 1) / CHUNK;
    q = NH / nch;
    r = NH % nch;
    full = (long long)q * ncd * nch;
    lenj = len_s;
    sortj = sort_s;
    if (packed) {
      total = 0;
      for (int i = 0; i < nch; ++i) total += lenj[i];
    } else {
      total = (long long)NH * ncd;
    }
  }
  __device__ int chains_of(int j) const { return (NH - j + nch - 1) / nch; }
  __device__ bool span(int x, int64_t& bos, int64_t& eos) const { return chain_span(*p, x, bos, eos); }
  __device__ int len_of(int j) const { return packed ? lenj[j] : chains_of(j) * ncd; }
  // w-th record in production order -> (chain CTA, stream position)
  __device__ void item(long long w, int& j, int& s) const {
    if (!packed) {
      if (w < full) {
        s = (int)(w / nch);
        j = (int)(w % nch);
      } else {
        const long long w2 = w - full;
        s = q * ncd + (int)(w2 / r);
        j = (int)(w2 % r);
      }
      return;
    }
    // the last interval starting at or before record w
    int lo = 0, hi = nch;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (seg_w()[mid] <= w) lo = mid; else hi = mid;
    }
    const int k = nch - lo;
    const long long off = w - seg_w()[lo];
    s = seg_s()[lo] + (int)(off / k);
    j = sortj[(int)(off % k)];
  }
  // fills the production-order table from the stream lengths (one thread)
  __device__ static void build_table(int nch, const int* lenj, const int* sortj, int* sg_s,
                                     long long* sg_w) {
    long long w = 0;
    for (int m = 0; m < nch; ++m) {
      const int k = nch - m;                               // active chain CTAs
      const int lo = (m == 0) ? 0 : lenj[sortj[k]];        // shortest stream still ahead ends
      const int hi = lenj[sortj[k - 1]];
      sg_s[m] = lo;
      sg_w[m] = w;
      w += (long long)k * (hi > lo ? hi - lo : 0);
    }
  }
  // stream position s of chain CTA j -> chain x and its chunk c
  __device__ void locate(int j, int s, int& x, int& c) const {
    if (!packed) {
      const int t = s / ncd;
      x = j + nch * t;
      c = s - t * ncd;
      return;
    }
    int lo = 0, hi = chains_of(j);
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (p->sstart[j + nch * mid] <= s) lo = mid; else hi = mid;
    }
    x = j + nch * lo;
    c = s - p->sstart[x];
  }
};

// --------------------------------------------------------------------------
// State-chain CTA.  warp 0: record / tile loader; warp 1: MMA issuer; warps 4-11: the
// state (two warpgroups, one column half each); warps 12-15: output stores.
// Per chunk the products are issued in this order (all M = 128, v rows):
//   U^T = V^T T'^T                      into D      (as soon as the chunk has landed)
//   D  += S (-W)^T                      -> Delta^T  (the critical path: N = 64 only)
//   O1  = S Q^T                         (while the state warps turn D into Delta)
//   S   = e^{gamma_C} S + (Delta^T diag(dec)) K
//   O2  = Delta^T Ahat^T                out = scale (e^{gamma_i} O1 + O2)
// --------------------------------------------------------------------------
template <bool kOut>
__device__ __forceinline__ void chain_cta(const CUtensorMap* tmQ, const CUtensorMap* tmK,
                                          const CUtensorMap* tmV, const CUtensorMap* tmO,
                                          const SplitParams& p, const Geo& geo, uint8_t* sm,
                                          uint32_t sb, uint64_t* bars, uint32_t tm,
                                          const Ctx& cx) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = p.H;
  // segment summaries: chain CTA nch + j is the P twin of chain CTA j (same chains, same
  // records and ring); it reads (-W)^T and the decays only and has no output
  const bool summ = p.twin != 0, ptwin = summ && (int)blockIdx.x >= geo.nch;
  constexpr bool has_out = kOut;                     // the output products and stores
  constexpr int NB = ChainBufs<kOut>::NB;
  constexpr uint32_t BUF = ChainBufs<kOut>::STRIDE, CK = ChainBufs<kOut>::K,
                     CV = ChainBufs<kOut>::V, RV = ChainBufs<kOut>::VEC;
  const bool need_v = !ptwin;                        // the value term U^T = V^T T'^T
  const int j = ptwin ? (int)blockIdx.x - geo.nch : (int)blockIdx.x;   // the stream's owner
  const int cnt = geo.chains_of(j);
  const int len = geo.len_of(j);
  const uint8_t* ringj = p.ring + (size_t)j * p.nslot * REC_BYTES;
  const int smask = p.nslot - 1;
  const uint32_t* readyj = p.ready + (size_t)j * FLAG_STRIDE;
  uint32_t* const consumed_me = p.consumed + (size_t)blockIdx.x * FLAG_STRIDE;

  if (warp < 4) {
    reg_dealloc<RC_CTL>();
    if (warp == 0) {
      // ------------------------------------------------------------ loader
      // Up to NB chunks in flight.  A ring slot is handed back (consumed) once its
      // record has landed in shared memory: at the latest when the buffer is needed
      // again (then the chunk that used it is done), earlier if the copy is seen landed;
      // the slots landed by then go back with one release.  A chunk cut short by its
      // sequence end lands on its own barrier first: the warp zeroes its K and V rows
      // past the end (so that they add nothing to U or the state update, whatever the
      // rows beyond the sequence hold) and only then marks the buffer full.
      int issued = 0, rel = 0;
      bool ok = true;
      uint32_t flag_next = 0;            // the next record's ready flag, read one chunk ahead
      uint32_t landed_uses = 0;          // bit b: parity of buffer b's next LANDED phase
      uint32_t part_of = 0;              // bit b: buffer b holds a partial chunk
      auto release_to = [&](int n) {
        fence_proxy_async_global();
        st_release_u32(consumed_me, (uint32_t)n);
        rel = n;
      };
      // without output the record's Ahat is not needed (the P twin: no T' either)
      const uint32_t rec_tx =
          !has_out ? (ptwin ? 16384u : 24576u) + (REC_BYTES - R_VEC) : REC_BYTES;
      const uint32_t tx = rec_tx + 2 * C_T_PANEL * (1u + (need_v ? 1u : 0u) + (has_out ? 1u : 0u));
      int s = 0, t = 0, c = 0, ncx = 0, hk = 0, h = 0;
      int64_t bos = 0, eos = 0;
      for (; s < len; ++s, ++c) {
        while (c >= ncx) {      // next chain with chunks (and its query/key head)
          const int x = j + geo.nch * (t++);
          geo.span(x, bos, eos);
          ncx = (int)n_chunks(eos - bos);
          h = x % H;
          hk = qk_of(p, h);
          c = 0;
        }
        const int b = s % NB;
        const int row0 = (int)(bos + (int64_t)c * CHUNK);
        const int64_t rem = eos - (bos + (int64_t)c * CHUNK);
        const int L = rem < CHUNK ? (int)rem : CHUNK;
        const bool part = L < CHUNK;
        uint64_t* txbar = part ? &bars[C_LANDED + b] : &bars[C_RECFULL + b];
        uint8_t* buf = sm + b * BUF;
        // the record's flag first (usually set long before: its latency hides behind the
        // wait for the buffer), then the buffer, free once the chunk that used it has had
        // its products and its output read
        if (lane == 0) {
          ok = flag_next >= (uint32_t)s + 1 || poll_ge(readyj + (s & smask), (uint32_t)s + 1, cx);
          // the producer's plain stores before its release, then our bulk reads
          if (ok) fence_proxy_async_global();
          ok = ok && (s < NB || wait_bar(&bars[C_RECFREE + b], ((s - NB) / NB) & 1, cx));
        }
        if (!(ok = __shfl_sync(0xffffffffu, ok, 0) != 0)) break;
        part_of = (part_of & ~(1u << b)) | ((part ? 1u : 0u) << b);
        if (lane == 0) {
          mbar_arrive_expect_tx(txbar, tx);
          const uint8_t* src = ringj + (size_t)(s & smask) * REC_BYTES;
          if (has_out) {
            bulk_g2s(buf, src, REC_BYTES, txbar);
          } else {
            // (-W)^T and, except for a P twin, T' (contiguous), then the decays
            bulk_g2s(buf + R_W, src + R_W, ptwin ? 16384u : 24576u, txbar);
            bulk_g2s(buf + RV, src + R_VEC, REC_BYTES - R_VEC, txbar);
          }
          tma_load_4d(buf + CK, tmK, txbar, 0, row0, 0, hk);
          if (has_out) tma_load_4d(buf + C_Q, tmQ, txbar, 0, row0, 0, hk);
          if (need_v) tma_load_4d(buf + CV, tmV, txbar, 0, row0, 0, h);
        }
        issued = s + 1;
        // the next record's flag, read now and looked at next time round
        if (lane == 0 && s + 1 < len) flag_next = ld_acquire_u32(readyj + ((s + 1) & smask));
        if (part) {
          const uint32_t ph = (landed_uses >> b) & 1u;
          landed_uses ^= 1u << b;
          bool okl = true;
          if (lane == 0) okl = wait_bar(txbar, ph, cx);
          if (!(ok = __shfl_sync(0xffffffffu, okl, 0) != 0)) break;
          // rows L..63 of K and V (two 64-column panels each): zero
          const int rows = CHUNK - L;
          const int per = rows * 8;               // 16-byte chunks per panel
          const int ntile = need_v ? 4 : 2;
          for (int idx = lane; idx < ntile * per; idx += 32) {
            const int tile = idx / per, rr = idx % per;
            uint8_t* base_t = buf + ((tile >> 1) ? CV : CK) + (tile & 1) * C_T_PANEL;
            *reinterpret_cast<uint4*>(base_t + (L + rr / 8) * 128 + (rr % 8) * 16) =
                make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[C_RECFULL + b]);
        }
        if (lane == 0) {
          // records up to s - NB have landed (their buffers came back); later ones are
          // tested against their buffers' current phases
          int n = rel;
          if (s >= NB && n < s - NB + 1) n = s - NB + 1;
          while (n < s && mbar_test(&bars[C_RECFULL + n % NB], (n / NB) & 1)) ++n;
          if (n >= rel + 2) release_to(n);   // two slots at a time (the ring has nslot)
        }
      }
      if (lane == 0) {
        if (ok && rel < len) {
          // records before len - NB landed before their buffers were taken again (and a
          // parity wait on a buffer's older phase could be mistaken for its newer one), so
          // only the last NB are waited for
          for (int n = rel > len - NB ? rel : (len > NB ? len - NB : 0); n < len && ok; ++n)
            ok = wait_bar(&bars[C_RECFULL + n % NB], (n / NB) & 1, cx);
          if (ok) release_to(len);
        }
        if (!ok) {
          raise_abort(cx);
          // let every copy still in flight land before leaving
          for (int q = issued > NB ? issued - NB : 0; q < issued; ++q) {
            const int b = q % NB;
            if ((part_of >> b) & 1u)
              mbar_wait(&bars[C_LANDED + b], ((landed_uses >> b) & 1u) ^ 1u, 100000000ull);
            else
              mbar_wait(&bars[C_RECFULL + b], (q / NB) & 1, 100000000ull);
          }
        }
      }
      __syncwarp();
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      // The chain's products come in a fixed order, so the issuer blocks on each
      // condition in turn (a suspended wait leaves the issue slots to the other warps).
      if (lane == 0) {
        for (int s = 0; s < len; ++s) {
          const int rb = s % NB;
          const uint32_t buf = sb + rb * BUF;
          if (!wait_bar(&bars[C_RECFULL + rb], (s / NB) & 1, cx)) {
            raise_abort(cx);
            break;
          }
          tc_fence_after();
          if (need_v) {
            // U^T = V^T T'^T (the accumulator's previous contents were read before the
            // previous chunk's DREADY, which this thread waited for)
            const uint64_t av = sdesc_sw128(buf + CV, C_T_PANEL, 1024);
            const uint64_t bt = sdesc_sw128(buf + R_T1, 0, 1024);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_bf16(tm + TM_D, av + (uint64_t)(kk * 2048 >> 4), bt + (uint64_t)(kk * 2), ID_AMN,
                       kk > 0 ? 1u : 0u);
          }
          // Delta^T = U^T - S W^T: the products on the chain's critical path
          if (!wait_bar(&bars[C_SREADY], s & 1, cx)) {
            raise_abort(cx);
            break;
          }
          tc_fence_after();
          {
            const uint64_t bw = sdesc_sw128(buf + R_W, 16384, 1024);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_bf16_ta(tm + TM_D, tm + TM_SB + kk * 8, bw + (uint64_t)(kk * 2048 >> 4), ID_MG64,
                          (need_v || kk > 0) ? 1u : 0u);
            mma_commit(&bars[C_MERGED]);
          }
          if (has_out) {
            // O1 = S Q^T, while the state warps form Delta (O1 of the previous chunk read)
            if (s >= 1 && !wait_bar(&bars[C_OFREE], (s - 1) & 1, cx)) {
              raise_abort(cx);
              break;
            }
            tc_fence_after();
            const uint64_t bq = sdesc_sw128(buf + C_Q, 0, 1024);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint64_t o = (uint64_t)(((kk >> 2) * C_T_PANEL + (kk & 3) * 32) >> 4);
              mma_bf16_ta(tm + TM_O1, tm + TM_SB + kk * 8, bq + o, ID_N64, kk > 0 ? 1u : 0u);
            }
          }
          // S <- e^{gamma_C} S + (Delta^T diag(dec)) K, then O2 = Delta^T Ahat^T
          if (!wait_bar(&bars[C_DREADY], s & 1, cx) || !wait_bar(&bars[C_SSCALED], s & 1, cx)) {
            raise_abort(cx);
            break;
          }
          tc_fence_after();
          const uint64_t bk = sdesc_sw128(buf + CK, C_T_PANEL, 1024);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16_ta(tm + TM_S, tm + TM_DDB + kk * 8, bk + (uint64_t)(kk * 2048 >> 4), ID_MG, 1u);
          mma_commit(&bars[C_SUDONE]);
          if (has_out) {
            const uint64_t ba = sdesc_sw128(buf + R_AH, 0, 1024);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_bf16_ta(tm + TM_O2, tm + TM_DB + kk * 8, ba + (uint64_t)(kk * 2), ID_N64,
                          kk > 0 ? 1u : 0u);
            mma_commit(&bars[C_ODONE]);
          }
          mma_commit(&bars[C_RECFREE + rb]);
        }
        if (*cx.abort_l) {
          // leave no product running into the TMEM that the CTA frees on its way out
          mma_commit(&bars[C_DRAIN]);
          mbar_wait(&bars[C_DRAIN], 0, 100000000ull);
        }
      }
      __syncwarp();
    }
  } else if (warp < 12) {
    reg_alloc<RC_STATE>();
    // -------------------------------------------------------------- state
    const int st_t = tid - 128;                       // 0..255
    const int w = st_t >> 7;                          // column half
    const int v = ((warp & 3) << 5) + lane;           // TMEM lane = state row
    const uint32_t tl = tm + ((uint32_t)((warp & 3) * 32) << 16);
    bool ok = true;
    int sbase = 0;
    for (int t = 0; t < cnt && ok; ++t) {
      const int x = j + geo.nch * t;
      const size_t soff = ((size_t)x * D + v) * D + 64 * w;   // states [N*H, V, K]
      int64_t bos, eos;
      const bool okr = geo.span(x, bos, eos);
      const int nc = (int)n_chunks(eos - bos);
      float* const fdst = summ ? (ptwin ? p.sumP : p.sumE) : p.final_state;
      // this thread's 64 entry values and final values: the [N,H,V,K] arguments, or the
      // chain's slot of the paged cache (padding: zeros in, nothing out)
      const float* s0p = p.s0 ? p.s0 + soff : nullptr;
      float* fp = fdst ? fdst + soff : nullptr;
      if (p.pool) {
        const int n = x / H, ps = p.state_idx[n];
        const bool live = ps > 0 && ps < p.num_slots;
        const size_t off = (((size_t)(live ? ps : 0) * H + x % H) * D + v) * D + 64 * w;
        s0p = (live && (!p.has_init || p.has_init[n])) ? p.pool + off : nullptr;
        fp = live ? p.pool + off : nullptr;
      }
      // entry state element (v, 64 w + e) without S0: zero, or the identity for the P twin
      auto s_init = [&](int e) -> float { return (ptwin && 64 * w + e == v) ? 1.f : 0.f; };
      // state replay: chunk c's entry state goes to ckpt[first slot of the sequence + c], a
      // BF16 [128 v][128 k] tile in the 128-byte-swizzled panel layout (this thread: row v of
      // panel w)
      uint8_t* ck = p.ckpt ? reinterpret_cast<uint8_t*>(p.ckpt) +
                                 ((size_t)chunk_slot_base(x / H, p.B, p.T, p.cu) * H + x % H) *
                                     CKPT_TILE_BYTES +
                                 (size_t)w * 16384 + (size_t)v * 128
                           : nullptr;
      const size_t ck_stride = (size_t)H * CKPT_TILE_BYTES;
      // A checkpoint row.  Without output, each state warp's 32 rows (4 KB of one panel)
      // go out by one bulk copy from the warp's staging area (direct stores from the 256
      // threads stall the chain's own products and loads on this SM): stage_ckpt parks the
      // row once the warp's previous copy has read the area, and after the next named
      // barrier of the state warps send_ckpt sends the 4 KB from lane 0, whose row is the
      // warp's first.
      uint8_t* const stage = sm + C_CST + (st_t >> 5) * 4096;
      auto stage_ckpt = [&](const uint32_t(&uu)[32]) {
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
        store_ckpt_row(stage + lane * 128, v, uu);   // (v mod 8 == lane mod 8)
        fence_proxy_async_smem();
      };
      auto send_ckpt = [&](uint8_t* row) {
        if (lane == 0) {
          bulk_s2g(row, stage, 4096);
          bulk_commit();
        }
      };
      if (nc == 0) {
        // an empty sequence passes its initial state through (an empty range: the identity
        // map; an invalid range: NaN)
        if (fp) {
          float4* dst = reinterpret_cast<float4*>(fp);
          const float4* src = reinterpret_cast<const float4*>(s0p);
          const float nanv = __int_as_float(0x7fc00000);
#pragma unroll
          for (int e = 0; e < 16; ++e)
            dst[e] = s0p ? src[e]
                   : !okr ? make_float4(nanv, nanv, nanv, nanv)
                          : make_float4(s_init(4 * e), s_init(4 * e + 1), s_init(4 * e + 2), s_init(4 * e + 3));
        }
        continue;
      }
      {
        // the entry state as the first product's BF16 operand needs nothing from the
        // record, so it goes out before the first buffer has landed (the products of the
        // CTA's previous chain that read it completed before that chain's last SUDONE);
        // the FP32 copy is scaled by the chunk's e^{gamma_C} once the buffer is in
        float xv[64];
        if (s0p) {
          const float4* src = reinterpret_cast<const float4*>(s0p);
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float4 f = src[e];
            xv[4 * e] = f.x; xv[4 * e + 1] = f.y; xv[4 * e + 2] = f.z; xv[4 * e + 3] = f.w;
          }
        } else {
#pragma unroll
          for (int e = 0; e < 64; ++e) xv[e] = s_init(e);
        }
        {
          uint32_t u[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) u[e] = pack_bf16x2(xv[2 * e], xv[2 * e + 1]);
          tmem_st16(tl + TM_SB + 32 * w, *reinterpret_cast<const uint32_t(*)[16]>(u));
          tmem_st16(tl + TM_SB + 32 * w + 16, *reinterpret_cast<const uint32_t(*)[16]>(u + 16));
          if (ck) {
            if constexpr (kOut) store_ckpt_row(ck, v, u);
            else stage_ckpt(u);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        named_bar(BAR_STATE, 256);
        if (st_t == 0) mbar_arrive(&bars[C_SREADY]);
        if (!kOut && ck) send_ckpt(ck);
        if (!(ok = group_wait(&bars[C_RECFULL + sbase % NB], (sbase / NB) & 1, BAR_STATE, 256,
                              cx)))
          break;
        const float g0 = *reinterpret_cast<const float*>(sm + (sbase % NB) * BUF + RV + V_GC);
#pragma unroll
        for (int e = 0; e < 64; ++e) xv[e] *= g0;
        tmem_st32(tl + TM_S + 64 * w, *reinterpret_cast<float(*)[32]>(xv));
        tmem_st32(tl + TM_S + 64 * w + 32, *reinterpret_cast<float(*)[32]>(xv + 32));
        tmem_st_wait();
        tc_fence_before();
        named_bar(BAR_STATE, 256);
        if (st_t == 0) mbar_arrive(&bars[C_SSCALED]);
      }
      for (int c = 0; c < nc && ok; ++c) {
        const int s = sbase + c;
        uint8_t* buf = sm + (s % NB) * BUF;
        if (!(ok = group_wait(&bars[C_MERGED], s & 1, BAR_STATE, 256, cx))) break;
        tc_fence_after();
        {
          // Delta^T for columns [32w, 32w + 32): the accumulator holds U^T - S W^T (the P
          // twin: -S W^T)
          float a[32];
          tmem_ld32(tl + TM_D + 32 * w, a);
          const float* dec = reinterpret_cast<const float*>(buf + RV + V_DEC) + 32 * w;
          tmem_ld_wait();
          uint32_t d1[16], d2[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            d1[e] = pack_bf16x2(a[2 * e], a[2 * e + 1]);
            d2[e] = pack_bf16x2(a[2 * e] * dec[2 * e], a[2 * e + 1] * dec[2 * e + 1]);
          }
          tmem_st16(tl + TM_DB + 16 * w, d1);
          tmem_st16(tl + TM_DDB + 16 * w, d2);
        }
        tmem_st_wait();
        tc_fence_before();
        named_bar(BAR_STATE, 256);
        if (st_t == 0) mbar_arrive(&bars[C_DREADY]);
        if (!(ok = group_wait(&bars[C_SUDONE], s & 1, BAR_STATE, 256, cx))) break;
        tc_fence_after();
        float xv[64];
        tmem_ld64(tl + TM_S + 64 * w, xv);
        if (c + 1 == nc) {
          if (fp) {
            float4* dst = reinterpret_cast<float4*>(fp);
#pragma unroll
            for (int e = 0; e < 16; ++e)
              dst[e] = make_float4(xv[4 * e], xv[4 * e + 1], xv[4 * e + 2], xv[4 * e + 3]);
          }
        } else {
          uint32_t u[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) u[e] = pack_bf16x2(xv[2 * e], xv[2 * e + 1]);
          tmem_st16(tl + TM_SB + 32 * w, *reinterpret_cast<const uint32_t(*)[16]>(u));
          tmem_st16(tl + TM_SB + 32 * w + 16, *reinterpret_cast<const uint32_t(*)[16]>(u + 16));
          if (!kOut && ck) stage_ckpt(u);
          tmem_st_wait();
          tc_fence_before();
          named_bar(BAR_STATE, 256);
          if (st_t == 0) mbar_arrive(&bars[C_SREADY]);
          // state replay: the next chunk's entry state, written while its first product runs
          if (ck) {
            if constexpr (kOut) store_ckpt_row(ck + (size_t)(c + 1) * ck_stride, v, u);
            else send_ckpt(ck + (size_t)(c + 1) * ck_stride);
          }
          const int s1 = s + 1;
          if (!(ok = group_wait(&bars[C_RECFULL + s1 % NB], (s1 / NB) & 1, BAR_STATE, 256, cx)))
            break;
          const float gn = *reinterpret_cast<const float*>(sm + (s1 % NB) * BUF + RV + V_GC);
#pragma unroll
          for (int e = 0; e < 64; ++e) xv[e] *= gn;
          tmem_st32(tl + TM_S + 64 * w, *reinterpret_cast<float(*)[32]>(xv));
          tmem_st32(tl + TM_S + 64 * w + 32, *reinterpret_cast<float(*)[32]>(xv + 32));
          tmem_st_wait();
          tc_fence_before();
          named_bar(BAR_STATE, 256);
          if (st_t == 0) mbar_arrive(&bars[C_SSCALED]);
        }
      }
      sbase += nc;
    }
    // every checkpoint copy has landed before the CTA leaves
    if (!kOut && lane == 0) bulk_wait_all();
  } else {
    reg_dealloc<RC_OUT>();
    // -------------------------------------------------------------- output
    const int v = ((warp & 3) << 5) + lane;
    const uint32_t tl = tm + ((uint32_t)((warp & 3) * 32) << 16);
    const size_t rs = (size_t)H * D;
    bool ok = true;
    int s = 0;
    for (int t = 0; t < (has_out ? cnt : 0) && ok; ++t) {
      const int x = j + geo.nch * t, h = x % H;
      int64_t bos, eos;
      geo.span(x, bos, eos);
      const int nc = (int)n_chunks(eos - bos);
      // paged cache: padding (a slot index outside [1, num_slots)) gives zero output
      const bool padded = p.pool && (p.state_idx[x / H] <= 0 || p.state_idx[x / H] >= p.num_slots);
      for (int c = 0; c < nc; ++c, ++s) {
        if (!(ok = group_wait(&bars[C_ODONE], s & 1, BAR_OUT, 128, cx))) break;
        tc_fence_after();
        const int rb = s % NB;
        const float* eg = reinterpret_cast<const float*>(sm + rb * BUF + RV + V_EG);
        const float sc = padded ? 0.f : p.scale;
        uint32_t ob[32];     // BF16 pairs: out rows 2e and 2e + 1 of this thread's column v
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float a1[32], a2[32];
          tmem_ld32(tl + TM_O1 + 32 * hh, a1);
          tmem_ld32(tl + TM_O2 + 32 * hh, a2);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int i = 32 * hh + 2 * e;
            ob[16 * hh + e] = pack_bf16x2(sc * fmaf(eg[i], a1[2 * e], a2[2 * e]),
                                          sc * fmaf(eg[i + 1], a1[2 * e + 1], a2[2 * e + 1]));
          }
        }
        auto out_at = [&](int i) -> uint16_t { return (uint16_t)(ob[i >> 1] >> (16 * (i & 1))); };
        // O1, O2 and the chunk's buffer (e^gamma read) are free for the next products and
        // records; the staging tile of two chunks back must have been read by its store
        tc_fence_before();
        if (v == 0) bulk_wait_read<1>();
        named_bar(BAR_OUT, 128);
        if (v == 0) {
          mbar_arrive(&bars[C_OFREE]);
          mbar_arrive(&bars[C_RECFREE + rb]);
        }
        const int64_t row0 = bos + (int64_t)c * CHUNK;
        const int L = (eos - row0) < CHUNK ? (int)(eos - row0) : CHUNK;
        if (L == CHUNK) {
          // a staging tile of its own takes the [64 token][128 v] tile in the panel layout;
          // one TMA store sends it out
          uint8_t* st = sm + C_OST + (s & 1) * 16384;
#pragma unroll
          for (int i = 0; i < 64; ++i)
            *reinterpret_cast<uint16_t*>(st + sw128_off(i, v, 8192)) = out_at(i);
          fence_proxy_async_smem();
          named_bar(BAR_OUT, 128);
          if (v == 0) {
            tma_store_4d(tmO, st, 0, (int)row0, 0, h);
            bulk_commit();
          }
        } else {
          // a chunk cut short by the sequence end: only its own rows are written
          uint16_t* orow = reinterpret_cast<uint16_t*>(p.out + ((size_t)row0 * H + h) * D + v);
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (i < L) orow[i * rs] = out_at(i);
        }
      }
    }
    if (v == 0) bulk_wait_all();   // every output store has landed before the CTA leaves
  }
}

// One warp stores 32 consecutive rows (row0 % 32 == 0, this lane's row = row0 + lane) of a
// panel-layout BF16 tile into global memory: each lane parks its 128-byte line in the
// warp's 4 KB of shared memory (already in the tile's swizzled order), and lane 0 sends
// the 4 KB with one bulk copy (whole lines into L2).  The staging area is reused only
// after the previous copy from it has been read; record_landed() waits for every copy.
// kTwo: the same rows also to gtile2.
template <bool kTwo>
__device__ __forceinline__ void store_rows(uint8_t* gtile, uint8_t* gtile2, uint8_t* stage,
                                           int row0, const uint32_t (&u)[32], int lane) {
  if (lane == 0) bulk_wait_read_all();
  __syncwarp();
  uint4* mine = reinterpret_cast<uint4*>(stage + lane * 128);
#pragma unroll
  for (int e = 0; e < 8; ++e)
    mine[e ^ (lane & 7)] = make_uint4(u[4 * e], u[4 * e + 1], u[4 * e + 2], u[4 * e + 3]);
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    bulk_s2g(gtile + (size_t)row0 * 128, stage, 4096);
    if constexpr (kTwo) bulk_s2g(gtile2 + (size_t)row0 * 128, stage, 4096);
    bulk_commit();
  }
}

// The warp's record stores have landed in global memory; then lane 0 counts the warp in
// on `pub` (four arrivals: the record may be released).
__device__ __forceinline__ void record_landed(int lane, uint64_t* pub) {
  if (lane == 0) {
    bulk_wait_all();
    fence_proxy_async_global();
    mbar_arrive(pub);
  }
  __syncwarp();
}

__device__ __forceinline__ void pack64(const float (&x)[64], uint32_t (&u)[32]) {
#pragma unroll
  for (int e = 0; e < 32; ++e) u[e] = pack_bf16x2(x[2 * e], x[2 * e + 1]);
}

// --------------------------------------------------------------------------
// The chunk's triangular solve on a preparation pipeline (four warps).
//
// T = (I + A)^{-1} for the strictly lower 64x64 A (FP32 rows in shared memory, leading
// dimension SOLVE_LD), delivered as the BF16 B operands T' = T diag(beta) and
// -T'' = -T diag(beta e^gamma) of the U and W products.  The blocking is that of
// solve_tc.cuh -- 16x16 diagonal blocks by substitution in FP32, then
// T_10 = -T_11 A_10 T_00 for the 32x32 halves and for the 64x64 matrix on TF32 mma --
// arranged for four warps, a barrier between the phases and a partial one inside phase 2:
//  phase 1: warp p (p = 0, 1), which wrote rows 32p..32p+31 of A, inverts the half's
//           two diagonal blocks (lanes 0-15 and 16-31, one column per lane, the block's
//           A in registers) and merges them into the half's lower-left block;
//  phase 2: one warp per 16x16 block of T[32:64, 0:32] = -T[32:64, 32:64] Y with
//           Y = A[32:64, 0:32] T[0:32, 0:32], each forming one Y block first.
// A product whose B operand is the previous product is taken in two steps: first the
// transpose X^T = N^T M^T of the inner product (both operands from shared memory), then
// the outer product with X^T's accumulator fragments as its B fragments -- valid once the
// k index of both outer operands is permuted (k-slot t <-> 2t, t + 4 <-> 2t + 1 within
// each 8-wide step), which keeps the intermediate in registers.
// --------------------------------------------------------------------------
namespace solve {

constexpr int L = SOLVE_LD;

__device__ __forceinline__ void mma4(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                     uint32_t a3, uint32_t b0, uint32_t b1) {
  const uint32_t a[4] = {a0, a1, a2, a3};
  const uint32_t b[2] = {b0, b1};
  mma_tf32_16x8x8(d, a, b);
}

// xt += M^T N^T for 16x16 blocks M (rows k, columns c) and N (rows n, columns k) in shared
// memory: xt[nt] are the C fragments of the 16x16 result [c][n], n in 8nt..8nt+7.
__device__ __forceinline__ void acc_tt(float (&xt)[2][4], const float* M, const float* N, int g,
                                       int t) {
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const float* mk = M + (8 * s + t) * L;
    const uint32_t a0 = f2tf32(mk[g]), a1 = f2tf32(mk[g + 8]);
    const uint32_t a2 = f2tf32(mk[4 * L + g]), a3 = f2tf32(mk[4 * L + g + 8]);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const float* nr = N + (8 * nt + g) * L + 8 * s + t;
      mma4(xt[nt], a0, a1, a2, a3, f2tf32(nr[0]), f2tf32(nr[4]));
    }
  }
}

// o += M X for a 16x16 block M in shared memory (rows i, columns k) and X given by the C
// fragments xt[s] of its transpose (X^T[n][k], k in 8s..8s+7); the k-slot permutation
// makes those fragments X's B fragments.  o[nt]: C fragments of [i][n], n in 8nt..8nt+7.
__device__ __forceinline__ void acc_nx(float (&o)[2][4], const float* M, const float (&xt)[2][4],
                                       int g, int t) {
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const float2 r0 = *reinterpret_cast<const float2*>(M + g * L + 8 * s + 2 * t);
    const float2 r1 = *reinterpret_cast<const float2*>(M + (g + 8) * L + 8 * s + 2 * t);
    const uint32_t a0 = f2tf32(r0.x), a2 = f2tf32(r0.y), a1 = f2tf32(r1.x), a3 = f2tf32(r1.y);
    mma4(o[0], a0, a1, a2, a3, f2tf32(xt[s][0]), f2tf32(xt[s][1]));
    mma4(o[1], a0, a1, a2, a3, f2tf32(xt[s][2]), f2tf32(xt[s][3]));
  }
}

// Block (R0.., C0..) of T from the C fragments of -T: FP32 into the T area (when `at`)
// and the BF16 operands T' and -T''.
__device__ __forceinline__ void put_block(float* at, uint8_t* t1, uint8_t* t2, const float* vs,
                                          int R0, int C0, const float (&o)[2][4], int g, int t) {
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    const int col = C0 + 8 * nt + 2 * t;
    const float2 b = *reinterpret_cast<const float2*>(vs + VEC_BETA + col);
    const float2 e = *reinterpret_cast<const float2*>(vs + VEC_EG + col);
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const int row = R0 + g + 8 * hf;
      const float x0 = -o[nt][2 * hf], x1 = -o[nt][2 * hf + 1];
      if (at) *reinterpret_cast<float2*>(at + row * L + col) = make_float2(x0, x1);
      const float p0 = x0 * b.x, p1 = x1 * b.y;
      const uint32_t off = sw128_off(row, col, 8192);
      *reinterpret_cast<uint32_t*>(t1 + off) = pack_bf16x2(p0, p1);
      *reinterpret_cast<uint32_t*>(t2 + off) = pack_bf16x2(-p0 * e.x, -p1 * e.y);
    }
  }
}

// Phase 1 for half p (one warp).
__device__ __forceinline__ void half(float* AT, uint8_t* t1, uint8_t* t2, const float* vs, int p,
                                     int lane) {
  {
    // diagonal block at o: this lane's column m of its inverse, by forward substitution
    const int m = lane & 15, o = 32 * p + 16 * (lane >> 4);
    float a[120];                      // A[o + i][o + j], j < i, at i (i - 1) / 2 + j
#pragma unroll
    for (int i = 1; i < 16; ++i) {
#pragma unroll
      for (int q = 0; q < (i + 3) / 4; ++q) {
        const float4 v = *reinterpret_cast<const float4*>(AT + (o + i) * L + o + 4 * q);
        const int b = i * (i - 1) / 2 + 4 * q;
        a[b] = v.x;
        if (4 * q + 1 < i) a[b + 1] = v.y;
        if (4 * q + 2 < i) a[b + 2] = v.z;
        if (4 * q + 3 < i) a[b + 3] = v.w;
      }
    }
    float acc[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = (i == m) ? 1.f : 0.f;
#pragma unroll
    for (int j = 0; j < 15; ++j) {
      const float x = acc[j];
#pragma unroll
      for (int i = j + 1; i < 16; ++i) acc[i] = fmaf(-a[i * (i - 1) / 2 + j], x, acc[i]);
    }
    __syncwarp();                      // every lane has its block's A in registers
    const float bm = vs[VEC_BETA + o + m], em = vs[VEC_EG + o + m];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      AT[(o + i) * L + o + m] = acc[i];
      const float p1 = acc[i] * bm;
      const uint32_t off = sw128_off(o + i, o + m, 8192);
      *reinterpret_cast<__nv_bfloat16*>(t1 + off) = __float2bfloat16_rn(p1);
      *reinterpret_cast<__nv_bfloat16*>(t2 + off) = __float2bfloat16_rn(-p1 * em);
    }
  }
  __syncwarp();
  // T_10 = -T_11 (A_10 T_00): Y^T = T_00^T A_10^T, then T_11 Y
  const int g = lane >> 2, t = lane & 3, o0 = 32 * p, o1 = o0 + 16;
  float yt[2][4] = {}, ob[2][4] = {};
  acc_tt(yt, AT + o0 * L + o0, AT + o1 * L + o0, g, t);
  acc_nx(ob, AT + o1 * L + o1, yt, g, t);
  __syncwarp();                        // A_10 read by every lane before T_10 replaces it
  put_block(AT, t1, t2, vs, o1, o0, ob, g, t);
}

// o += M N for 16x16 blocks M (rows i, columns k) and N (rows k, columns n) in shared
// memory, with acc_nx's k-slot permutation on both operands.
__device__ __forceinline__ void acc_nn(float (&o)[2][4], const float* M, const float* N, int g,
                                       int t) {
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const float2 r0 = *reinterpret_cast<const float2*>(M + g * L + 8 * s + 2 * t);
    const float2 r1 = *reinterpret_cast<const float2*>(M + (g + 8) * L + 8 * s + 2 * t);
    const uint32_t a0 = f2tf32(r0.x), a2 = f2tf32(r0.y), a1 = f2tf32(r1.x), a3 = f2tf32(r1.y);
    const float* n0 = N + (8 * s + 2 * t) * L + g;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
      mma4(o[nt], a0, a1, a2, a3, f2tf32(n0[8 * nt]), f2tf32(n0[L + 8 * nt]));
  }
}

// Phase 2 for the block (2 + M, c) of T (one warp), T[32:64, 0:32] = -T[32:64, 32:64] Y with
// Y = A[32:64, 0:32] T[0:32, 0:32].  The warp forms its Y block (M, c) = sum_{j >= c}
// A[2 + M][j] T[j][c] into the free upper-right quadrant of the A/T area (rows 16 M,
// columns 32 + 16 c); block (2, c) needs only that one, block (3, c) also Y (0, c), for
// which it waits on named barrier `yb` (the (2, c) warps arrive there once theirs is out).
template <int M>
__device__ __forceinline__ void lower(float* AT, uint8_t* t1, uint8_t* t2, const float* vs, int c,
                                      int yb, int lane) {
  const int g = lane >> 2, t = lane & 3;
  float* Y = AT + 32 + 16 * c;
  {
    float y[2][4] = {};
    for (int j = c; j < 2; ++j)
      acc_nn(y, AT + (32 + 16 * M) * L + 16 * j, AT + 16 * j * L + 16 * c, g, t);
    float* ym = Y + 16 * M * L;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      *reinterpret_cast<float2*>(ym + g * L + 8 * nt + 2 * t) = make_float2(y[nt][0], y[nt][1]);
      *reinterpret_cast<float2*>(ym + (g + 8) * L + 8 * nt + 2 * t) =
          make_float2(y[nt][2], y[nt][3]);
    }
  }
  __syncwarp();
  if (M == 0) named_bar_arrive(yb, 128);
  else named_bar(yb, 128);
  float ob[2][4] = {};
#pragma unroll
  for (int kb = 0; kb <= M; ++kb)
    acc_nn(ob, AT + (32 + 16 * M) * L + 32 + 16 * kb, Y + 16 * kb * L, g, t);
  put_block(nullptr, t1, t2, vs, 32 + 16 * M, 16 * c, ob, g, t);
}

}  // namespace solve

// --------------------------------------------------------------------------
// Preparation CTA.  Items (chunk records) are claimed one at a time, in stream order,
// from a grid-wide counter, so that a pipeline waiting for a full ring slot holds up
// only the chain that slot belongs to.  Per pipeline p (p = 0, 1) one warp each:
//   feeder (warp 2p): claim, gate/beta and the chunk's decay vectors, the K/Q tiles by TMA
//     into one of two buffers;
//   KQ issuer (warp 2p + 1): [K;Q] K^T of each item once its tiles have landed and the
//     previous item's accumulator was read out -- typically during the previous solve;
//   publisher (warp 14 + p): the release of each finished record and the ring-slot check
//     of the next;
// and four warps (4-7, 8-11) that turn the products into the record, one of whose threads
// issues (-W)^T as soon as the solve is done (warps 12, 13 are idle).  Every role waits
// (suspended) only on what it needs, so none of them holds up another.
// A pipeline's item u: [K;Q] K^T (issued while item u-1 is still in its solve), the
// decayed A and Ahat, the solve to T' and -T'', (-W)^T = K^T (-T'')^T; the record it
// writes holds (-W)^T, T', Ahat and the decay vectors.
// --------------------------------------------------------------------------
// kCopy: the state replay, whose records are also kept per chunk-head for the backward (a
// separate instantiation, so that the forward's preparation carries none of that code)
template <bool kCopy>
__device__ __forceinline__ void prep_cta(const CUtensorMap* tmQ, const CUtensorMap* tmK,
                                         const CUtensorMap* tmQ4, const CUtensorMap* tmK4,
                                         const CUtensorMap* tmV4, const SplitParams& p,
                                         const Geo& geo, uint8_t* sm, uint32_t sb,
                                         uint64_t* bars, uint32_t tm, const Ctx& cx) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = p.H;
  // segment summaries: no Q (its map is K's) and no Ahat in the records, whose ring slots
  // are read by two chain CTAs
  const bool summ = p.twin != 0;
  // item g -> (chain CTA, stream position, head, first row, length)
  // (fx: the index of the record's copy for the backward, slot * H + h, or -1)
  auto item = [&](long long g, int& jj, int& s, int& h, int& row0, int& L, int& fx) {
    geo.item(g, jj, s);
    int x, c;
    geo.locate(jj, s, x, c);
    int64_t bos, eos;
    geo.span(x, bos, eos);
    h = x % H;
    row0 = (int)(bos + (int64_t)c * CHUNK);
    L = (eos - row0) < CHUNK ? (int)(eos - row0) : CHUNK;
    if constexpr (kCopy) {
      const int n = x / H;
      fx = ((geo.packed ? p.slot0[n] : n * geo.ncd) + c) * H + h;
    } else {
      fx = -1;
    }
  };
  auto vec_of = [&](int pp, int use) {
    return reinterpret_cast<float*>(sm + pp * P_STRIDE + P_VEC + (use & 1) * P_VEC_SLOT);
  };

  if (warp < 4) {
    reg_dealloc<RP_CTL>();
    if (warp == 0 || warp == 2) {
      // ------------------------------------------------------------ feeder
      const int pp = warp >> 1;
      uint8_t* base = sm + pp * P_STRIDE;
      // pipeline 0 keeps [K;Q] in its tile rows, pipeline 1 [Q;K] (see the pipelines)
      const uint32_t kq_k = pp ? 8192u : 0u, kq_q = pp ? 0u : 8192u;
      // The first two items of every pipeline are fixed (pipeline q = 2 (CTA index) + pp
      // of the 2 nprep takes items q and 2 nprep + q), so that the launch starts without
      // waiting on the counter; the rest are claimed from it, after those 4 nprep.
      const int nq = 2 * p.nprep, q = 2 * ((int)blockIdx.x - (p.nch * (p.twin ? 2 : 1))) + pp;
      // lane 0's claim in flight (its result is read one use later, so that the atomic's
      // round trip overlaps a whole use)
      auto claim_start = [&]() -> uint32_t { return lane == 0 ? atomicAdd(p.next_item, 1u) : 0u; };
      auto claim_end = [&](uint32_t c) -> int {
        return __shfl_sync(0xffffffffu, (int)c, 0) + 2 * nq;
      };
      // An item's geometry, its gate/beta values (two tokens per lane, loaded one use
      // ahead so that their latency overlaps the waits), and its tiles warmed in L2 (V
      // for the chain CTA that will load it).
      struct Next {
        int g, jj, s, h, hk, row0, L, fx;   // hk: the query/key head of value head h
        float g0, g1, b0, b1;
      };
      auto fetch = [&](int g) {
        Next n{g, 0, 0, 0, 0, 0, 0, -1, 0.f, 0.f, 0.f, 0.f};
        if (g >= geo.total) return n;
        item(g, n.jj, n.s, n.h, n.row0, n.L, n.fx);
        n.hk = qk_of(p, n.h);
        const int e0 = 2 * lane, e1 = e0 + 1;
        const size_t o0 = (size_t)(n.row0 + e0) * H + n.h, o1 = (size_t)(n.row0 + e1) * H + n.h;
        if (e0 < n.L) { n.g0 = p.g[o0]; n.b0 = p.beta[o0]; }
        if (e1 < n.L) { n.g1 = p.g[o1]; n.b1 = p.beta[o1]; }
        if (lane == 0) {
          tma_prefetch_l2_4d(tmK4, 0, n.row0, 0, n.hk);
          if (!summ) tma_prefetch_l2_4d(tmQ4, 0, n.row0, 0, n.hk);
          tma_prefetch_l2_4d(tmV4, 0, n.row0, 0, n.h);
        }
        return n;
      };
      int last = -1;                 // last use with a tile copy
      bool ok = true;
      // items are claimed three uses ahead: `cur` is this use's, `nxt` the next one's,
      // and the claim in flight the one after (every item below geo.total is processed: a
      // pipeline's items only grow, so once one is past the end, so are the ones after it)
      Next cur = fetch(q);
      int gnn = nq + q;
      uint32_t inflight = claim_start();
      for (int use = 0; ok; ++use) {
        const bool done = cur.g >= geo.total;
        const int jj = cur.jj, s = cur.s, hk = cur.hk, row0 = cur.row0, L = cur.L;
        const long long gitem = cur.g;
        const int ub = use & 1;        // vector slot and tile buffer of this use
        // the [K;Q] tile first (it needs only the item's rows), then the vectors while it lands
        uint8_t* const kq = base + P_KQ + ub * P_KQ_BUF;
        if (!done) {
          // tile buffer ub: the product that read it last, (-W)^T of item use - 2, is done
          // (before the item's vector slot comes back, so this wait cannot hold that up)
          if (use >= 2 &&
              !(ok = warp_wait(&bars[P_ITEMFREE + 2 * pp + ub], ((use - 2) >> 1) & 1, cx)))
            break;
          if (lane == 0) {
            mbar_arrive_expect_tx(&bars[P_FULL + 2 * pp + ub], 2 * 16384);
#pragma unroll
            for (int pnl = 0; pnl < 2; ++pnl) {
              tma_load_3d(kq + pnl * P_KQ_PANEL + kq_k, tmK, &bars[P_FULL + 2 * pp + ub], 64 * pnl, hk,
                          row0);
              tma_load_3d(kq + pnl * P_KQ_PANEL + kq_q, tmQ, &bars[P_FULL + 2 * pp + ub], 64 * pnl, hk,
                          row0);
            }
          }
          last = use;
        }
        // the slot and the buffer are free once the item two uses back has finished (one
        // barrier per slot, so a phase can never be mistaken for the one two items later)
        if (use >= 2 && !(ok = warp_wait(&bars[P_VECFREE + 2 * pp + ub], ((use - 2) >> 1) & 1, cx)))
          break;
        float* vs = vec_of(pp, use);
        if (!done) {
          // gamma = in-chunk cumulative gate; decays e^{gamma}, e^{gamma_C - gamma}, and
          // the factors e^{+-(gamma - mid)} (used when the chunk's gamma range is <= 80)
          const int e0 = 2 * lane, e1 = e0 + 1;
          const float g0 = cur.g0, g1 = cur.g1, b0 = cur.b0, b1 = cur.b1;
          float sum = g0 + g1;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const float t = __shfl_up_sync(0xffffffffu, sum, o);
            if (lane >= o) sum += t;
          }
          const float excl = sum - (g0 + g1);
          const float a0 = excl + g0, a1 = excl + g0 + g1;
          float mx = fmaxf(a0, a1), mn = fminf(a0, a1);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
          }
          const bool fact = (mx - mn) <= 80.f;
          const float mid = 0.5f * (mx + mn);
          const float gC = __shfl_sync(0xffffffffu, a1, 31);
          vs[VEC_BETA + e0] = b0;
          vs[VEC_BETA + e1] = b1;
          vs[VEC_GAM + e0] = a0;
          vs[VEC_GAM + e1] = a1;
          vs[VEC_EG + e0] = expf(a0);
          vs[VEC_EG + e1] = expf(a1);
          vs[VEC_DEC + e0] = expf(gC - a0);
          vs[VEC_DEC + e1] = expf(gC - a1);
          vs[VEC_EP + e0] = fact ? expf(a0 - mid) : 0.f;
          vs[VEC_EP + e1] = fact ? expf(a1 - mid) : 0.f;
          vs[VEC_EM + e0] = fact ? expf(mid - a0) : 0.f;
          vs[VEC_EM + e1] = fact ? expf(mid - a1) : 0.f;
          if (lane == 0) {
            vs[VEC_FLAG] = fact ? 1.f : 0.f;
            vs[VEC_FLAG + 1] = mid;
          }
        }
        if (lane == 0) {
          int* vi = reinterpret_cast<int*>(vs) + VEC_ITEM;
          vi[0] = done ? -1 : (int)gitem;
          vi[1] = jj;
          vi[2] = s;
          vi[3] = cur.fx;
        }
        __syncwarp();
        if (!done) {
          if (L < CHUNK) {
            // rows past the sequence end: zero K and Q so they add nothing to any product
            if (!(ok = warp_wait(&bars[P_FULL + 2 * pp + ub], (use >> 1) & 1, cx))) break;
            const int rows = CHUNK - L;
            for (int idx = lane; idx < 4 * rows * 8; idx += 32) {
              const int t4 = idx / (rows * 8), rem = idx % (rows * 8);
              const int row = L + rem / 8, ch = rem % 8, pnl = t4 & 1, which = t4 >> 1;
              uint8_t* tb = kq + pnl * P_KQ_PANEL + (which == 1 ? kq_q : kq_k);
              *reinterpret_cast<uint4*>(tb + row * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[P_HEAD + 2 * pp + ub]);
        if (done) break;
        // the next item's gate/beta loads and L2 prefetches, then the claim after it (the
        // atomic's round trip is waited for only here, off the way to this use's HEAD)
        const Next nxt = fetch(gnn);
        if (nxt.g < geo.total) {
          gnn = claim_end(inflight);
          inflight = claim_start();
        }
        cur = nxt;
      }
      // never leave with a tile copy in flight (the last two uses may each have one)
      for (int u = last - 1; u <= last; ++u)
        if (u >= 0) mbar_wait(&bars[P_FULL + 2 * pp + (u & 1)], (u >> 1) & 1, 100000000ull);
      __syncwarp();
    } else {
      // ------------------------------------------------------------ KQ issuer
      // warp 1 issues pipeline 0's [K;Q] K^T, warp 3 pipeline 1's: item u's as soon as its
      // tiles have landed (FULL) and the pipeline has read out item u-1's (KQFREE).
      const int pp = warp >> 1;
      if (lane == 0) {
        const uint32_t base = sb + pp * P_STRIDE, tp = tm + 256 * pp;
        const uint32_t kq_k = pp ? 8192u : 0u;
        for (int u = 0;; ++u) {
          if (!wait_bar(&bars[P_HEAD + 2 * pp + (u & 1)], (u >> 1) & 1, cx)) { raise_abort(cx); break; }
          if (reinterpret_cast<const int*>(vec_of(pp, u))[VEC_ITEM] < 0) break;
          if (!wait_bar(&bars[P_FULL + 2 * pp + (u & 1)], (u >> 1) & 1, cx) ||
              (u > 0 && !wait_bar(&bars[P_KQFREE + pp], (u - 1) & 1, cx))) {
            raise_abort(cx);
            break;
          }
          tc_fence_after();
          const uint32_t kq = base + P_KQ + (u & 1) * P_KQ_BUF;
          const uint64_t aq = sdesc_sw128(kq, 0, 1024);
          const uint64_t bk = sdesc_sw128(kq + kq_k, 0, 1024);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t o = (uint64_t)(((kk >> 2) * P_KQ_PANEL + (kk & 3) * 32) >> 4);
            mma_bf16(tp + TP_KQ, aq + o, bk + o, ID_N64, kk > 0 ? 1u : 0u);
          }
          mma_commit(&bars[P_KQDONE + pp]);
        }
        if (*cx.abort_l) {
          // leave no product running into the TMEM that the CTA frees on its way out
          mma_commit(&bars[P_DRAIN + 2 * pp]);
          mbar_wait(&bars[P_DRAIN + 2 * pp], 0, 100000000ull);
        }
      }
      __syncwarp();
    }
  } else if (warp < 12) {
    reg_alloc<RP_PIPE>();
    // ---------------------------------------------------------- pipelines
    const int pp = (warp - 4) >> 2;
    const int r = ((warp & 3) << 5) + lane;          // TMEM lane
    const int bid = BAR_PREP0 + pp;
    const uint32_t tl = tm + 256 * pp + ((uint32_t)((warp & 3) * 32) << 16);
    uint8_t* base = sm + pp * P_STRIDE;
    float* AT = reinterpret_cast<float*>(base + P_AT);
    // the A/T area, once T' and T'' are built, is this warp's store staging (4 KB); the
    // Ahat rows, stored during phase 1 of the solve, are staged in the X area
    uint8_t* stage = base + P_AT + (warp & 3) * 4096;
    uint8_t* stage_ah = base + P_X + ((warp & 3) & 1) * 4096;
    // TMEM lanes (rows of [K;Q] K^T) of this pipeline's A rows: pipeline 1 holds [Q;K], so
    // its solve's phase 1 runs on the other two SM sub-partitions than pipeline 0's
    const bool arow = (pp == 0) == (r < 64);
    // T' and -T'' are zero above the diagonal blocks for every item: the solve writes only
    // the blocks on and below the diagonal
    for (int idx = r; idx < 2 * 512; idx += 128)
      reinterpret_cast<uint4*>(base + P_T1)[idx] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    bool ok = true;
    bool pend = false;     // the previous item's record stores may be in flight
    bool w_issued = false;     // thread r == 0: it has issued a (-W)^T product
    for (int use = 0; ok; ++use) {
      const float* vs = vec_of(pp, use);
      // the controller's item slot and vectors for this use (HEAD), then the chunk's
      // [K;Q] K^T; meanwhile the previous record's stores land (then it may be released)
      if (!(ok = group_wait(&bars[P_HEAD + 2 * pp + (use & 1)], (use >> 1) & 1, bid, 128, cx))) break;
      if (pend) record_landed(lane, &bars[P_PUB + pp]);
      pend = false;
      const int gi = reinterpret_cast<const int*>(vs)[VEC_ITEM];
      if (gi < 0) break;
      const int jj = reinterpret_cast<const int*>(vs)[VEC_ITEM + 1];
      const int s = reinterpret_cast<const int*>(vs)[VEC_ITEM + 2];
      const int fx = reinterpret_cast<const int*>(vs)[VEC_ITEM + 3];
      if (!(ok = group_wait(&bars[P_KQDONE + pp], use & 1, bid, 128, cx))) break;
      tc_fence_after();
      uint32_t ah[32];     // rows 64-127: this row of Ahat (BF16 pairs), stored at the end
      {
        const bool fact = vs[VEC_FLAG] != 0.f;
        const int i = r & 63;
        const float gi = vs[VEC_GAM + i], epi = vs[VEC_EP + i];
        const float bi = arow ? vs[VEC_BETA + i] : 1.f;
        float x[64];
        tmem_ld64(tl + TP_KQ, x);
        if (fact) {
          const float f = bi * epi;
          const float4* em4 = reinterpret_cast<const float4*>(vs + VEC_EM);
#pragma unroll
          for (int j4 = 0; j4 < 16; ++j4) {
            const float4 e4 = em4[j4];
            x[4 * j4] *= f * e4.x;
            x[4 * j4 + 1] *= f * e4.y;
            x[4 * j4 + 2] *= f * e4.z;
            x[4 * j4 + 3] *= f * e4.w;
          }
        } else {
#pragma unroll
          for (int jx = 0; jx < 64; ++jx) x[jx] *= bi * expf(jx <= i ? gi - vs[VEC_GAM + jx] : 0.f);
        }
        if (arow) {            // A_ij = beta_i Gamma_ij (k_i . k_j), j < i (the solve
                               // reads nothing on or above the diagonal)
          float4* row = reinterpret_cast<float4*>(AT + i * SOLVE_LD);
#pragma unroll
          for (int j4 = 0; j4 < 16; ++j4) {
            const int jx = 4 * j4;
            if (jx < i) row[j4] = make_float4(x[jx], x[jx + 1], x[jx + 2], x[jx + 3]);
          }
        } else {               // Ahat_ij = Gamma_ij (q_i . k_j), j <= i
#pragma unroll
          for (int jx = 0; jx < 64; ++jx)
            if (jx > i) x[jx] = 0.f;
          pack64(x, ah);
        }
      }
      // this warp's part of the KQ accumulator is read out (four arrivals): the issuer
      // may start the next item's [K;Q] K^T
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[P_KQFREE + pp]);
      // T = (I + A)^{-1} as T' = T diag(beta) and -T'' = -T diag(beta e^gamma).  Phase 1
      // needs only the rows this warp wrote; meanwhile the Ahat warps store their rows to
      // the record's ring slot once the publisher has seen it free (s mod nslot).
      uint8_t* rec = p.ring + ((size_t)jj * p.nslot + (s & (p.nslot - 1))) * REC_BYTES;
      // state replay: the record's copy for the backward (Ahat, (-W)^T and the decays)
      uint8_t* rec2 = kCopy ? p.fac + (size_t)fx * REC2_BYTES : nullptr;
      bool ok1 = true;
      if (arow) {
        solve::half(AT, base + P_T1, base + P_T2, vs, (warp & 3) & 1, lane);
      } else {
        ok1 = __all_sync(0xffffffffu, wait_bar(&bars[P_SLOTOK + pp], use & 1, cx)) != 0;
        if (ok1 && !summ)
          store_rows<kCopy>(rec + R_AH, kCopy ? rec2 + R_AH : nullptr, stage_ah,
                            ((warp & 3) * 32) & 63, ah, lane);
      }
      if (!(ok = named_bar_and(bid, 128, ok1))) {
        if (r == 0) raise_abort(cx);
        break;
      }
      // the two heavier blocks (row block 3) go to sub-partitions 2, 3 in pipeline 0 and to
      // 0, 1 in pipeline 1, so that each sub-partition gets one of them
      if (((warp & 3) < 2) == (pp == 0))
        solve::lower<0>(AT, base + P_T1, base + P_T2, vs, warp & 1, BAR_SOLVE0 + pp, lane);
      else
        solve::lower<1>(AT, base + P_T1, base + P_T2, vs, warp & 1, BAR_SOLVE0 + pp, lane);
      fence_proxy_async_smem();
      named_bar(bid, 128);
      if (r == 0) {
        // (-W)^T = K^T (-T'')^T, issued here as soon as -T'' is complete (the previous
        // item's (-W)^T was read out before its last barrier); its commits tell this
        // pipeline (WDONE) and the feeder (ITEMFREE: the tile buffer is free)
        tc_fence_after();
        const uint32_t kq = sb + pp * P_STRIDE + P_KQ + (use & 1) * P_KQ_BUF;
        const uint64_t ak = sdesc_sw128(kq + (pp ? 8192u : 0u), P_KQ_PANEL, 1024);
        const uint64_t b2 = sdesc_sw128(sb + pp * P_STRIDE + P_T2, 0, 1024);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16(tm + 256 * pp + TP_WT, ak + (uint64_t)(kk * 2048 >> 4), b2 + (uint64_t)(kk * 2),
                   ID_AMN, kk > 0 ? 1u : 0u);
        mma_commit(&bars[P_WDONE + pp]);
        mma_commit(&bars[P_ITEMFREE + 2 * pp + (use & 1)]);
        w_issued = true;
        // T' goes to the record as it is: the chain CTA's B operand of U^T = V^T T'^T
        bulk_s2g(rec + R_T1, base + P_T1, 8192);
        bulk_commit();
      }
      if (!(ok = group_wait(&bars[P_WDONE + pp], use & 1, bid, 128, cx))) break;
      tc_fence_after();
      {
        float x[64];
        uint32_t u[32];
        tmem_ld64(tl + TP_WT, x);
        pack64(x, u);
        store_rows<kCopy>(rec + R_W, kCopy ? rec2 + R_W : nullptr, stage, (warp & 3) * 32, u, lane);
      }
      // the decays e^{gamma_C - gamma_j}, e^{gamma_i} and e^{gamma_C}
      if (r < 64) reinterpret_cast<float*>(rec + R_VEC + V_DEC)[r] = vs[VEC_DEC + r];
      else reinterpret_cast<float*>(rec + R_VEC + V_EG)[r - 64] = vs[VEC_EG + r - 64];
      if (r == 0) reinterpret_cast<float*>(rec + R_VEC + V_GC)[0] = vs[VEC_EG + 63];
      if constexpr (kCopy) {
        if (r < 64) reinterpret_cast<float*>(rec2 + R_VEC + V_DEC)[r] = vs[VEC_DEC + r];
        else reinterpret_cast<float*>(rec2 + R_VEC + V_EG)[r - 64] = vs[VEC_EG + r - 64];
        if (r == 0) reinterpret_cast<float*>(rec2 + R_VEC + V_GC)[0] = vs[VEC_EG + 63];
      }
      // The A/T and X areas and T', which the next item writes again, are free once every
      // warp has seen its own stores land (record_landed at the next item's start) and
      // passed the KQDONE barrier after that; this barrier is for the vector slot.
      pend = true;
      tc_fence_before();
      named_bar(bid, 128);
      if (r == 0) mbar_arrive(&bars[P_VECFREE + 2 * pp + (use & 1)]);
    }
    // the last record (and, on the abort path, every bulk store) lands before leaving
    if (pend) record_landed(lane, &bars[P_PUB + pp]);
    else if (lane == 0) bulk_wait_all();
    if (w_issued && *cx.abort_l) {
      // leave no (-W)^T product running into the TMEM that the CTA frees on its way out
      mma_commit(&bars[P_DRAIN + 2 * pp + 1]);
      mbar_wait(&bars[P_DRAIN + 2 * pp + 1], 0, 100000000ull);
    }
  } else {
    reg_dealloc<RP_AUX>();
    const int pp = warp & 1;
    if (warp >= 14) {
      // ------------------------------------------------------------ publisher
      // Record u-1 is released once its stores have landed (PUB: the pipeline's warps
      // arrive when they start item u), and item u's ring slot must have been copied out
      // by its chain CTA before the pipeline writes to it (SLOTOK).
      if (lane == 0) {
        int pj = -1, ps = 0;
        long long pg = -1;
        for (int u = 0;; ++u) {
          if (!wait_bar(&bars[P_HEAD + 2 * pp + (u & 1)], (u >> 1) & 1, cx)) { raise_abort(cx); break; }
          const int* vi = reinterpret_cast<const int*>(vec_of(pp, u)) + VEC_ITEM;
          const int g = vi[0], jj = vi[1], s = vi[2];
          if (pj >= 0) {
            if (!wait_bar(&bars[P_PUB + pp], (u - 1) & 1, cx)) { raise_abort(cx); break; }
            if (pg != p.drop_item)
              st_release_u32(p.ready + (size_t)pj * FLAG_STRIDE + (ps & (p.nslot - 1)),
                             (uint32_t)ps + 1);
            pj = -1;
          }
          if (g < 0) break;
          const uint32_t need = (uint32_t)(s - p.nslot + 1);
          const bool ok = s < p.nslot ||
                          (poll_ge(p.consumed + (size_t)jj * FLAG_STRIDE, need, cx) &&
                           (!summ || poll_ge(p.consumed + (size_t)(jj + geo.nch) * FLAG_STRIDE,
                                             need, cx)));
          if (!ok) {
            raise_abort(cx);
            break;
          }
          mbar_arrive(&bars[P_SLOTOK + pp]);
          pj = jj;
          ps = s;
          pg = g;
        }
      }
      __syncwarp();
    }
  }
}

// kOut: the launch has output products (the forward); without them (state replay, segment
// summaries) the chain CTAs keep three chunks in flight.
template <bool kCopy, bool kOut>
__global__ void __launch_bounds__(NTHR, 1)
    gdn_fwd_split_kernel(const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmQ4,
                         const __grid_constant__ CUtensorMap tmK4,
                         const __grid_constant__ CUtensorMap tmV4,
                         const __grid_constant__ CUtensorMap tmO, const SplitParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(sm);
  const bool is_chain = (int)blockIdx.x < p.nch * (p.twin ? 2 : 1);
  uint8_t* bar_area = sm + (is_chain ? C_BAR : P_BAR);
  uint64_t* bars = reinterpret_cast<uint64_t*>(bar_area);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_area + 256);
  volatile int* abort_l = reinterpret_cast<volatile int*>(bar_area + 264);
  const int tid = threadIdx.x, warp = tid >> 5;
  int* len_s = reinterpret_cast<int*>(bar_area + BAR_BYTES);
  int* sort_s = len_s + 64;
  int* seg_s = sort_s + 64;
  long long* seg_w = reinterpret_cast<long long*>(seg_s + 66);
  const bool packed = p.cu || p.bounds;
  if (packed && tid < p.nch) {
    len_s[tid] = p.lenj[tid];
    sort_s[tid] = p.sortj[tid];
  }
  Geo geo;
  const Ctx cx{abort_l, &p};

  if (tid == 0) {
    if (is_chain) {
      for (int i = 0; i < C_COUNT; ++i) mbar_init(&bars[i], 1);
      // a record buffer is free once its chunk's products are done (MMA commit) and its
      // output tile, staged in it, has been read out (output warps)
      for (int i = 0; i < 3; ++i) mbar_init(&bars[C_RECFREE + i], kOut ? 2 : 1);
    } else {
      for (int i = 0; i < P_COUNT; ++i) mbar_init(&bars[i], 1);
      mbar_init(&bars[P_KQFREE], 4);
      mbar_init(&bars[P_KQFREE + 1], 4);
      mbar_init(&bars[P_PUB], 4);
      mbar_init(&bars[P_PUB + 1], 4);
    }
    *abort_l = 0;
    fence_mbar_init();
    if (is_chain) {
      prefetch_tmap(&tmK4);
      if (!p.twin) prefetch_tmap(&tmQ4);
      prefetch_tmap(&tmV4);
      if (p.out) prefetch_tmap(&tmO);
    } else {
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmQ);
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (packed) {
    if (tid == 0) Geo::build_table(p.nch, len_s, sort_s, seg_s, seg_w);
    __syncthreads();
  }
  const uint32_t tm = *tmem_slot;
  geo.init(p, len_s, sort_s);

  if (is_chain)
    chain_cta<kOut>(&tmQ4, &tmK4, &tmV4, &tmO, p, geo, sm, sb, bars, tm, cx);
  else
    prep_cta<kCopy>(&tmQ, &tmK, &tmQ4, &tmK4, &tmV4, p, geo, sm, sb, bars, tm, cx);

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tm, TM_COLS);
  }
}

// Packed inputs and token ranges: each chain's first stream position in its chain CTA, each chain CTA's
// stream length, and the chain CTAs ordered by stream length (longest first).  One CTA.
__global__ void split_setup_kernel(const SplitParams p) {
  __shared__ int len_s[MAX_NCH];
  const int NH = p.N * p.H, nch = p.nch, tid = threadIdx.x;
  if (p.fac && tid == 0) {
    // the backward's slot numbering: each sequence's chunks follow those of the one before
    int acc = 0;
    for (int n = 0; n < p.N; ++n) {
      p.slot0[n] = acc;
      int64_t b, e;
      chain_span(p, n * p.H, b, e);
      acc += (int)n_chunks(e - b);
    }
  }
  for (int x = tid; x < NH; x += blockDim.x) {
    int64_t b, e;
    chain_span(p, x, b, e);
    p.sstart[x] = (int)n_chunks(e - b);
  }
  __syncthreads();
  if (tid < nch) {
    int acc = 0;
    for (int x = tid; x < NH; x += nch) {
      const int n = p.sstart[x];
      p.sstart[x] = acc;
      acc += n;
    }
    len_s[tid] = acc;
    p.lenj[tid] = acc;
  }
  __syncthreads();
  if (tid < nch) {
    int r = 0;
    for (int i = 0; i < nch; ++i)
      r += (len_s[i] > len_s[tid]) || (len_s[i] == len_s[tid] && i < tid);
    p.sortj[r] = tid;
  }
}

// Workspace: [0, 256) status word; [256, 260) abort flag; [384, 388) the item counter of
// the preparation CTAs; from 512 consumed (one 128-byte line per chain CTA, P twins
// included), then ready (one line per stream-owning chain CTA): the flags polled by
// different CTAs never share a line; the ring from 32768 (one per stream-owning chain
// CTA); then (packed inputs and token ranges) the chain stream starts [N*H], stream
// lengths [64] and their order [64].
constexpr size_t WS_ABORT = 256, WS_NEXT = 384, WS_CONSUMED = 512,
                 WS_READY = WS_CONSUMED + 2 * MAX_NCH * 128;
constexpr size_t WS_FLAGS_END = WS_READY + (size_t)MAX_NCH * 128;
constexpr size_t WS_RING = 32768;
static_assert(WS_FLAGS_END <= WS_RING, "workspace flags");

int chain_ctas(int N, int H) {
  const long long nh = (long long)N * H;
  return (int)(nh < MAX_NCH ? nh : MAX_NCH);
}
// segment summaries: chain CTAs that own streams (each has a P twin)
int summary_chain_ctas(int R, int H) {
  const long long nh = (long long)R * H;
  if (nh <= SF_SUMMARY_CHAINS) return (int)nh;
  // as few chain CTAs as keep the most chains per CTA at ceil(nh / SF_SUMMARY_CHAINS); the
  // SMs left over prepare records
  const long long k = (nh + SF_SUMMARY_CHAINS - 1) / SF_SUMMARY_CHAINS;
  return (int)((nh + k - 1) / k);
}
size_t ws_ring_end(int nch) { return WS_RING + (size_t)nch * NSLOT_MAX * REC_BYTES; }
size_t ws_total(int nch, int N, int H) {
  return ws_ring_end(nch) + (((size_t)N * H + 2 * MAX_NCH + N) * sizeof(int) + 255) / 256 * 256;
}

// The launch shared by the forward, the state replay and the segment summaries: flags
// reset, the packed-geometry setup, tensor maps, then one cooperative launch over every
// SM (chain CTAs first).  p arrives with its inputs, outputs, mode and nch set.
cudaError_t launch_split(SplitParams& p, const void* q, const void* k, const void* v, void* out,
                         int chain_blocks, void* ws, int* status, cudaStream_t st) {
  int dev = 0, nsm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int nprep = nsm - chain_blocks;
  if (nprep < 1) return cudaErrorInvalidConfiguration;
  const int rows = p.B * p.T;
  // the preparation loads [K;Q] panel by panel (3-D maps); the state chains load whole
  // tiles, prefetch and store through the 4-D views
  CUtensorMap mq, mk, mq4, mk4, mv4;
  if (!make_bf16_map(&mk, k, rows, p.HK) || !make_bf16_map_4d(&mk4, k, rows, p.HK) ||
      !make_bf16_map_4d(&mv4, v, rows, p.H))
    return cudaErrorInvalidValue;
  mq = mk;   // summaries have no q: K stands in (its products are not used)
  mq4 = mk4;
  if (q && (!make_bf16_map(&mq, q, rows, p.HK) || !make_bf16_map_4d(&mq4, q, rows, p.HK)))
    return cudaErrorInvalidValue;
  // the state replay that keeps the records for the backward takes the copying instantiation
  const bool with_out = p.out && !p.twin;
  if (p.fac && with_out) return cudaErrorInvalidValue;   // the replay has no output
  const void* kern =
      p.fac      ? reinterpret_cast<const void*>(gdn_fwd_split_kernel<true, false>)
      : with_out ? reinterpret_cast<const void*>(gdn_fwd_split_kernel<false, true>)
                 : reinterpret_cast<const void*>(gdn_fwd_split_kernel<false, false>);
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  char* w = reinterpret_cast<char*>(ws);
  e = cudaMemsetAsync(w + WS_ABORT, 0, WS_FLAGS_END - WS_ABORT, st);
  if (e != cudaSuccess) return e;
  const int NH = p.N * p.H;
  p.qk_group = p.H / p.HK;
  p.status = status;
  p.abort_g = reinterpret_cast<int*>(w + WS_ABORT);
  p.next_item = reinterpret_cast<uint32_t*>(w + WS_NEXT);
  p.consumed = reinterpret_cast<uint32_t*>(w + WS_CONSUMED);
  p.ready = reinterpret_cast<uint32_t*>(w + WS_READY);
  p.ring = reinterpret_cast<uint8_t*>(w + WS_RING);
  // the short ring only where every chain CTA owns one chain of the same length (dense
  // inputs, N H <= 64): with several chains per CTA, or packed lengths, the streams'
  // lengths differ and the preparation needs the slack of the long one
  const bool one_chain_each = !p.cu && !p.bounds && (long long)p.N * p.H <= MAX_NCH;
  p.nslot = (with_out && one_chain_each) ? NSLOT_OUT : NSLOT_MAX;
  p.sstart = reinterpret_cast<int*>(w + ws_ring_end(p.nch));
  p.lenj = p.sstart + (size_t)NH;
  p.sortj = p.lenj + MAX_NCH;
  p.slot0 = p.sortj + MAX_NCH;
  p.nprep = nprep;
  p.wait_limit = kWaitLimitCycles;
  p.drop_item = -1;
  if (g_inject.item >= 0) {
    p.drop_item = g_inject.item;
    p.wait_limit = g_inject.wait_limit;
    g_inject = InjectedTimeout{};
  }
  if (p.cu || p.bounds) {
    split_setup_kernel<<<1, 256, 0, st>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  // the output map (the K map stands in when there is no output: it is never used then)
  CUtensorMap mo = mk4;
  if (out && !make_bf16_map_4d(&mo, out, rows, p.H)) return cudaErrorInvalidValue;
  void* args[] = {&mq, &mk, &mq4, &mk4, &mv4, &mo, &p};
  return cudaLaunchCooperativeKernel(kern,
                                     dim3(chain_blocks + nprep), dim3(NTHR), args, SMEM_ALLOC, st);
}

}  // namespace

void inject_split_timeout(long long item, long long wait_limit_cycles) {
  g_inject.item = item;
  g_inject.wait_limit = wait_limit_cycles;
}

size_t split_fwd_workspace(int N, int H) { return ws_total(chain_ctas(N, H), N, H); }
size_t split_summary_workspace(int R, int H) { return ws_total(summary_chain_ctas(R, H), R, H); }

cudaError_t launch_split_fwd(const ChainParams& cp, void* ws, int* status, cudaStream_t st) {
  if (cp.T <= 0 || cp.N < 1 || cp.H < 1 || (cp.cu && cp.B != 1) || (cp.HK > 0 && cp.H % cp.HK))
    return cudaErrorInvalidValue;
  SplitParams p{};
  p.g = cp.g;
  p.beta = cp.beta;
  p.s0 = cp.s0;
  p.out = reinterpret_cast<__nv_bfloat16*>(cp.out);
  p.final_state = cp.final_state;
  p.ckpt = cp.ckpt;
  p.fac = cp.ckpt ? reinterpret_cast<uint8_t*>(cp.fac) : nullptr;
  p.pool = cp.pool;
  p.state_idx = cp.state_idx;
  p.has_init = cp.has_init;
  p.num_slots = cp.num_slots;
  p.cu = cp.cu;
  p.B = cp.B;
  p.T = cp.T;
  p.H = cp.H;
  p.N = cp.N;
  p.HK = cp.HK > 0 ? cp.HK : cp.H;
  p.nch = chain_ctas(cp.N, cp.H);
  p.scale = cp.scale;
  return launch_split(p, cp.q, cp.k, cp.v, cp.out, p.nch, ws, status, st);
}

cudaError_t launch_split_summary(const ChainParams& cp, void* ws, int* status, cudaStream_t st) {
  if (cp.T <= 0 || cp.N < 1 || cp.H < 1 || !cp.bounds || !cp.P || !cp.E || (cp.HK > 0 && cp.H % cp.HK))
    return cudaErrorInvalidValue;
  SplitParams p{};
  p.g = cp.g;
  p.beta = cp.beta;
  p.bounds = cp.bounds;
  p.sumP = cp.P;
  p.sumE = cp.E;
  p.twin = 1;
  p.B = cp.B;
  p.T = cp.T;
  p.H = cp.H;
  p.N = cp.N;
  p.HK = cp.HK > 0 ? cp.HK : cp.H;
  p.nch = summary_chain_ctas(cp.N, cp.H);
  p.scale = 1.f;
  return launch_split(p, nullptr, cp.k, cp.v, nullptr, 2 * p.nch, ws, status, st);
}

}  // namespace sfg
