// chain_tc.cuh -- the body of the backward's reverse cotangent chain on tcgen05 (BF16,
// K = V = 128): one CTA per (sequence, head) chain, used by the chain's own kernel
// (bwd_chain_tc.cu) and by the launch that runs it beside the token gradients
// (bwd_grad_tc.cu).
//
// StateFlow section 3.1, Eq. 6-7 (the chunk algebra differentiated): walking a sequence
// backwards, per chunk with exit cotangent dS,
//     dDelta^T = scale dO^T Aqk + (dS K^T) diag(dec)
//     dS      <- e^{gamma_C} dS + (diag(scale e^gamma) dO)^T Q - dDelta^T W,
// and the cotangent left at the sequence start is d_initial_state.  One CTA per
// (sequence, head) chain keeps dS FP32 in TMEM (the 128 v rows on the lanes, the 128 k
// columns) with a BF16 copy there as the A operand of dS K^T.  Per chunk (all M = 128):
//   P1  = dO^T Aqk              N = 64,  K = 64    (independent of dS: issued ahead)
//   X   = dS K^T                N = 64,  K = 128   (the chain's critical path)
//   dS += dO^T Qg               N = 128, K = 64    (Qg = scale diag(e^gamma) Q; once the
//                                                   state warps scaled dS)
//   dS += dDelta^T (-W)         N = 128, K = 64    (A: dDelta^T BF16 in TMEM)
// The factors are the backward's chunk records of chunk_record.cuh (Aqk = Ahat, (-W)^T, the
// decays and Qg), kept by the state replay with Qg added by qg_kernel (bwd_chain_tc.cu), or
// made whole by mma_bwd_factor_kernel<128>, one bulk copy each; K and dO come by TMA; two
// chunks are in flight.  Each chunk's exit cotangent goes to the tape as the BF16 swizzled
// tile the token-gradient kernel reads.
//
// Warps: 0 loads, 1 issues the products (one thread), 4-11 hold the cotangent (two
// warpgroups, one 64-column half each); in a launch shared with the token gradients
// (bwd_grad_tc.cu), 12-15 idle, and the tape count is published after each tile.  Every
// wait is bounded; a thread that gives up writes SF_ERR_TIMEOUT to the status word and
// raises the CTA's abort flag, which every waiting thread polls; the issuer drains its
// products before the TMEM is freed.
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>

#include "api_internal.cuh"
#include "chunk_record.cuh"
#include "common.cuh"
#include "simt_chunk.cuh"
#include "tc_ptx.cuh"

namespace sfg {
namespace chaintc {

using namespace tc;

constexpr int D = 128;
constexpr int NT = 384;
constexpr int NB = 2;                   // chunk buffers
constexpr uint32_t PANEL = 8192;        // 64-row tile panel
constexpr uint32_t B_FAC = 0;           // the chunk record (R_* offsets, with Qg)
constexpr uint32_t B_K = 50176;         // K [64 j][128 k]
constexpr uint32_t B_DO = 66560;        // dO [64 i][128 v]
constexpr uint32_t BUF = 82944;
constexpr uint32_t O_BAR = NB * BUF;
constexpr uint32_t SMEM_ALLOC = O_BAR + 256 + 1024;
static_assert(B_K >= REC2_BYTES && B_K % 1024 == 0 && B_DO == B_K + 2 * PANEL &&
              BUF == B_DO + 2 * PANEL && BUF % 1024 == 0, "chain buffer");
static_assert(R_W % 1024 == 0 && R_AH % 1024 == 0 && R_QG % 1024 == 0, "tile alignment");
static_assert(SMEM_ALLOC <= 232448, "shared memory");

// TMEM columns (512 allocated)
constexpr uint32_t TM_DS = 0;      // dS FP32 [128 v][128 k]
constexpr uint32_t TM_DSB = 128;   // dS BF16 pairs (64 columns)
constexpr uint32_t TM_P1 = 192;    // dO^T (scale Aqk)
constexpr uint32_t TM_X = 256;     // dS K^T
constexpr uint32_t TM_DDB = 320;   // dDelta^T BF16 pairs (32 columns)

constexpr uint32_t ID_P1 = idesc_bf16(128, 64, true, true);    // A, B MN-major
constexpr uint32_t ID_X = idesc_bf16(128, 64, false, false);   // A in TMEM, B K-major
constexpr uint32_t ID_U1 = idesc_bf16(128, 128, true, true);   // A, B MN-major, N = 128
constexpr uint32_t ID_U2 = idesc_bf16(128, 128, false, false); // A in TMEM, B K-major, N = 128

enum { C_FULL = 0, C_LANDED = 2, C_FREE = 4, C_XDONE = 6, C_DREADY, C_SREADY, C_SSCALED,
       C_SUDONE, C_DRAIN, C_COUNT };
constexpr int BAR_STATE = 1;
constexpr unsigned long long WAIT_NS = 2000000000ull;

struct Cx {
  int* status;
  volatile int* abort;
};

__device__ __forceinline__ void note_timeout(const Cx& cx, uint32_t what) {
  *cx.abort = 1;
  if (!cx.status) return;
  atomicCAS(cx.status, 0, (int)SF_ERR_TIMEOUT);
  atomicCAS(cx.status + 1, 0,
            (int)(0x40000000u | (blockIdx.x << 12) | ((threadIdx.x >> 5) << 6) | (what & 63u)));
}

// Bounded wait; false when it gave up or another thread of the CTA did.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, const Cx& cx) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if (*cx.abort) return false;
    if (globaltimer_ns() - t0 > WAIT_NS) {
      note_timeout(cx, (smem_u32(bar) & 255u) >> 3);
      return false;
    }
  }
}

// The 256 state threads wait together and agree on the outcome.
__device__ __forceinline__ bool group_wait(uint64_t* bar, uint32_t parity, const Cx& cx) {
  return named_bar_and(BAR_STATE, 256, wait_bar(bar, parity, cx));
}

__device__ __forceinline__ uint64_t kstep_k(int kk) {
  return (uint64_t)(((uint32_t)(kk >> 2) * PANEL + (uint32_t)(kk & 3) * 32u) >> 4);
}
__device__ __forceinline__ uint64_t kstep_mn(int kk) { return (uint64_t)(kk * 2048 >> 4); }

// Row v of one panel of a tape tile from the 64 values' BF16 pairs u (16-byte chunk c of row
// v at ((c ^ (v mod 8)) << 4)).
__device__ __forceinline__ void store_tile_row(uint8_t* row, int v, const uint32_t (&u)[32]) {
#pragma unroll
  for (int c = 0; c < 8; ++c)
    *reinterpret_cast<uint4*>(row + ((c ^ (v & 7)) << 4)) =
        make_uint4(u[4 * c], u[4 * c + 1], u[4 * c + 2], u[4 * c + 3]);
}

// Fused launch: the tape tiles this CTA has written so far, published for the token-gradient
// CTAs (every cotangent thread's stores, then one release store of the count).
__device__ __forceinline__ void publish_tape(uint32_t* flag, uint32_t count, int st_t) {
  if (!flag) return;
  __threadfence();
  named_bar(BAR_STATE, 256);
  if (st_t == 0) st_release_u32(flag, count);
}

// The chain x = n H + h of p: sm, 1024-aligned shared memory of SMEM_ALLOC bytes; tape_flag:
// the published tape count (fused launch) or NULL.  A fused launch's CTA leaves with its
// TMEM freed, its barriers invalidated and 128 registers per thread.
// Registers of the loader / issuer warpgroup in a fused launch.
constexpr int kCtlRegs = 56;

template <bool kFused>
__device__ __forceinline__ void chain_cta(const CUtensorMap* mk, const CUtensorMap* mdo,
                                          const ChainParams& p, const float* fac, int x,
                                          uint32_t* tape_flag, uint8_t* sm) {
  const uint32_t sb = smem_u32(sm);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + O_BAR);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + O_BAR + 8 * C_COUNT);
  int* abort_s = reinterpret_cast<int*>(sm + O_BAR + 8 * C_COUNT + 4);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = p.H, h = x % H, n = x / H;
  const int hk = qk_head(h, H, p.HK);
  int64_t bos, eos;
  seq_span(n, p.B, p.T, p.cu, bos, eos);
  const int nc = (int)n_chunks(eos - bos);
  const int64_t slot0 = chunk_slot_base(n, p.B, p.T, p.cu);
  const Cx cx{p.status, abort_s};

  if (tid == 0) {
    for (int i = 0; i < C_COUNT; ++i) mbar_init(&bars[i], 1);
    *abort_s = 0;
    fence_mbar_init();
    if (nc > 0) {
      prefetch_tmap(mk);
      prefetch_tmap(mdo);
    }
  }
  if (warp == 0) tmem_alloc(tslot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tslot;

  // In a fused launch of 512 threads (128 registers each) the cotangent warps take 168 and
  // the others give theirs up, each role's code under its own register limit; a launch of
  // its own has 168 for every thread.
  if (warp < 4) {
    if constexpr (kFused) reg_dealloc<kCtlRegs>();
    if (warp == 0) {
      // ------------------------------------------------------------ loader
      // chunk ci = nc - 1 - s of the sequence into buffer s % NB, once the chunk two back has
      // had its last product; a chunk cut short by the sequence end lands on its own barrier
      // first, and its K and dO rows past the end are zeroed (rows of other tokens, or NaN
      // padding, must not reach the products).
      bool ok = true;
      int issued = 0;
      uint32_t landed = 0, part_of = 0;   // per buffer: LANDED parity, partial chunk
      for (int s = 0; s < nc && ok; ++s) {
        const int b = s % NB, ci = nc - 1 - s;
        const int64_t c0 = bos + (int64_t)ci * CHUNK;
        const int L = (eos - c0) < CHUNK ? (int)(eos - c0) : CHUNK;
        const bool part = L < CHUNK;
        uint8_t* buf = sm + b * BUF;
        if (lane == 0) ok = s < NB || wait_bar(&bars[C_FREE + b], ((s - NB) / NB) & 1, cx);
        if (!(ok = __shfl_sync(0xffffffffu, ok, 0) != 0)) break;
        part_of = (part_of & ~(1u << b)) | ((part ? 1u : 0u) << b);
        uint64_t* bar = part ? &bars[C_LANDED + b] : &bars[C_FULL + b];
        const uint32_t pl = (landed >> b) & 1u;
        if (part) landed ^= 1u << b;
        if (lane == 0) {
          const uint8_t* src =
              reinterpret_cast<const uint8_t*>(fac) + ((size_t)(slot0 + ci) * H + h) * REC2_BYTES;
          mbar_arrive_expect_tx(bar, REC2_BYTES + 4 * PANEL);
          bulk_g2s(buf + B_FAC, src, REC2_BYTES, bar);
  #pragma unroll
          for (int pp = 0; pp < 2; ++pp) {
            tma_load_3d(buf + B_K + pp * PANEL, mk, bar, 64 * pp, hk, (int)c0);
            tma_load_3d(buf + B_DO + pp * PANEL, mdo, bar, 64 * pp, h, (int)c0);
          }
        }
        issued = s + 1;
        if (part) {
          bool okl = true;
          if (lane == 0) okl = wait_bar(bar, pl, cx);
          if (!(ok = __shfl_sync(0xffffffffu, okl, 0) != 0)) break;
          const int per = (CHUNK - L) * 8;   // 16-byte chunks per panel
          for (int idx = lane; idx < 4 * per; idx += 32) {
            const int tile = idx / per, rr = idx % per;   // K, dO panels (contiguous)
            uint8_t* t = buf + B_K + tile * PANEL;
            *reinterpret_cast<uint4*>(t + (L + rr / 8) * 128 + (rr % 8) * 16) =
                make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[C_FULL + b]);
        }
      }
      if (lane == 0 && !ok) {
        // let every copy still in flight land before leaving
        for (int q = issued > NB ? issued - NB : 0; q < issued; ++q) {
          const int bq = q % NB;
          if ((part_of >> bq) & 1u)
            mbar_wait(&bars[C_LANDED + bq], ((landed >> bq) & 1u) ^ 1u, 100000000ull);
          else
            mbar_wait(&bars[C_FULL + bq], (q / NB) & 1, 100000000ull);
        }
      }
      __syncwarp();
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      if (lane == 0) {
        bool ok = true;
        for (int s = 0; s < nc && ok; ++s) {
          const int b = s % NB;
          const uint32_t buf = sb + b * BUF;
          ok = wait_bar(&bars[C_FULL + b], (s / NB) & 1, cx) &&
               (s == 0 || wait_bar(&bars[C_DREADY], (s - 1) & 1, cx));   // P1 of s - 1 read
          if (!ok) break;
          tc_fence_after();
          {
            // P1 = dO^T Aqk
            const uint64_t a = sdesc_sw128(buf + B_DO, PANEL, 1024);
            const uint64_t bq = sdesc_sw128(buf + B_FAC + R_AH, PANEL, 1024);
  #pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_bf16(tm + TM_P1, a + kstep_mn(kk), bq + kstep_mn(kk), ID_P1, kk > 0);
          }
          if (!(ok = wait_bar(&bars[C_SREADY], s & 1, cx))) break;
          tc_fence_after();
          {
            // X = dS K^T
            const uint64_t bk = sdesc_sw128(buf + B_K, 0, 1024);
  #pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_bf16_ta(tm + TM_X, tm + TM_DSB + kk * 8, bk + kstep_k(kk), ID_X, kk > 0);
            mma_commit(&bars[C_XDONE]);
          }
          if (!(ok = wait_bar(&bars[C_SSCALED], s & 1, cx))) break;
          tc_fence_after();
          {
            // dS += dO^T Qg
            const uint64_t a = sdesc_sw128(buf + B_DO, PANEL, 1024);
            const uint64_t bq = sdesc_sw128(buf + B_FAC + R_QG, PANEL, 1024);
  #pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_bf16(tm + TM_DS, a + kstep_mn(kk), bq + kstep_mn(kk), ID_U1, 1u);
          }
          if (!(ok = wait_bar(&bars[C_DREADY], s & 1, cx))) break;
          tc_fence_after();
          {
            // dS += dDelta^T (-W): B = (-W)^T [128 k][64 i] read K-major
            const uint64_t bw = sdesc_sw128(buf + B_FAC + R_W, 0, 1024);
  #pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_bf16_ta(tm + TM_DS, tm + TM_DDB + kk * 8, bw + (uint64_t)(kk * 2), ID_U2, 1u);
            mma_commit(&bars[C_SUDONE]);
            mma_commit(&bars[C_FREE + b]);
          }
        }
        if (!ok) {
          // leave no product running into the TMEM that the CTA frees on its way out
          mma_commit(&bars[C_DRAIN]);
          mbar_wait(&bars[C_DRAIN], 0, 100000000ull);
        } else {
          // the buffers' last release arrivals are in before the shared memory goes away
          for (int q = nc > NB ? nc - NB : 0; q < nc; ++q)
            mbar_wait(&bars[C_FREE + q % NB], (q / NB) & 1, 100000000ull);
        }
      }
      __syncwarp();
    }
  } else if (warp < 12) {
    if constexpr (kFused) reg_alloc<168>();
    // -------------------------------------------------------------- cotangent
    const int st_t = tid - 128;                   // 0..255
    const int w = st_t >> 7;                      // column half
    const int v = ((warp & 3) << 5) + lane;       // TMEM lane = cotangent row
    const uint32_t tl = tm + ((uint32_t)((warp & 3) * 32) << 16);
    const size_t soff = (((size_t)n * H + h) * D + v) * D + 64 * w;   // [N, H, V, K]
    const size_t tstride = (size_t)H * 2 * D * D;
    uint8_t* tape = reinterpret_cast<uint8_t*>(p.tape) + ((size_t)slot0 * H + h) * 2 * D * D +
                    (size_t)w * 16384 + (size_t)v * 128;
    float xv[64];
    if (p.dsf) {
      const float4* src = reinterpret_cast<const float4*>(p.dsf + soff);
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const float4 f = src[e];
        xv[4 * e] = f.x; xv[4 * e + 1] = f.y; xv[4 * e + 2] = f.z; xv[4 * e + 3] = f.w;
      }
    } else {
#pragma unroll
      for (int e = 0; e < 64; ++e) xv[e] = 0.f;
    }
    bool ok = true;
    if (nc > 0) {
      // the last chunk's exit cotangent: the tape, the BF16 copy, then scaled by its e^{gamma_C}
      uint32_t u[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) u[e] = pack_bf16x2(xv[2 * e], xv[2 * e + 1]);
      tmem_st16(tl + TM_DSB + 32 * w, *reinterpret_cast<const uint32_t(*)[16]>(u));
      tmem_st16(tl + TM_DSB + 32 * w + 16, *reinterpret_cast<const uint32_t(*)[16]>(u + 16));
      store_tile_row(tape + (size_t)(nc - 1) * tstride, v, u);
      publish_tape(tape_flag, 1u, st_t);
      tmem_st_wait();
      tc_fence_before();
      named_bar(BAR_STATE, 256);
      if (st_t == 0) mbar_arrive(&bars[C_SREADY]);
      if ((ok = group_wait(&bars[C_FULL], 0, cx))) {
        const float g = reinterpret_cast<const float*>(sm + B_FAC + R_VEC + V_GC)[0];
#pragma unroll
        for (int e = 0; e < 64; ++e) xv[e] *= g;
        tmem_st32(tl + TM_DS + 64 * w, *reinterpret_cast<float(*)[32]>(xv));
        tmem_st32(tl + TM_DS + 64 * w + 32, *reinterpret_cast<float(*)[32]>(xv + 32));
        tmem_st_wait();
        tc_fence_before();
        named_bar(BAR_STATE, 256);
        if (st_t == 0) mbar_arrive(&bars[C_SSCALED]);
      }
    }
    for (int s = 0; s < nc && ok; ++s) {
      const uint8_t* buf = sm + (s % NB) * BUF;
      if (!(ok = group_wait(&bars[C_XDONE], s & 1, cx))) break;
      tc_fence_after();
      {
        // dDelta^T for columns [32w, 32w + 32): scale P1 + (dS K^T) diag(dec)
        float a[32], x[32];
        tmem_ld32(tl + TM_P1 + 32 * w, a);
        tmem_ld32(tl + TM_X + 32 * w, x);
        const float* dec = reinterpret_cast<const float*>(buf + B_FAC + R_VEC + V_DEC) + 32 * w;
        const float scale = p.scale;
        tmem_ld_wait();
        uint32_t d[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          d[e] = pack_bf16x2(fmaf(dec[2 * e], x[2 * e], scale * a[2 * e]),
                             fmaf(dec[2 * e + 1], x[2 * e + 1], scale * a[2 * e + 1]));
        tmem_st16(tl + TM_DDB + 16 * w, d);
      }
      tmem_st_wait();
      tc_fence_before();
      named_bar(BAR_STATE, 256);
      if (st_t == 0) mbar_arrive(&bars[C_DREADY]);
      if (!(ok = group_wait(&bars[C_SUDONE], s & 1, cx))) break;
      tc_fence_after();
      tmem_ld32(tl + TM_DS + 64 * w, *reinterpret_cast<float(*)[32]>(xv));
      tmem_ld32(tl + TM_DS + 64 * w + 32, *reinterpret_cast<float(*)[32]>(xv + 32));
      tmem_ld_wait();
      if (s + 1 == nc) break;   // xv: the cotangent at the sequence start
      // the next chunk's exit cotangent: BF16 copy for its products, the tape, then the scaling
      uint32_t u[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) u[e] = pack_bf16x2(xv[2 * e], xv[2 * e + 1]);
      tmem_st16(tl + TM_DSB + 32 * w, *reinterpret_cast<const uint32_t(*)[16]>(u));
      tmem_st16(tl + TM_DSB + 32 * w + 16, *reinterpret_cast<const uint32_t(*)[16]>(u + 16));
      tmem_st_wait();
      tc_fence_before();
      named_bar(BAR_STATE, 256);
      if (st_t == 0) mbar_arrive(&bars[C_SREADY]);
      store_tile_row(tape + (size_t)(nc - 2 - s) * tstride, v, u);
      publish_tape(tape_flag, (uint32_t)s + 2u, st_t);
      const int s1 = s + 1;
      if (!(ok = group_wait(&bars[C_FULL + s1 % NB], (s1 / NB) & 1, cx))) break;
      const float g =
          reinterpret_cast<const float*>(sm + (s1 % NB) * BUF + B_FAC + R_VEC + V_GC)[0];
#pragma unroll
      for (int e = 0; e < 64; ++e) xv[e] *= g;
      tmem_st32(tl + TM_DS + 64 * w, *reinterpret_cast<float(*)[32]>(xv));
      tmem_st32(tl + TM_DS + 64 * w + 32, *reinterpret_cast<float(*)[32]>(xv + 32));
      tmem_st_wait();
      tc_fence_before();
      named_bar(BAR_STATE, 256);
      if (st_t == 0) mbar_arrive(&bars[C_SSCALED]);
    }
    if (ok && p.ds0) {
      float4* dst = reinterpret_cast<float4*>(p.ds0 + soff);
#pragma unroll
      for (int e = 0; e < 16; ++e)
        dst[e] = make_float4(xv[4 * e], xv[4 * e + 1], xv[4 * e + 2], xv[4 * e + 3]);
    }
  } else {
    if constexpr (kFused) reg_dealloc<kCtlRegs>();   // warps 12-15 of a fused launch: idle
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tm, 512);
  if constexpr (kFused) {
    // the CTA goes on to token gradients: 128 registers per thread again (the cotangent
    // warps give theirs back first), and its barriers' memory is reused
    if (warp >= 4 && warp < 12) reg_dealloc<128>();
    else reg_alloc<128>();
    if (tid == 0)
      for (int i = 0; i < C_COUNT; ++i) mbar_inval(&bars[i]);
    __syncthreads();
  }
}

}  // namespace chaintc
}  // namespace sfg
