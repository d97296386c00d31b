// simt_chunk.cu -- FP32 CUDA-core kernels of the chunked gated delta rule.
//
// These kernels carry every matrix product in FP32 on the CUDA cores.  They
// are the path for FP32 inputs (which need FP32 accuracy end to end) and for
// head size 64, and they compute the backward for every supported dtype.
// The BF16, head-size-128 forward and segment summaries run on the split
// tensor-core kernel instead (fwd_split.cu); the two never substitute for each
// other at run time.
//
// Work decomposition (StateFlow, section 2.2, Eq. 2: Pre / ST / Out per chunk;
// section 3.4.1, Eq. 16: the state transition is tiled along the value
// dimension, so a (sequence, head) chain runs as D/BV CTAs, each owning BV
// rows of the [V,K] state -- rows of the state evolve independently given
// the chunk's factors, which every CTA recomputes).
#include <type_traits>

#include "bwd_chain_tc.cuh"
#include "common.cuh"
#include "simt_chunk.cuh"

namespace sfg {

namespace {

constexpr int NT = 256;   // threads per CTA

__device__ __forceinline__ void bar() { __syncthreads(); }
struct CtaBar {
  __device__ __forceinline__ void operator()() const { __syncthreads(); }
};

template <typename Tin>
__device__ __forceinline__ float ldg_f(const Tin* p) { return to_f(p[0]); }

}  // namespace

// ---------------------------------------------------------------------------
// Forward chain kernel.  MODE: FWD (outputs + final state), SUMMARY (the
// range's affine map: rows [0,V) of the augmented state start at zero with
// the value term on and give S_ext; rows [V,V+K) start at the identity with
// the value term off and give P -- the probing construction of the Attention
// Gym "Context Parallelism" section), REPLAY (writes each chunk's entry state
// to `ckpt`, no output; the backward's state replay).
// grid = (rows/BV, H, N or R), block = 256.
// ---------------------------------------------------------------------------
template <typename Tin, int D, int BV, int MODE>
__global__ void __launch_bounds__(NT) simt_chain_kernel(const ChainParams p) {
  constexpr int LDK = D + 1;      // [64][D] tiles
  constexpr int LDV = BV + 1;     // [64][BV] tiles
  constexpr int LD6 = 65;         // [64][64] tiles
  extern __shared__ float sm[];
  float* sK = sm;
  float* sQ = sK + 64 * LDK;
  float* sW = sQ + 64 * LDK;
  float* sV = sW + 64 * LDK;
  float* sU = sV + 64 * LDV;
  float* sS = sU + 64 * LDV;      // [BV][LDK]
  float* sA = sS + BV * LDK;
  float* sT = sA + 64 * LD6;
  float* sQK = sT + 64 * LD6;
  float* sg = sQK + 64 * LD6;
  float* sb = sg + 64;
  float* sgam = sb + 64;
  float* seg = sgam + 64;
  float* sdec = seg + 64;
  float* sscr = sU;               // solve scratch (1024 floats) aliases U/W region
  static_assert(64 * LDV + 64 * LDK >= 1024, "scratch");

  const int tid = threadIdx.x;
  const int h = blockIdx.y, item = blockIdx.z;
  const int r0 = blockIdx.x * BV;           // first (augmented) state row of this CTA
  const int H = p.H, HK = p.HK, hk = qk_head(h, H, HK);
  const Tin* q = (const Tin*)p.q;
  const Tin* k = (const Tin*)p.k;
  const Tin* v = (const Tin*)p.v;

  int64_t bos, eos;
  bool valid = true;
  if (MODE == MODE_SUMMARY) {
    const int64_t total = (int64_t)p.B * p.T;
    const int64_t s0 = p.bounds[2 * item], s1 = p.bounds[2 * item + 1];
    valid = (s0 >= 0 && s1 >= s0 && s1 <= total && (s1 == s0 || s0 / p.T == (s1 - 1) / p.T));
    bos = valid ? s0 : 0;
    eos = valid ? s1 : 0;
  } else {
    seq_span(item, p.B, p.T, p.cu, bos, eos);
  }
  const bool value_on = (MODE != MODE_SUMMARY) || (r0 < D);

  // where this chain's entry state comes from and its final state goes: the [N,H,V,K]
  // arguments, or a slot of the paged cache (padding: zeros in, nothing out, zero output)
  const size_t HDD = (size_t)H * D * D;
  const float* s0src = p.s0 ? p.s0 + (size_t)item * HDD : nullptr;
  float* fdst = p.final_state ? p.final_state + (size_t)item * HDD : nullptr;
  bool padded = false;
  if (MODE == MODE_FWD && p.pool) {
    const int ps = p.state_idx[item];
    padded = ps <= 0 || ps >= p.num_slots;
    s0src = (!padded && (!p.has_init || p.has_init[item])) ? p.pool + (size_t)ps * HDD : nullptr;
    fdst = padded ? nullptr : p.pool + (size_t)ps * HDD;
  }
  for (int idx = tid; idx < BV * D; idx += NT) {
    const int r = idx / D, c = idx % D;
    float s;
    if (MODE == MODE_SUMMARY) {
      const int ar = r0 + r;
      s = (ar >= D && c == ar - D) ? 1.f : 0.f;
    } else {
      s = s0src ? s0src[((size_t)h * D + r0 + r) * D + c] : 0.f;
    }
    sS[r * LDK + c] = s;
  }
  int64_t slot = 0;
  if (MODE == MODE_REPLAY) slot = chunk_slot_base(item, p.B, p.T, p.cu);

  for (int64_t c0 = bos; c0 < eos; c0 += CHUNK, ++slot) {
    const int L = (int)((eos - c0) < CHUNK ? (eos - c0) : CHUNK);
    bar();
    if (MODE == MODE_REPLAY) {
      float* dst = p.ckpt + ((size_t)slot * H + h) * D * D;
      for (int idx = tid; idx < BV * D; idx += NT) {
        const int r = idx / D, c = idx % D;
        dst[(size_t)(r0 + r) * D + c] = sS[r * LDK + c];
      }
    }
    for (int idx = tid; idx < 64 * D; idx += NT) {
      const int i = idx / D, c = idx % D;
      const size_t off = ((size_t)(c0 + i) * HK + hk) * D + c;
      sK[i * LDK + c] = (i < L) ? ldg_f(k + off) : 0.f;
      if (MODE == MODE_FWD) sQ[i * LDK + c] = (i < L) ? ldg_f(q + off) : 0.f;
    }
    for (int idx = tid; idx < 64 * BV; idx += NT) {
      const int i = idx / BV, c = idx % BV;
      sV[i * LDV + c] = (i < L && value_on) ? ldg_f(v + ((size_t)(c0 + i) * H + h) * D + r0 + c)
                                            : 0.f;
    }
    if (tid < 64) {
      const size_t off = (size_t)(c0 + tid) * H + h;
      sg[tid] = (tid < L) ? p.g[off] : 0.f;
      sb[tid] = (tid < L) ? p.beta[off] : 0.f;
    }
    bar();
    if (tid < 32) warp_cumsum64(sg, sgam, tid);
    bar();
    if (tid < 64) {
      seg[tid] = expf(sgam[tid]);
      sdec[tid] = expf(sgam[63] - sgam[tid]);
    }
    // A (strictly lower) and the decayed causal Q K^T (lower incl. diagonal)
    for (int idx = tid; idx < 64 * 64; idx += NT) {
      const int i = idx >> 6, j = idx & 63;
      float a = 0.f, qk = 0.f;
      if (j <= i) {
        const float dcy = expf(sgam[i] - sgam[j]);
        if (j < i) {
          float s = 0.f;
          for (int c = 0; c < D; ++c) s += sK[i * LDK + c] * sK[j * LDK + c];
          a = sb[i] * dcy * s;
        }
        if (MODE == MODE_FWD) {
          float s = 0.f;
          for (int c = 0; c < D; ++c) s += sQ[i * LDK + c] * sK[j * LDK + c];
          qk = dcy * s;
        }
      }
      sA[i * LD6 + j] = a;
      if (MODE == MODE_FWD) sQK[i * LD6 + j] = qk;
    }
    bar();
    solve_unit_lower64(sA, sT, LD6, sscr, tid, NT, CtaBar());
    // W = T diag(beta e^gamma) K ; U = T diag(beta) V
    for (int idx = tid; idx < 64 * D; idx += NT) {
      const int i = idx / D, c = idx % D;
      float s = 0.f;
      for (int j = 0; j <= i; ++j) s += sT[i * LD6 + j] * sb[j] * seg[j] * sK[j * LDK + c];
      sW[i * LDK + c] = s;
    }
    for (int idx = tid; idx < 64 * BV; idx += NT) {
      const int i = idx / BV, c = idx % BV;
      float s = 0.f;
      if (value_on)
        for (int j = 0; j <= i; ++j) s += sT[i * LD6 + j] * sb[j] * sV[j * LDV + c];
      sU[i * LDV + c] = s;
    }
    bar();
    // Delta = U - W S^T   ([64][BV], S holds this CTA's BV rows)
    for (int idx = tid; idx < 64 * BV; idx += NT) {
      const int i = idx / BV, r = idx % BV;
      float s = 0.f;
      for (int c = 0; c < D; ++c) s += sW[i * LDK + c] * sS[r * LDK + c];
      sU[i * LDV + r] -= s;
    }
    bar();
    if (MODE == MODE_FWD) {
      Tin* out = (Tin*)p.out;
      for (int idx = tid; idx < 64 * BV; idx += NT) {
        const int i = idx / BV, r = idx % BV;
        if (i >= L) continue;
        float s1 = 0.f, s2 = 0.f;
        for (int c = 0; c < D; ++c) s1 += sQ[i * LDK + c] * sS[r * LDK + c];
        for (int j = 0; j <= i; ++j) s2 += sQK[i * LD6 + j] * sU[j * LDV + r];
        out[((size_t)(c0 + i) * H + h) * D + r0 + r] =
            from_f<Tin>(padded ? 0.f : p.scale * (seg[i] * s1 + s2));
      }
      bar();
    }
    // S <- e^{gamma_C} S + Delta^T diag(dec) K
    const float gC = seg[63];
    for (int idx = tid; idx < BV * D; idx += NT) {
      const int r = idx / D, c = idx % D;
      float s = 0.f;
      for (int j = 0; j < 64; ++j) s += sU[j * LDV + r] * sdec[j] * sK[j * LDK + c];
      sS[r * LDK + c] = gC * sS[r * LDK + c] + s;
    }
  }
  bar();
  if (MODE == MODE_FWD) {
    if (fdst)
      for (int idx = tid; idx < BV * D; idx += NT) {
        const int r = idx / D, c = idx % D;
        fdst[((size_t)h * D + r0 + r) * D + c] = sS[r * LDK + c];
      }
  } else if (MODE == MODE_SUMMARY) {
    const float nan = __int_as_float(0x7fc00000);
    for (int idx = tid; idx < BV * D; idx += NT) {
      const int r = idx / D, c = idx % D, ar = r0 + r;
      const float s = valid ? sS[r * LDK + c] : nan;
      if (ar < D)
        p.E[(((size_t)item * H + h) * D + ar) * D + c] = s;
      else
        p.P[(((size_t)item * H + h) * D + ar - D) * D + c] = s;
    }
  }
}

// ---------------------------------------------------------------------------
// Reverse state-cotangent chain (StateFlow Eq. 6-7; "StateBwd" of Eq. 18).
// Per chunk, walking backwards, with dSn the cotangent of the chunk's exit
// state:  dDelta = scale Aqk^T dO + diag(dec) K dSn^T
//         dS_entry = e^{gamma_C} dSn + scale dO^T diag(e^gamma) Q - dDelta^T W
// Rows of dS are independent given the chunk factors, so the chain is tiled
// along V like the forward.  Each chunk's dSn is written to `tape`; the
// cotangent at the sequence start is d_initial_state.
// grid = (D/BV, H, N), block = 256.
// ---------------------------------------------------------------------------
template <typename Tin, int D, int BV>
__global__ void __launch_bounds__(NT) simt_bwd_chain_kernel(const ChainParams p) {
  constexpr int LDK = D + 1, LDV = BV + 1, LD6 = 65;
  extern __shared__ float sm[];
  float* sK = sm;
  float* sQ = sK + 64 * LDK;
  float* sW = sQ + 64 * LDK;
  float* sdO = sW + 64 * LDK;     // [64][BV]
  float* sdD = sdO + 64 * LDV;    // [64][BV] dDelta
  float* sS = sdD + 64 * LDV;     // [BV][LDK] running cotangent rows
  float* sA = sS + BV * LDK;
  float* sT = sA + 64 * LD6;
  float* sQK = sT + 64 * LD6;
  float* sg = sQK + 64 * LD6;
  float* sb = sg + 64;
  float* sgam = sb + 64;
  float* seg = sgam + 64;
  float* sdec = seg + 64;
  float* sscr = sdO;
  static_assert(2 * 64 * LDV + BV * LDK >= 1024, "scratch");

  const int tid = threadIdx.x;
  const int h = blockIdx.y, n = blockIdx.z, r0 = blockIdx.x * BV;
  const int H = p.H, HK = p.HK, hk = qk_head(h, H, HK);
  const Tin* q = (const Tin*)p.q;
  const Tin* k = (const Tin*)p.k;
  const Tin* dO = (const Tin*)p.dout;
  int64_t bos, eos;
  seq_span(n, p.B, p.T, p.cu, bos, eos);
  const int64_t nc = n_chunks(eos - bos);
  const int64_t slot0 = chunk_slot_base(n, p.B, p.T, p.cu);

  for (int idx = tid; idx < BV * D; idx += NT) {
    const int r = idx / D, c = idx % D;
    sS[r * LDK + c] =
        p.dsf ? p.dsf[(((size_t)n * H + h) * D + r0 + r) * D + c] : 0.f;
  }
  for (int64_t ci = nc - 1; ci >= 0; --ci) {
    const int64_t c0 = bos + ci * CHUNK;
    const int L = (int)((eos - c0) < CHUNK ? (eos - c0) : CHUNK);
    bar();
    {
      float* dst = p.tape + ((size_t)(slot0 + ci) * H + h) * D * D;
      for (int idx = tid; idx < BV * D; idx += NT) {
        const int r = idx / D, c = idx % D;
        dst[(size_t)(r0 + r) * D + c] = sS[r * LDK + c];
      }
    }
    for (int idx = tid; idx < 64 * D; idx += NT) {
      const int i = idx / D, c = idx % D;
      const size_t off = ((size_t)(c0 + i) * HK + hk) * D + c;
      sK[i * LDK + c] = (i < L) ? ldg_f(k + off) : 0.f;
      sQ[i * LDK + c] = (i < L) ? ldg_f(q + off) : 0.f;
    }
    for (int idx = tid; idx < 64 * BV; idx += NT) {
      const int i = idx / BV, c = idx % BV;
      sdO[i * LDV + c] = (i < L) ? ldg_f(dO + ((size_t)(c0 + i) * H + h) * D + r0 + c) : 0.f;
    }
    if (tid < 64) {
      const size_t off = (size_t)(c0 + tid) * H + h;
      sg[tid] = (tid < L) ? p.g[off] : 0.f;
      sb[tid] = (tid < L) ? p.beta[off] : 0.f;
    }
    bar();
    if (tid < 32) warp_cumsum64(sg, sgam, tid);
    bar();
    if (tid < 64) {
      seg[tid] = expf(sgam[tid]);
      sdec[tid] = expf(sgam[63] - sgam[tid]);
    }
    for (int idx = tid; idx < 64 * 64; idx += NT) {
      const int i = idx >> 6, j = idx & 63;
      float a = 0.f, qk = 0.f;
      if (j <= i) {
        const float dcy = expf(sgam[i] - sgam[j]);
        float s1 = 0.f, s2 = 0.f;
        for (int c = 0; c < D; ++c) {
          s1 += sK[i * LDK + c] * sK[j * LDK + c];
          s2 += sQ[i * LDK + c] * sK[j * LDK + c];
        }
        if (j < i) a = sb[i] * dcy * s1;
        qk = dcy * s2;
      }
      sA[i * LD6 + j] = a;
      sQK[i * LD6 + j] = qk;
    }
    bar();
    // the solve's scratch aliases sdO: stash dO in sdD meanwhile
    for (int idx = tid; idx < 64 * BV; idx += NT) sdD[idx] = sdO[(idx / BV) * LDV + idx % BV];
    bar();
    solve_unit_lower64(sA, sT, LD6, sscr, tid, NT, CtaBar());
    for (int idx = tid; idx < 64 * BV; idx += NT) sdO[(idx / BV) * LDV + idx % BV] = sdD[idx];
    for (int idx = tid; idx < 64 * D; idx += NT) {
      const int i = idx / D, c = idx % D;
      float s = 0.f;
      for (int j = 0; j <= i; ++j) s += sT[i * LD6 + j] * sb[j] * seg[j] * sK[j * LDK + c];
      sW[i * LDK + c] = s;
    }
    bar();
    // dDelta = scale Aqk^T dO + diag(dec) K dSn^T
    for (int idx = tid; idx < 64 * BV; idx += NT) {
      const int j = idx / BV, r = idx % BV;
      float s1 = 0.f, s2 = 0.f;
      for (int i = j; i < 64; ++i) s1 += sQK[i * LD6 + j] * sdO[i * LDV + r];
      for (int c = 0; c < D; ++c) s2 += sK[j * LDK + c] * sS[r * LDK + c];
      sdD[j * LDV + r] = p.scale * s1 + sdec[j] * s2;
    }
    bar();
    // dS_entry = e^{gamma_C} dSn + scale dO^T diag(e^gamma) Q - dDelta^T W
    const float gC = seg[63];
    for (int idx = tid; idx < BV * D; idx += NT) {
      const int r = idx / D, c = idx % D;
      float s1 = 0.f, s2 = 0.f;
      for (int i = 0; i < 64; ++i) {
        s1 += sdO[i * LDV + r] * seg[i] * sQ[i * LDK + c];
        s2 += sdD[i * LDV + r] * sW[i * LDK + c];
      }
      sS[r * LDK + c] = gC * sS[r * LDK + c] + p.scale * s1 - s2;
    }
  }
  bar();
  if (p.ds0)
    for (int idx = tid; idx < BV * D; idx += NT) {
      const int r = idx / D, c = idx % D;
      p.ds0[(((size_t)n * H + h) * D + r0 + r) * D + c] = sS[r * LDK + c];
    }
}

// ---------------------------------------------------------------------------
// Token gradients of one chunk ("OutputGrad" + "PrepGrad" of StateFlow
// Eq. 18), fully parallel over chunks: given the chunk's entry state S (from
// the replay) and its exit cotangent dSn (from the chain), recompute the
// chunk factors and back-propagate through Out, ST and Pre.  The steps follow
// the chunk algebra in common.cuh, differentiated term by term.
// grid = (slots, H), block = 256.  Q/K/V/dO are staged in smem in the input
// dtype; the per-thread dq/dk accumulators live in registers.
// ---------------------------------------------------------------------------
// One chunk (backward slot `slot`); false when the slot holds no chunk.
template <typename Tin, int D>
__device__ __forceinline__ bool simt_grad_chunk(const ChainParams& p, int64_t slot) {
  constexpr int LDI = D + 8;      // input tiles (Tin)
  constexpr int LDF = D + 1;      // fp32 [64][D] tiles
  constexpr int LD6 = 65;
  constexpr int PER = 64 * D / NT;
  extern __shared__ float sm[];
  float* sT = sm;
  float* sM = sT + 64 * LD6;      // Ak (Gamma o K K^T, strict) -> dA
  float* sP = sM + 64 * LD6;      // Aqk -> G -> dT
  float* B1 = sP + 64 * LD6;      // W -> dW
  float* B2 = B1 + 64 * LDF;      // U -> Delta -> T^T dDelta
  float* B3 = B2 + 64 * LDF;      // dDelta
  float* sg = B3 + 64 * LDF;
  float* sb = sg + 64;
  float* sgam = sb + 64;
  float* seg = sgam + 64;
  float* sdec = seg + 64;
  float* sdgam = sdec + 64;
  float* sred = sdgam + 64;       // 64 scratch
  Tin* sQ = (Tin*)(sred + 64);
  Tin* sK = sQ + 64 * LDI;
  Tin* sV = sK + 64 * LDI;
  Tin* sdO = sV + 64 * LDI;

  const int tid = threadIdx.x, h = blockIdx.y, H = p.H, HK = p.HK, hk = qk_head(h, H, HK);
  // locate (sequence, chunk) of this slot
  int n = -1;
  int64_t bos = 0, eos = 0, ci = 0;
  if (!locate_chunk(slot, p.B, p.T, p.cu, p.N, n, bos, eos, ci)) return false;
  const int64_t c0 = bos + ci * CHUNK;
  const int L = (int)((eos - c0) < CHUNK ? (eos - c0) : CHUNK);
  const float* S = p.ckpt + ((size_t)slot * H + h) * D * D;
  const float* dSn = p.tape + ((size_t)slot * H + h) * D * D;
  const Tin* q = (const Tin*)p.q;
  const Tin* k = (const Tin*)p.k;
  const Tin* v = (const Tin*)p.v;
  const Tin* dO = (const Tin*)p.dout;
  const float scale = p.scale;

  for (int idx = tid; idx < 64 * D; idx += NT) {
    const int i = idx / D, c = idx % D;
    const size_t off = ((size_t)(c0 + i) * H + h) * D + c;
    const size_t oqk = ((size_t)(c0 + i) * HK + hk) * D + c;
    const Tin z = from_f<Tin>(0.f);
    sQ[i * LDI + c] = (i < L) ? q[oqk] : z;
    sK[i * LDI + c] = (i < L) ? k[oqk] : z;
    sV[i * LDI + c] = (i < L) ? v[off] : z;
    sdO[i * LDI + c] = (i < L) ? dO[off] : z;
  }
  if (tid < 64) {
    const size_t off = (size_t)(c0 + tid) * H + h;
    sg[tid] = (tid < L) ? p.g[off] : 0.f;
    sb[tid] = (tid < L) ? p.beta[off] : 0.f;
    sdgam[tid] = 0.f;
  }
  __syncthreads();
  if (tid < 32) warp_cumsum64(sg, sgam, tid);
  __syncthreads();
  if (tid < 64) {
    seg[tid] = expf(sgam[tid]);
    sdec[tid] = expf(sgam[63] - sgam[tid]);
  }
#define QF(i, c) to_f(sQ[(i) * LDI + (c)])
#define KF(i, c) to_f(sK[(i) * LDI + (c)])
#define VF(i, c) to_f(sV[(i) * LDI + (c)])
#define DOF(i, c) to_f(sdO[(i) * LDI + (c)])
  // Ak = Gamma o K K^T (strict lower), Aqk = Gamma o Q K^T (lower incl. diag)
  for (int idx = tid; idx < 64 * 64; idx += NT) {
    const int i = idx >> 6, j = idx & 63;
    float ak = 0.f, aq = 0.f;
    if (j <= i) {
      const float dcy = expf(sgam[i] - sgam[j]);
      float s1 = 0.f, s2 = 0.f;
      for (int c = 0; c < D; ++c) {
        s1 += KF(i, c) * KF(j, c);
        s2 += QF(i, c) * KF(j, c);
      }
      if (j < i) ak = dcy * s1;
      aq = dcy * s2;
    }
    sM[i * LD6 + j] = ak;
    sP[i * LD6 + j] = aq;
  }
  __syncthreads();
  // A = diag(beta) Ak into B3 (as a [64][65] tile), solve -> T (scratch B2)
  for (int idx = tid; idx < 64 * 64; idx += NT) {
    const int i = idx >> 6, j = idx & 63;
    B3[i * LD6 + j] = sb[i] * sM[i * LD6 + j];
  }
  __syncthreads();
  solve_unit_lower64(B3, sT, LD6, B2, tid, NT, CtaBar());
  // W, U
  for (int idx = tid; idx < 64 * D; idx += NT) {
    const int i = idx / D, c = idx % D;
    float sw = 0.f, su = 0.f;
    for (int j = 0; j <= i; ++j) {
      const float t = sT[i * LD6 + j] * sb[j];
      sw += t * seg[j] * KF(j, c);
      su += t * VF(j, c);
    }
    B1[i * LDF + c] = sw;
    B2[i * LDF + c] = su;
  }
  __syncthreads();
  // Delta = U - W S^T (B2);  dDelta = scale Aqk^T dO + diag(dec) K dSn^T (B3)
  for (int idx = tid; idx < 64 * D; idx += NT) {
    const int i = idx / D, r = idx % D;
    float s = 0.f, s1 = 0.f, s2 = 0.f;
    for (int c = 0; c < D; ++c) {
      s += B1[i * LDF + c] * S[(size_t)r * D + c];
      s2 += KF(i, c) * dSn[(size_t)r * D + c];
    }
    for (int m = i; m < 64; ++m) s1 += sP[m * LD6 + i] * DOF(m, r);
    B2[i * LDF + r] -= s;
    B3[i * LDF + r] = scale * s1 + sdec[i] * s2;
  }
  __syncthreads();
  float dq[PER], dk[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) { dq[e] = 0.f; dk[e] = 0.f; }
  // dAqk = scale dO Delta^T; rho = dAqk o Aqk -> dgamma; G = dAqk o Gamma (in sP)
  for (int idx = tid; idx < 64 * 64; idx += NT) {
    const int i = idx >> 6, j = idx & 63;
    float gval = 0.f;
    if (j <= i) {
      float s = 0.f;
      for (int r = 0; r < D; ++r) s += DOF(i, r) * B2[j * LDF + r];
      const float dA = scale * s;
      const float rho = dA * sP[i * LD6 + j];
      atomicAdd(&sdgam[i], rho);
      atomicAdd(&sdgam[j], -rho);
      gval = dA * expf(sgam[i] - sgam[j]);
    }
    sP[i * LD6 + j] = gval;    // each element read and written by its owner only
  }
  __syncthreads();
  // dq += scale e^gamma (dO S) + G K ; dk += G^T Q ; dgamma += q . dQfirst
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    const int idx = tid + e * NT, i = idx / D, c = idx % D;
    float s = 0.f, sg2 = 0.f, sk = 0.f;
    for (int r = 0; r < D; ++r) s += DOF(i, r) * S[(size_t)r * D + c];
    const float first = scale * seg[i] * s;
    for (int j = 0; j <= i; ++j) sg2 += sP[i * LD6 + j] * KF(j, c);
    for (int m = i; m < 64; ++m) sk += sP[m * LD6 + i] * QF(m, c);
    dq[e] += first + sg2;
    dk[e] += sk;
    atomicAdd(&sdgam[i], QF(i, c) * first);
  }
  // exit state: Z = Delta dSn; dk += dec o Z; ddec = rowsum(K o Z)
  if (tid < 64) sred[tid] = 0.f;
  __syncthreads();
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    const int idx = tid + e * NT, j = idx / D, c = idx % D;
    float z = 0.f;
    for (int r = 0; r < D; ++r) z += B2[j * LDF + r] * dSn[(size_t)r * D + c];
    dk[e] += sdec[j] * z;
    atomicAdd(&sred[j], KF(j, c) * z);
  }
  // <dSn, S> for the e^{gamma_C} S term
  float part = 0.f;
  for (int idx = tid; idx < D * D; idx += NT) part += dSn[idx] * S[idx];
  __syncthreads();
  atomicAdd(&sdgam[63], seg[63] * part);
  if (tid < 64) {
    const float t = sdec[tid] * sred[tid];
    atomicAdd(&sdgam[tid], -t);
    atomicAdd(&sdgam[63], t);
  }
  // dW = -dDelta S (B1);  T^T dDelta (B2, Delta no longer needed)
  __syncthreads();
  for (int idx = tid; idx < 64 * D; idx += NT) {
    const int i = idx / D, c = idx % D;
    float s = 0.f, t = 0.f;
    for (int r = 0; r < D; ++r) s += B3[i * LDF + r] * S[(size_t)r * D + c];
    for (int m = i; m < 64; ++m) t += sT[m * LD6 + i] * B3[m * LDF + c];
    B1[i * LDF + c] = -s;
    B2[i * LDF + c] = t;
  }
  if (tid < 64) sred[tid] = 0.f;
  __syncthreads();
  // dv = beta T^T dDelta ; dbeta += rowsum(V o T^T dDelta)
  {
    Tin* dv = (Tin*)p.dv;
    for (int idx = tid; idx < 64 * D; idx += NT) {
      const int i = idx / D, c = idx % D;
      const float t = B2[i * LDF + c];
      if (i < L) dv[((size_t)(c0 + i) * H + h) * D + c] = from_f<Tin>(sb[i] * t);
      atomicAdd(&sred[i], VF(i, c) * t);
    }
  }
  // dT = dDelta (diag(beta) V)^T + dW (diag(beta e^gamma) K)^T  (into sP)
  for (int idx = tid; idx < 64 * 64; idx += NT) {
    const int i = idx >> 6, j = idx & 63;
    float s1 = 0.f, s2 = 0.f;
    for (int c = 0; c < D; ++c) {
      s1 += B3[i * LDF + c] * VF(j, c);
      s2 += B1[i * LDF + c] * KF(j, c);
    }
    sP[i * LD6 + j] = sb[j] * s1 + sb[j] * seg[j] * s2;
  }
  __syncthreads();
  // T^T dW (B3, dDelta done) ; dk += beta e^gamma T^T dW ; kt = rowsum(K o T^T dW)
  for (int idx = tid; idx < 64 * D; idx += NT) {
    const int i = idx / D, c = idx % D;
    float t = 0.f;
    for (int m = i; m < 64; ++m) t += sT[m * LD6 + i] * B1[m * LDF + c];
    B3[i * LDF + c] = t;
  }
  __syncthreads();
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    const int idx = tid + e * NT, i = idx / D, c = idx % D;
    dk[e] += sb[i] * seg[i] * B3[i * LDF + c];
  }
  // kt_i = sum_c K_ic (T^T dW)_ic -> dbeta += e^gamma kt, dgamma += beta e^gamma kt
  // (reuse B1 row sums via a strided reduction in registers + smem atomics)
  __syncthreads();
  if (tid < 64) {
    float kt = 0.f;
    for (int c = 0; c < D; ++c) kt += KF(tid, c) * B3[tid * LDF + c];
    sred[tid] += seg[tid] * kt;                  // dbeta contributions so far in sred
    sdgam[tid] += sb[tid] * seg[tid] * kt;
  }
  // dA = -(T^T dT T^T) strictly lower: X = dT T^T (B1 as [64][65]), dA = -T^T X (sM)
  __syncthreads();
  for (int idx = tid; idx < 64 * 64; idx += NT) {
    const int i = idx >> 6, j = idx & 63;
    float s = 0.f;
    for (int m = 0; m <= j; ++m) s += sP[i * LD6 + m] * sT[j * LD6 + m];
    B1[i * LD6 + j] = s;
  }
  __syncthreads();
  for (int idx = tid; idx < 64 * 64; idx += NT) {
    const int i = idx >> 6, j = idx & 63;
    float dA = 0.f;
    if (j < i) {
      float s = 0.f;
      for (int m = i; m < 64; ++m) s += sT[m * LD6 + i] * B1[m * LD6 + j];
      dA = -s;
    }
    B2[i * LD6 + j] = dA;      // keep sM (Ak) intact
  }
  __syncthreads();
  // from A_ij = beta_i Ak_ij: dbeta_i += sum_j dA_ij Ak_ij; dgamma_i/j +- dA beta Ak;
  // dKK_ij = dA_ij beta_i Gamma_ij (into sP)
  for (int idx = tid; idx < 64 * 64; idx += NT) {
    const int i = idx >> 6, j = idx & 63;
    float dkk = 0.f;
    if (j < i) {
      const float dA = B2[i * LD6 + j], ak = sM[i * LD6 + j];
      atomicAdd(&sred[i], dA * ak);
      const float rho = dA * sb[i] * ak;
      atomicAdd(&sdgam[i], rho);
      atomicAdd(&sdgam[j], -rho);
      dkk = dA * sb[i] * expf(sgam[i] - sgam[j]);
    }
    sP[i * LD6 + j] = dkk;
  }
  __syncthreads();
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    const int idx = tid + e * NT, i = idx / D, c = idx % D;
    float s = 0.f;
    for (int j = 0; j < i; ++j) s += sP[i * LD6 + j] * KF(j, c);
    for (int m = i + 1; m < 64; ++m) s += sP[m * LD6 + i] * KF(m, c);
    dk[e] += s;
  }
  // write dq, dk
  {
    Tin* dqo = (Tin*)p.dq;
    Tin* dko = (Tin*)p.dk;
#pragma unroll
    for (int e = 0; e < PER; ++e) {
      const int idx = tid + e * NT, i = idx / D, c = idx % D;
      if (i < L) {
        const size_t off = ((size_t)(c0 + i) * H + h) * D + c;
        if (p.dqk_f32) {         // grouped heads: per value head, summed afterwards
          reinterpret_cast<float*>(p.dq)[off] = dq[e];
          reinterpret_cast<float*>(p.dk)[off] = dk[e];
        } else {
          dqo[off] = from_f<Tin>(dq[e]);
          dko[off] = from_f<Tin>(dk[e]);
        }
      }
    }
  }
  __syncthreads();
  // dgate = reverse cumsum of dgamma; dbeta
  if (tid < 32) {
    // reverse inclusive scan of 64 values by one warp
    const int lane = tid;
    const float a = sdgam[63 - 2 * lane], b = sdgam[62 - 2 * lane];
    float s = a + b;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float t = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += t;
    }
    const float excl = s - (a + b);
    sgam[63 - 2 * lane] = excl + a;
    sgam[62 - 2 * lane] = excl + a + b;
  }
  __syncthreads();
  if (tid < L) {
    const size_t off = (size_t)(c0 + tid) * H + h;
    p.dg[off] = sgam[tid];
    p.dbeta[off] = sred[tid];
  }
#undef QF
#undef KF
#undef VF
#undef DOF
  return true;
}

// Slots blockIdx.x, blockIdx.x + gridDim.x, ... until the first empty one.
template <typename Tin, int D>
__global__ void __launch_bounds__(NT) simt_bwd_grad_kernel(const ChainParams p, int64_t slots) {
  for (int64_t slot = blockIdx.x; slot < slots; slot += gridDim.x) {
    if (!simt_grad_chunk<Tin, D>(p, slot)) break;
    __syncthreads();   // shared memory is rewritten by the next chunk
  }
}

// ---------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------
template <typename Tin, int D, int BV, int MODE>
static size_t chain_smem() {
  return sizeof(float) * (3 * 64 * (D + 1) + 2 * 64 * (BV + 1) + BV * (D + 1) + 3 * 64 * 65 +
                          5 * 64);
}

template <typename Tin, int D, int BV, int MODE>
static cudaError_t launch_chain_t(const ChainParams& p, int items, cudaStream_t st) {
  const size_t smem = chain_smem<Tin, D, BV, MODE>();
  auto kern = simt_chain_kernel<Tin, D, BV, MODE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int rows = (MODE == MODE_SUMMARY) ? 2 * D : D;
  dim3 grid(rows / BV, p.H, items);
  kern<<<grid, NT, smem, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_simt_chain(const ChainParams& p, int mode, bool bf16, int D, int items,
                              cudaStream_t st) {
#define SF_CHAIN(T_, D_, M_)                                                   \
  if (D == D_ && mode == M_) return launch_chain_t<T_, D_, 32, M_>(p, items, st);
  if (bf16) {
    // (BF16 with K = 128 runs on the tensor-core split kernel only)
    SF_CHAIN(__nv_bfloat16, 64, MODE_FWD)
    SF_CHAIN(__nv_bfloat16, 64, MODE_SUMMARY)
    SF_CHAIN(__nv_bfloat16, 64, MODE_REPLAY)
  } else {
    SF_CHAIN(float, 64, MODE_FWD)
    SF_CHAIN(float, 128, MODE_FWD)
    SF_CHAIN(float, 64, MODE_SUMMARY)
    SF_CHAIN(float, 128, MODE_SUMMARY)
    SF_CHAIN(float, 64, MODE_REPLAY)
    SF_CHAIN(float, 128, MODE_REPLAY)
  }
#undef SF_CHAIN
  return cudaErrorInvalidValue;
}

template <typename Tin, int D>
static cudaError_t launch_bwd_t(const ChainParams& p, int64_t slots, cudaStream_t st,
                                bool chain_only) {
  cudaError_t e;
  if constexpr (std::is_same<Tin, __nv_bfloat16>::value) {
    // K = V = 128, dense, records kept by the replay: the reverse chain and the token
    // gradients in one tcgen05 launch
    if (D == 128 && !chain_only && p.fac_ready && tc_bwd_fusable(p)) {
      if ((e = launch_tc_bwd_qg(p, p.fac, slots, st)) != cudaSuccess) return e;
      return launch_tc_bwd_fused(p, p.fac, st);
    }
    // BF16: reverse chain and token gradients on the tensor cores
    if ((e = launch_mma_bwd_chain(p, p.fac, D, slots, st)) != cudaSuccess) return e;
    if (chain_only) return cudaSuccess;
    // K = V = 128 (after the split kernel's replay): token gradients on tcgen05
    if (D == 128) return launch_tc_bwd_grad(p, slots, st);
    return launch_mma_bwd_grad(p, true, D, slots, st);
  } else {
  // FP32 inputs keep FP32 products on the CUDA cores (1e-4 parity)
  constexpr int BV = 32;
  const size_t smem = sizeof(float) * (3 * 64 * (D + 1) + 2 * 64 * (BV + 1) + BV * (D + 1) +
                                       3 * 64 * 65 + 5 * 64);
  auto kern = simt_bwd_chain_kernel<Tin, D, BV>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<dim3(D / BV, p.H, p.N), NT, smem, st>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess || chain_only) return e;
  const size_t smem2 = sizeof(float) * (3 * 64 * 65 + 3 * 64 * (D + 1) + 7 * 64) +
                       sizeof(Tin) * 4 * 64 * (D + 8);
  auto kern2 = simt_bwd_grad_kernel<Tin, D>;
  e = cudaFuncSetAttribute(kern2, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem2);
  if (e != cudaSuccess) return e;
  if (slots > 0) kern2<<<dim3((unsigned)slot_grid(p, slots), p.H), NT, smem2, st>>>(p, slots);
  return cudaGetLastError();
  }
}

cudaError_t launch_simt_bwd(const ChainParams& p, bool bf16, int D, int64_t slots,
                            cudaStream_t st, bool chain_only) {
  if (bf16 && D == 64) return launch_bwd_t<__nv_bfloat16, 64>(p, slots, st, chain_only);
  if (bf16 && D == 128) return launch_bwd_t<__nv_bfloat16, 128>(p, slots, st, chain_only);
  if (!bf16 && D == 64) return launch_bwd_t<float, 64>(p, slots, st, chain_only);
  return cudaErrorInvalidValue;
}

}  // namespace sfg
