// bwd_grad_mma.cu -- token gradients of one chunk of the chunked gated delta rule on the
// warp-level tensor cores, FP32 accumulation: for BF16 inputs every product but the four of
// the dA path (T^T dDelta, T^T dW, dT T^T, T^T X1) takes BF16 operand pairs (mma.sync
// m16n8k16; the forward's tensor-core operand precision: W and U from BF16 T'' and T' as
// there); those four stay TF32 (m16n8k8), and FP32 inputs use TF32 throughout.
//
// StateFlow section 3.4.2, Eq. 18 ("OutputGrad" and "PrepGrad"): given the chunk's entry
// state S (state replay) and the cotangent dSn of its exit state (reverse state chain),
// the chunk's factors are recomputed and the gradient is pushed back through Out, ST and
// Pre -- the chunk algebra of common.cuh differentiated term by term:
//
//   Ak = Gamma o K K^T (strict), Aqk = Gamma o Q K^T (incl. diagonal), A = diag(beta) Ak
//   T = (I + A)^-1, W = T diag(beta e^gamma) K, U = T diag(beta) V, Delta = U - W S^T
//   dDelta = scale Aqk^T dO + diag(dec) K dSn^T
//   dAqk = scale dO Delta^T -> G = dAqk o Gamma,   dq = scale diag(e^gamma) dO S + G K
//   dk  = G^T Q + diag(dec) (Delta dSn) + diag(beta e^gamma) T^T dW + dKK K + dKK^T K
//   dW  = -dDelta S,   dv = diag(beta) T^T dDelta,   dT = dDelta (beta V)^T + dW (beta e^gamma K)^T
//   dA  = -(T^T dT T^T) strictly lower,  dKK = dA o (beta Gamma)
//   dgate = reverse cumulative sum of dgamma (collected from every decay factor), dbeta.
//
// Every product is a set of 16x8 output tiles per warp (16 warps); a warp owns the same tiles of
// every 64 x D product, so dq and dk accumulate in its registers across products.  The
// shared-memory tiles and the order of the steps are those of simt_bwd_grad_kernel.
#include <type_traits>

#include "common.cuh"
#include "mma_tiles.cuh"
#include "simt_chunk.cuh"
#include "solve_tc.cuh"

namespace sfg {
namespace {

using namespace mt;
constexpr int NWG = 16;          // warps
constexpr int NTG = 32 * NWG;
// Leading dimensions (floats) of the FP32 tiles.  4 mod 32 where TF32 fragments are loaded
// (8 rows x 4 columns per instruction fall on distinct banks); 8 mod 32 for the [64][D]
// tiles of BF16 inputs, read as BF16 pairs (8-byte loads, 8 rows x 8 columns per half-warp).
constexpr int G_LD6 = 68;
template <typename Tin, int D>
__host__ __device__ constexpr int g_ldf() {
  return D + (std::is_same<Tin, __nv_bfloat16>::value ? 8 : 4);
}

struct CtaBarG {
  __device__ __forceinline__ void operator()() const { __syncthreads(); }
};

}  // namespace

// One chunk (backward slot `slot`); false when the slot holds no chunk.
template <typename Tin, int D>
__device__ __forceinline__ bool grad_chunk(const ChainParams& p, int64_t slot) {
  constexpr int LDI = D + 8;      // input tiles (Tin)
  constexpr int LDF = g_ldf<Tin, D>();  // fp32 [64][D] tiles
  // products with k = D on BF16 operand pairs for BF16 inputs (TF32 for FP32 inputs)
  constexpr bool B16 = std::is_same<Tin, __nv_bfloat16>::value;
  constexpr int LD6 = G_LD6;
  constexpr int NTD = D / 8;      // 8-column tiles of a 64 x D output
  constexpr int TD = 4 * NTD / NWG;  // tiles per warp of a 64 x D output
  constexpr int T6 = 32 / NWG;       // tiles per warp of a 64 x 64 output
  extern __shared__ float sm[];
  float* sT = sm;
  float* sM = sT + 64 * LD6;      // Ak (Gamma o K K^T, strict)
  float* sP = sM + 64 * LD6;      // Aqk -> G -> dT -> dKK
  float* B1 = sP + 64 * LD6;      // W -> dW -> X1
  float* B2 = B1 + 64 * LDF;      // U -> Delta -> T^T dDelta -> dA
  float* B3 = B2 + 64 * LDF;      // solve input, then dDelta
  float* sg = B3 + 64 * LDF;
  float* sb = sg + 64;
  float* sgam = sb + 64;
  float* seg = sgam + 64;
  float* sdec = seg + 64;
  float* sdgam = sdec + 64;
  float* sred = sdgam + 64;       // dbeta accumulator
  float* sz = sred + 64;          // per-row sums of K o (Delta dSn)
  float* sbeg = sz + 64;          // beta e^gamma
  float* ssc = sbeg + 64;         // scale e^gamma
  Tin* sQ = reinterpret_cast<Tin*>(ssc + 64);
  Tin* sK = sQ + 64 * LDI;
  Tin* sV = sK + 64 * LDI;
  Tin* sdO = sV + 64 * LDI;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, h = blockIdx.y, H = p.H;
  const int HK = p.HK, hk = qk_head(h, H, HK);
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

  {
    // 16-byte loads, all of a thread's issued together
    constexpr int PV = 16 / sizeof(Tin);          // elements per 16 bytes
    constexpr int NV = 64 * D / PV / NTG;         // 16-byte pieces per thread per tile
    uint4 vq[NV], vk[NV], vv[NV], vo[NV];
#pragma unroll
    for (int e = 0; e < NV; ++e) {
      const int idx = (tid + NTG * e) * PV, i = idx / D, c = idx % D;
      const size_t off = ((size_t)(c0 + i) * H + h) * D + c;
      const size_t oqk = ((size_t)(c0 + i) * HK + hk) * D + c;
      const uint4 z = make_uint4(0, 0, 0, 0);
      vq[e] = (i < L) ? *reinterpret_cast<const uint4*>(q + oqk) : z;
      vk[e] = (i < L) ? *reinterpret_cast<const uint4*>(k + oqk) : z;
      vv[e] = (i < L) ? *reinterpret_cast<const uint4*>(v + off) : z;
      vo[e] = (i < L) ? *reinterpret_cast<const uint4*>(dO + off) : z;
    }
#pragma unroll
    for (int e = 0; e < NV; ++e) {
      const int idx = (tid + NTG * e) * PV, i = idx / D, c = idx % D;
      *reinterpret_cast<uint4*>(sQ + i * LDI + c) = vq[e];
      *reinterpret_cast<uint4*>(sK + i * LDI + c) = vk[e];
      *reinterpret_cast<uint4*>(sV + i * LDI + c) = vv[e];
      *reinterpret_cast<uint4*>(sdO + i * LDI + c) = vo[e];
    }
  }
  if (tid < 64) {
    const size_t off = (size_t)(c0 + tid) * H + h;
    sg[tid] = (tid < L) ? p.g[off] : 0.f;
    sb[tid] = (tid < L) ? p.beta[off] : 0.f;
    sdgam[tid] = 0.f;
    sred[tid] = 0.f;
    sz[tid] = 0.f;
  }
  __syncthreads();
  if (tid < 32) warp_cumsum64(sg, sgam, tid);
  __syncthreads();
  if (tid < 64) {
    const float eg = expf(sgam[tid]);
    seg[tid] = eg;
    sdec[tid] = expf(sgam[63] - sgam[tid]);
    sbeg[tid] = sb[tid] * eg;
    ssc[tid] = scale * eg;
  }
  __syncthreads();
  const auto Qv = view(sQ, LDI, 1), Kv = view(sK, LDI, 1), Vv = view(sV, LDI, 1),
             dOv = view(sdO, LDI, 1);
  const auto Sv = rm(S, D);
  const auto SvT = cm(S, D);

  // Ak = Gamma o K K^T (strict lower), Aqk = Gamma o Q K^T (lower incl. diagonal)
  {
    float a1[T6][4], a2[T6][4];
    zero(a1);
    zero(a2);
    gemmx<B16, T6, 8, NWG, true>(a1, rm(sK, LDI), cm(sK, LDI), D, warp, lane);
    gemmx<B16, T6, 8, NWG, true>(a2, rm(sQ, LDI), cm(sK, LDI), D, warp, lane);
    each<T6, 8, NWG, true>(a1, warp, lane, [&](int i, int j, float& x) {
      sM[i * LD6 + j] = (j < i) ? expf(sgam[i] - sgam[j]) * x : 0.f;
    });
    each<T6, 8, NWG, true>(a2, warp, lane, [&](int i, int j, float& x) {
      sP[i * LD6 + j] = (j <= i) ? expf(sgam[i] - sgam[j]) * x : 0.f;
    });
  }
  __syncthreads();
  // A = diag(beta) Ak into B3 (as a [64][65] tile), T = (I + A)^-1 into sT (scratch B2)
  for (int idx = tid; idx < 64 * 64; idx += NTG) {
    const int i = idx >> 6, j = idx & 63;
    B3[i * LD6 + j] = sb[i] * sM[i * LD6 + j];
  }
  __syncthreads();
  // BF16 inputs: the off-diagonal merges on TF32 mma (the forward's solve); FP32 inputs
  // keep the FP32 substitution
  static_assert(LD6 == SOLVE_LD, "solve layout");
  if constexpr (std::is_same<Tin, __nv_bfloat16>::value)
    solve64_tc(B3, sT, B2, tid, NTG, CtaBarG());
  else
    solve_unit_lower64(B3, sT, LD6, B2, tid, NTG, CtaBarG());
  const auto Tv = view(sT, LD6, 1), TvT = view(sT, 1, LD6);
  // W = T diag(beta e^gamma) K -> B1 ; U = T diag(beta) V -> B2
  {
    float acc[TD][4];
    zero(acc);
    gemmx<B16, TD, NTD, NWG, true>(acc, cols_scaled(rm(sT, LD6), sbeg), rm(sK, LDI), 64, warp, lane);
    each<TD, NTD, NWG, true>(acc, warp, lane, [&](int i, int c, float& x) { B1[i * LDF + c] = x; });
    zero(acc);
    gemmx<B16, TD, NTD, NWG, true>(acc, cols_scaled(rm(sT, LD6), sb), rm(sV, LDI), 64, warp, lane);
    each<TD, NTD, NWG, true>(acc, warp, lane, [&](int i, int c, float& x) { B2[i * LDF + c] = x; });
  }
  __syncthreads();
  const auto B1v = view(B1, LDF, 1), B3v = view(B3, LDF, 1);
  // Delta = U - W S^T (B2);  dDelta = scale Aqk^T dO + diag(dec) K dSn^T (B3)
  {
    float acc[TD][4];
    zero(acc);
    gemmx<B16, TD, NTD, NWG, true>(acc, rm(B1, LDF), SvT, D, warp, lane);
    float acc2[TD][4];
    zero(acc2);
    gemmx<B16, TD, NTD, NWG, true>(acc2, cm(sP, LD6), rm(sdO, LDI), 64, warp, lane);
    float acc3[TD][4];
    zero(acc3);
    gemmx<B16, TD, NTD, NWG, true>(acc3, rm(sK, LDI), cm(dSn, D), D, warp, lane);
    __syncthreads();   // every warp has read W (B1), U (B2) as operands of its own tiles only
    each<TD, NTD, NWG, true>(acc, warp, lane, [&](int i, int r, float& x) { B2[i * LDF + r] -= x; });
    each<TD, NTD, NWG, true>(acc3, warp, lane, [&](int i, int, float& x) { x *= sdec[i]; });
#pragma unroll
    for (int ti = 0; ti < TD; ++ti)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc2[ti][e] = scale * acc2[ti][e] + acc3[ti][e];
    each<TD, NTD, NWG, true>(acc2, warp, lane, [&](int i, int r, float& x) { B3[i * LDF + r] = x; });
  }
  __syncthreads();
  float dq[TD][4], dk[TD][4];
  zero(dq);
  zero(dk);
  // dAqk = scale dO Delta^T; rho = dAqk o Aqk -> dgamma; G = dAqk o Gamma (into sP)
  {
    float a1[T6][4];
    zero(a1);
    gemmx<B16, T6, 8, NWG, true>(a1, rm(sdO, LDI), cm(B2, LDF), D, warp, lane);
    __syncthreads();   // sP (Aqk) fully read as an operand before it is overwritten
    each<T6, 8, NWG, true>(a1, warp, lane, [&](int i, int j, float& x) {
      float gval = 0.f;
      if (j <= i) {
        const float dA = scale * x;
        const float rho = dA * sP[i * LD6 + j];
        atomicAdd(&sdgam[i], rho);
        atomicAdd(&sdgam[j], -rho);
        gval = dA * expf(sgam[i] - sgam[j]);
      }
      sP[i * LD6 + j] = gval;
    });
  }
  __syncthreads();
  // dq += scale e^gamma (dO S) + G K ; dk += G^T Q ; dgamma += q . (scale e^gamma dO S)
  {
    float acc[TD][4];
    zero(acc);
    gemmx<B16, TD, NTD, NWG, true>(acc, rows_scaled(rm(sdO, LDI), ssc), Sv, D, warp, lane);
    row_dot<TD, NTD, NWG, true>(acc, Qv, sdgam, warp, lane);
#pragma unroll
    for (int ti = 0; ti < TD; ++ti)
#pragma unroll
      for (int e = 0; e < 4; ++e) dq[ti][e] += acc[ti][e];
    gemmx<B16, TD, NTD, NWG, true>(dq, rm(sP, LD6), rm(sK, LDI), 64, warp, lane);
    gemmx<B16, TD, NTD, NWG, true>(dk, cm(sP, LD6), rm(sQ, LDI), 64, warp, lane);
  }
  // exit state: Z = Delta dSn ; dk += dec o Z ; ddec = rowsum(K o Z)
  {
    float acc[TD][4];
    zero(acc);
    gemmx<B16, TD, NTD, NWG, true>(acc, rm(B2, LDF), rm(dSn, D), D, warp, lane);
    row_dot<TD, NTD, NWG, true>(acc, Kv, sz, warp, lane);
    each<TD, NTD, NWG, true>(acc, warp, lane, [&](int i, int, float& x) { x *= sdec[i]; });
#pragma unroll
    for (int ti = 0; ti < TD; ++ti)
#pragma unroll
      for (int e = 0; e < 4; ++e) dk[ti][e] += acc[ti][e];
  }
  // <dSn, S> for the e^{gamma_C} S term
  {
    float part = 0.f;
    const float4* a4 = reinterpret_cast<const float4*>(dSn);
    const float4* b4 = reinterpret_cast<const float4*>(S);
#pragma unroll 8
    for (int idx = tid; idx < D * D / 4; idx += NTG) {
      const float4 x = a4[idx], y = b4[idx];
      part += x.x * y.x + x.y * y.y + x.z * y.z + x.w * y.w;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (lane == 0) atomicAdd(&sdgam[63], seg[63] * part);
  }
  __syncthreads();
  if (tid < 64) {
    const float t = sdec[tid] * sz[tid];
    atomicAdd(&sdgam[tid], -t);
    atomicAdd(&sdgam[63], t);
  }
  // dW = -dDelta S (B1) ;  X = T^T dDelta (B2, Delta no longer needed)
  {
    float acc[TD][4], acc2[TD][4];
    zero(acc);
    zero(acc2);
    gemmx<B16, TD, NTD, NWG, true>(acc, rm(B3, LDF), Sv, D, warp, lane);
    gemm<TD, NTD, NWG, true>(acc2, TvT, B3v, 64, warp, lane);
    __syncthreads();
    each<TD, NTD, NWG, true>(acc, warp, lane, [&](int i, int c, float& x) { B1[i * LDF + c] = -x; });
    each<TD, NTD, NWG, true>(acc2, warp, lane, [&](int i, int c, float& x) { B2[i * LDF + c] = x; });
  }
  __syncthreads();
  // dv = beta X ; dbeta += rowsum(V o X)  (a warp covers 32 columns of one row: warp sum,
  // then one atomic per row segment)
  {
    Tin* dv = (Tin*)p.dv;
    for (int idx = tid; idx < 64 * D; idx += NTG) {
      const int i = idx / D, c = idx % D;
      const float t = B2[i * LDF + c];
      if (i < L) dv[((size_t)(c0 + i) * H + h) * D + c] = from_f<Tin>(sb[i] * t);
      float r = Vv(i, c) * t;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
      if (lane == 0) atomicAdd(&sred[i], r);
    }
  }
  // dT = dDelta (diag(beta) V)^T + dW (diag(beta e^gamma) K)^T  (into sP)
  {
    float a1[T6][4];
    zero(a1);
    gemmx<B16, T6, 8, NWG, true>(a1, rm(B3, LDF), cols_scaled(cm(sV, LDI), sb), D, warp, lane);
    gemmx<B16, T6, 8, NWG, true>(a1, rm(B1, LDF), cols_scaled(cm(sK, LDI), sbeg), D, warp, lane);
    each<T6, 8, NWG, true>(a1, warp, lane, [&](int i, int j, float& x) { sP[i * LD6 + j] = x; });
  }
  __syncthreads();
  // Y = T^T dW ; dk += beta e^gamma Y ; kt = rowsum(K o Y) -> dbeta += e^gamma kt,
  // dgamma += beta e^gamma kt
  {
    float acc[TD][4];
    zero(acc);
    gemm<TD, NTD, NWG, true>(acc, TvT, B1v, 64, warp, lane);
    if (tid < 64) sz[tid] = 0.f;
    __syncthreads();
    row_dot<TD, NTD, NWG, true>(acc, Kv, sz, warp, lane);
    each<TD, NTD, NWG, true>(acc, warp, lane, [&](int i, int, float& x) { x *= sbeg[i]; });
#pragma unroll
    for (int ti = 0; ti < TD; ++ti)
#pragma unroll
      for (int e = 0; e < 4; ++e) dk[ti][e] += acc[ti][e];
  }
  __syncthreads();
  if (tid < 64) {
    sred[tid] += seg[tid] * sz[tid];
    sdgam[tid] += sbeg[tid] * sz[tid];
  }
  // dA = -(T^T dT T^T) strictly lower: X1 = dT T^T (B1 as [64][65]), dA = -T^T X1 (B2)
  {
    float a1[T6][4];
    zero(a1);
    gemm<T6, 8, NWG, true>(a1, view(sP, LD6, 1), TvT, 64, warp, lane);
    each<T6, 8, NWG, true>(a1, warp, lane, [&](int i, int j, float& x) { B1[i * LD6 + j] = x; });
  }
  __syncthreads();
  {
    float a1[T6][4];
    zero(a1);
    gemm<T6, 8, NWG, true>(a1, TvT, view(B1, LD6, 1), 64, warp, lane);
    each<T6, 8, NWG, true>(a1, warp, lane, [&](int i, int j, float& x) { B2[i * LD6 + j] = (j < i) ? -x : 0.f; });
  }
  __syncthreads();
  // from A_ij = beta_i Ak_ij: dbeta_i += sum_j dA_ij Ak_ij; dgamma_i/j +- dA beta Ak;
  // dKK_ij = dA_ij beta_i Gamma_ij (into sP)
  // (a warp covers 32 columns j of one row i: the row-i sums go through a warp sum)
  for (int idx = tid; idx < 64 * 64; idx += NTG) {
    const int i = idx >> 6, j = idx & 63;
    float dkk = 0.f, r1 = 0.f, rho = 0.f;
    if (j < i) {
      const float dA = B2[i * LD6 + j], ak = sM[i * LD6 + j];
      r1 = dA * ak;
      rho = dA * sb[i] * ak;
      atomicAdd(&sdgam[j], -rho);
      dkk = dA * sb[i] * expf(sgam[i] - sgam[j]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      r1 += __shfl_xor_sync(0xffffffffu, r1, o);
      rho += __shfl_xor_sync(0xffffffffu, rho, o);
    }
    if (lane == 0) {
      atomicAdd(&sred[i], r1);
      atomicAdd(&sdgam[i], rho);
    }
    sP[i * LD6 + j] = dkk;
  }
  __syncthreads();
  // dk += dKK K + dKK^T K
  gemmx<B16, TD, NTD, NWG, true>(dk, rm(sP, LD6), rm(sK, LDI), 64, warp, lane);
  gemmx<B16, TD, NTD, NWG, true>(dk, cm(sP, LD6), rm(sK, LDI), 64, warp, lane);
  // write dq, dk
  {
    Tin* dqo = (Tin*)p.dq;
    Tin* dko = (Tin*)p.dk;
    if (p.dqk_f32) {
      // grouped heads: FP32 per value head, summed over each block afterwards
      float* dqf = reinterpret_cast<float*>(p.dq);
      float* dkf = reinterpret_cast<float*>(p.dk);
      each<TD, NTD, NWG, true>(dq, warp, lane, [&](int i, int c, float& x) {
        if (i < L) dqf[((size_t)(c0 + i) * H + h) * D + c] = x;
      });
      each<TD, NTD, NWG, true>(dk, warp, lane, [&](int i, int c, float& x) {
        if (i < L) dkf[((size_t)(c0 + i) * H + h) * D + c] = x;
      });
    } else {
      each<TD, NTD, NWG, true>(dq, warp, lane, [&](int i, int c, float& x) {
        if (i < L) dqo[((size_t)(c0 + i) * H + h) * D + c] = from_f<Tin>(x);
      });
      each<TD, NTD, NWG, true>(dk, warp, lane, [&](int i, int c, float& x) {
        if (i < L) dko[((size_t)(c0 + i) * H + h) * D + c] = from_f<Tin>(x);
      });
    }
  }
  __syncthreads();
  // dgate = reverse cumulative sum of dgamma; dbeta
  if (tid < 32) {
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
  return true;
}

// Slots blockIdx.x, blockIdx.x + gridDim.x, ... until the first empty one (the grid may be
// smaller than the slot count: packed inputs whose offsets end early leave slots empty).
template <typename Tin, int D>
__global__ void __launch_bounds__(NTG) mma_bwd_grad_kernel(const ChainParams p, int64_t slots) {
  for (int64_t slot = blockIdx.x; slot < slots; slot += gridDim.x) {
    if (!grad_chunk<Tin, D>(p, slot)) break;
    __syncthreads();   // shared memory is rewritten by the next chunk
  }
}

template <typename Tin, int D>
static cudaError_t launch_grad_t(const ChainParams& p, int64_t slots, cudaStream_t st) {
  const size_t smem = sizeof(float) * (3 * 64 * G_LD6 + 3 * 64 * g_ldf<Tin, D>() + 11 * 64) +
                      sizeof(Tin) * 4 * 64 * (D + 8);
  auto kern = mma_bwd_grad_kernel<Tin, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (slots > 0) kern<<<dim3((unsigned)slot_grid(p, slots), p.H), NTG, smem, st>>>(p, slots);
  return cudaGetLastError();
}

cudaError_t launch_mma_bwd_grad(const ChainParams& p, bool bf16, int D, int64_t slots,
                                cudaStream_t st) {
  if (bf16 && D == 64) return launch_grad_t<__nv_bfloat16, 64>(p, slots, st);
  if (!bf16 && D == 64) return launch_grad_t<float, 64>(p, slots, st);
  return cudaErrorInvalidValue;
}

}  // namespace sfg
