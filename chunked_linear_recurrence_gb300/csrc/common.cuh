// common.cuh -- device helpers shared by the chunked gated-delta-rule kernels.
//
// Chunk algebra used throughout (per 64-token chunk, entry state S [V,K],
// gamma_i = cumulative natural-log gate inside the chunk; this is the WY/UT
// form the Attention Gym "Linear Attention" page names -- WY factors, a
// hierarchical 16x16-block triangular solve, raw QK/KK contracted before the
// masked non-positive decay differences are applied):
//
//   A_ij  = beta_i e^{gamma_i-gamma_j} (k_i.k_j), j < i;   T = (I + A)^-1
//   U     = T diag(beta) V;          W = T diag(beta e^gamma) K
//   Delta = U - W S^T                                   ("V_new", StateFlow Eq. 2)
//   O     = scale (diag(e^gamma) Q S^T + (M o Gamma o Q K^T) Delta)
//   S'    = e^{gamma_C} S + Delta^T diag(e^{gamma_C-gamma}) K
//
// Every decay factor is the exponential of a non-positive difference, so no
// intermediate overflows however negative the gates are.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace sfg {

constexpr int CHUNK = 64;

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// Token rows [bos, eos) of sequence n (flattened b*T + t), clamped into
// [0, B*T] so that malformed offsets can never address memory out of bounds.
__device__ __forceinline__ void seq_span(int n, int B, int T, const int32_t* cu,
                                         int64_t& bos, int64_t& eos) {
  const int64_t total = (int64_t)B * T;
  if (cu) {
    bos = cu[n];
    eos = cu[n + 1];
  } else {
    bos = (int64_t)n * T;
    eos = bos + T;
  }
  bos = bos < 0 ? 0 : (bos > total ? total : bos);
  eos = eos < bos ? bos : (eos > total ? total : eos);
}

__device__ __forceinline__ int64_t n_chunks(int64_t len) { return (len + CHUNK - 1) / CHUNK; }

// First per-chunk slot of sequence n in a [slots, H, V, K] workspace array:
// dense inputs use n * ceil(T/64); packed inputs the running sum of
// ceil(len_m/64) over the earlier sequences (so slots <= ceil(T/64) + N).
__device__ __forceinline__ int64_t chunk_slot_base(int n, int B, int T, const int32_t* cu) {
  if (!cu) return (int64_t)n * n_chunks(T);
  int64_t s = 0;
  for (int m = 0; m < n; ++m) {
    int64_t b, e;
    seq_span(m, B, T, cu, b, e);
    s += n_chunks(e - b);
  }
  return s;
}

// Chunk `slot` of the backward's chunk numbering (dense: n * ceil(T/64) + c; packed: the
// chunks of sequences 0 .. n-1 come first) -> sequence n, its rows [bos, eos) and the chunk
// index ci within it.  False when the slot holds no chunk; every later slot is then empty
// too, so a loop over slots may stop there.
__device__ __forceinline__ bool locate_chunk(int64_t slot, int B, int T, const int32_t* cu, int N,
                                             int& n, int64_t& bos, int64_t& eos, int64_t& ci) {
  if (!cu) {
    const int64_t nc = n_chunks(T);
    if (nc == 0) return false;
    n = (int)(slot / nc);
    ci = slot % nc;
    if (n >= N) return false;
    seq_span(n, B, T, nullptr, bos, eos);
    return true;
  }
  int64_t s = 0;
  for (int m = 0; m < N; ++m) {
    int64_t b, e;
    seq_span(m, B, T, cu, b, e);
    const int64_t c = n_chunks(e - b);
    if (slot < s + c) {
      n = m;
      ci = slot - s;
      bos = b;
      eos = e;
      return true;
    }
    s += c;
  }
  return false;
}

// Inclusive prefix sum of 64 values held in smem, by one warp (2 per lane).
__device__ __forceinline__ void warp_cumsum64(const float* in, float* out, int lane) {
  const float a = in[2 * lane], b = in[2 * lane + 1];
  float s = a + b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float t = __shfl_up_sync(0xffffffffu, s, o);
    if (lane >= o) s += t;
  }
  const float excl = s - (a + b);
  out[2 * lane] = excl + a;
  out[2 * lane + 1] = excl + a + b;
}

// T = (I + A)^{-1} for a strictly lower-triangular 64x64 FP32 matrix A
// (row-major, leading dimension ld; entries on/above the diagonal ignored).
// Hierarchical: the four 16x16 diagonal blocks by forward substitution (one
// thread per block column), then the 32x32 and 64x64 levels by
//   T_10 = -T_11 A_10 T_00.
// T gets zeros above the diagonal.  `scratch` needs 1024 floats.  All
// `nthr` threads (tid in [0, nthr)) must call it; it ends with a barrier
// among them (bar_sync is the caller's barrier for that thread set).
template <typename Bar>
__device__ void solve_unit_lower64(const float* A, float* T, int ld, float* scratch, int tid,
                                   int nthr, Bar bar_sync) {
  for (int idx = tid; idx < 64 * 64; idx += nthr) {
    const int i = idx >> 6, j = idx & 63;
    if (j >= i) T[i * ld + j] = (i == j) ? 1.f : 0.f;
  }
  if (tid < 64) {
    const int b = tid >> 4, m = tid & 15, base = 16 * b;
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float s = (i == m) ? 1.f : 0.f;
#pragma unroll
      for (int j = 0; j < i; ++j) s -= A[(base + i) * ld + base + j] * x[j];
      x[i] = s;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i)
      if (i > m) T[(base + i) * ld + base + m] = x[i];
  }
  bar_sync();
  // 32-level: in each 32-block p, X = A_10 T_00 then T_10 = -T_11 X (16x16 blocks)
  for (int idx = tid; idx < 512; idx += nthr) {
    const int p = idx >> 8, i = (idx >> 4) & 15, m = idx & 15;
    const int r = 32 * p + 16 + i, c0 = 32 * p;
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) s += A[r * ld + c0 + j] * T[(c0 + j) * ld + c0 + m];
    scratch[idx] = s;
  }
  bar_sync();
  for (int idx = tid; idx < 512; idx += nthr) {
    const int p = idx >> 8, i = (idx >> 4) & 15, m = idx & 15;
    const int r = 32 * p + 16 + i, c0 = 32 * p;
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) s += T[r * ld + c0 + 16 + j] * scratch[(p << 8) + (j << 4) + m];
    T[r * ld + c0 + m] = -s;
  }
  bar_sync();
  // 64-level: X = A_[10] T_[00] (32x32), T_[10] = -T_[11] X
  for (int idx = tid; idx < 1024; idx += nthr) {
    const int i = idx >> 5, m = idx & 31;
    float s = 0.f;
#pragma unroll 8
    for (int j = m; j < 32; ++j) s += A[(32 + i) * ld + j] * T[j * ld + m];
    scratch[idx] = s;
  }
  bar_sync();
  for (int idx = tid; idx < 1024; idx += nthr) {
    const int i = idx >> 5, m = idx & 31;
    float s = 0.f;
#pragma unroll 8
    for (int j = 0; j <= i; ++j) s += T[(32 + i) * ld + 32 + j] * scratch[(j << 5) + m];
    T[(32 + i) * ld + m] = -s;
  }
  bar_sync();
}

}  // namespace sfg
