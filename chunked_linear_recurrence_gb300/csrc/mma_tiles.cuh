// mma_tiles.cuh -- warp-level tensor-core tiles for the backward kernels: element views
// of shared/global operands, tile GEMMs over a warp's fixed set of 16x8 output tiles
// (mma.sync m16n8k8 with TF32 operands, or m16n8k16 with BF16 operand pairs; FP32
// accumulation, the same accumulator layout), and tile epilogues.
#pragma once

#include "common.cuh"
#include "solve_tc.cuh"

namespace sfg {
namespace mt {

// Element (r, c) views of the operands.
template <typename T>
struct View {
  const T* p;
  int sr, sc;
  __device__ __forceinline__ float operator()(int r, int c) const { return to_f(p[r * sr + c * sc]); }
};
template <typename T>
__device__ __forceinline__ View<T> view(const T* p, int sr, int sc) { return View<T>{p, sr, sc}; }

// BF16 pairs: the low half holds the first element (the lower k index of an mma operand).
__device__ __forceinline__ uint32_t pk(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ float2 upk(uint32_t u) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u));
}
// Two adjacent elements p[0], p[1] as a BF16 pair (p 4-byte aligned for BF16, 8-byte for FP32).
__device__ __forceinline__ uint32_t pair_at(const __nv_bfloat16* p) {
  return *reinterpret_cast<const uint32_t*>(p);
}
__device__ __forceinline__ uint32_t pair_at(const float* p) {
  const float2 f = *reinterpret_cast<const float2*>(p);
  return pk(f.x, f.y);
}
// Two separate elements as a BF16 pair (BF16 elements keep their bits).
__device__ __forceinline__ uint32_t pair_of(const __nv_bfloat16* lo, const __nv_bfloat16* hi) {
  return (uint32_t)__bfloat16_as_ushort(*lo) | ((uint32_t)__bfloat16_as_ushort(*hi) << 16);
}
__device__ __forceinline__ uint32_t pair_of(const float* lo, const float* hi) { return pk(*lo, *hi); }
// Two adjacent elements as FP32 (for views that scale before rounding).
__device__ __forceinline__ float2 f2_at(const float* p) { return *reinterpret_cast<const float2*>(p); }
__device__ __forceinline__ float2 f2_at(const __nv_bfloat16* p) { return upk(pair_at(p)); }

// Row-major (element (r, c) at p[r ld + c]) and column-major (at p[c ld + r]) views with
// the BF16 pair accessors of the m16n8k16 operands: pc(r, c) = (x(r, c), x(r, c + 1)),
// pr(r, c) = (x(r, c), x(r + 1, c)).  The pair along the contiguous index is one load
// (ld even, the first index of the pair even).
template <typename T>
struct RM {
  const T* p;
  int ld;
  __device__ __forceinline__ float operator()(int r, int c) const { return to_f(p[r * ld + c]); }
  __device__ __forceinline__ uint32_t pc(int r, int c) const { return pair_at(p + r * ld + c); }
  __device__ __forceinline__ uint32_t pr(int r, int c) const {
    return pair_of(p + r * ld + c, p + (r + 1) * ld + c);
  }
  // the same pairs in FP32
  __device__ __forceinline__ float2 fc(int r, int c) const { return f2_at(p + r * ld + c); }
  __device__ __forceinline__ float2 fr(int r, int c) const {
    return make_float2(to_f(p[r * ld + c]), to_f(p[(r + 1) * ld + c]));
  }
};
template <typename T>
struct CM {
  const T* p;
  int ld;
  __device__ __forceinline__ float operator()(int r, int c) const { return to_f(p[c * ld + r]); }
  __device__ __forceinline__ uint32_t pc(int r, int c) const {
    return pair_of(p + c * ld + r, p + (c + 1) * ld + r);
  }
  __device__ __forceinline__ uint32_t pr(int r, int c) const { return pair_at(p + c * ld + r); }
  __device__ __forceinline__ float2 fc(int r, int c) const {
    return make_float2(to_f(p[c * ld + r]), to_f(p[(c + 1) * ld + r]));
  }
  __device__ __forceinline__ float2 fr(int r, int c) const { return f2_at(p + c * ld + r); }
};
template <typename T>
__device__ __forceinline__ RM<T> rm(const T* p, int ld) { return RM<T>{p, ld}; }
template <typename T>
__device__ __forceinline__ CM<T> cm(const T* p, int ld) { return CM<T>{p, ld}; }

// rows scaled by s[r]
template <typename V>
struct RowScaled {
  V v;
  const float* s;
  __device__ __forceinline__ float operator()(int r, int c) const { return s[r] * v(r, c); }
  // (pairs: scaled in FP32, then rounded once)
  __device__ __forceinline__ uint32_t pc(int r, int c) const {
    const float2 x = v.fc(r, c);
    return pk(s[r] * x.x, s[r] * x.y);
  }
  __device__ __forceinline__ uint32_t pr(int r, int c) const {
    const float2 x = v.fr(r, c);
    return pk(s[r] * x.x, s[r + 1] * x.y);
  }
};
// columns scaled by s[c]
template <typename V>
struct ColScaled {
  V v;
  const float* s;
  __device__ __forceinline__ float operator()(int r, int c) const { return s[c] * v(r, c); }
  __device__ __forceinline__ uint32_t pc(int r, int c) const {
    const float2 x = v.fc(r, c);
    return pk(s[c] * x.x, s[c + 1] * x.y);
  }
  __device__ __forceinline__ uint32_t pr(int r, int c) const {
    const float2 x = v.fr(r, c);
    return pk(s[c] * x.x, s[c] * x.y);
  }
};
template <typename V>
__device__ __forceinline__ RowScaled<V> rows_scaled(V v, const float* s) { return RowScaled<V>{v, s}; }
template <typename V>
__device__ __forceinline__ ColScaled<V> cols_scaled(V v, const float* s) { return ColScaled<V>{v, s}; }

// Which 16x8 output tiles a warp owns.  Plain (BLK = false): tile id = warp + NW ti of an
// output with NTN 8-column tiles per 16-row band.  Blocked (BLK = true): each warp owns a
// WM x WN block of tiles (WM 16-row bands, WN 8-column tiles), so that every A fragment it
// loads serves WN products and every B fragment WM of them.
template <int NTILE, int NTN, int NW, bool BLK>
struct TileMap {
  static constexpr int MBANDS = NW * NTILE / NTN;
  static constexpr int WM = (BLK && NTILE >= 4 && NTILE % 2 == 0 && MBANDS % 2 == 0) ? 2 : 1;
  static constexpr int WN = BLK ? NTILE / WM : 1;
  static_assert(!BLK || (MBANDS / WM) * (NTN / WN) == NW, "warp blocks tile the output");
  __device__ static __forceinline__ void at(int warp, int ti, int& m0, int& n0) {
    if (BLK) {
      const int wm = warp / (NTN / WN), wn = warp % (NTN / WN);
      m0 = (wm * WM + ti / WN) * 16;
      n0 = (wn * WN + ti % WN) * 8;
    } else {
      const int id = warp + NW * ti;
      m0 = (id / NTN) * 16;
      n0 = (id % NTN) * 8;
    }
  }
};

// acc[ti] += A[m0:m0+16, 0:K] B[0:K, n0:n0+8] for this warp's tiles (TileMap).  The k loop
// is outermost and all of a k step's fragments are loaded before its products, so that a
// warp has them all in flight at once (operands in global memory take an L2 round trip).
template <int NTILE, int NTN, int NW = 8, bool BLK = false, typename AV, typename BV>
__device__ __forceinline__ void gemm(float (&acc)[NTILE][4], const AV& A, const BV& B, int K,
                                     int warp, int lane) {
  using M = TileMap<NTILE, NTN, NW, BLK>;
  // distinct A fragments (16-row bands) and B fragments (8-column tiles) of the warp's tiles
  constexpr int NA = BLK ? M::WM : NTILE;
  constexpr bool kShareB = !BLK && (NW % NTN) == 0;
  constexpr int NB = BLK ? M::WN : (kShareB ? 1 : NTILE);
  const int g = lane >> 2, t = lane & 3;
  for (int k0 = 0; k0 < K; k0 += 8) {
    uint32_t a[NA][4], b[NB][2];
#pragma unroll
    for (int ia = 0; ia < NA; ++ia) {
      int m0, n0;
      M::at(warp, BLK ? ia * M::WN : ia, m0, n0);
      a[ia][0] = f2tf32(A(m0 + g, k0 + t));
      a[ia][1] = f2tf32(A(m0 + g + 8, k0 + t));
      a[ia][2] = f2tf32(A(m0 + g, k0 + t + 4));
      a[ia][3] = f2tf32(A(m0 + g + 8, k0 + t + 4));
    }
#pragma unroll
    for (int ib = 0; ib < NB; ++ib) {
      int m0, n0;
      M::at(warp, ib, m0, n0);
      b[ib][0] = f2tf32(B(k0 + t, n0 + g));
      b[ib][1] = f2tf32(B(k0 + t + 4, n0 + g));
    }
#pragma unroll
    for (int ti = 0; ti < NTILE; ++ti) {
      const int ia = BLK ? ti / M::WN : ti;
      const int ib = BLK ? ti % M::WN : (kShareB ? 0 : ti);
      mma_tf32_16x8x8(acc[ti], a[ia], b[ib]);
    }
  }
}

__device__ __forceinline__ void mma_bf16_16x8x16(float (&d)[4], const uint32_t (&a)[4],
                                                 const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// gemm with BF16 operands (m16n8k16, K a multiple of 16): A and B give BF16 pairs along k,
// A.pc(m, k) = (A(m, k), A(m, k + 1)) and B.pr(k, n) = (B(k, n), B(k + 1, n)).  Lane (g, t)
// holds rows m0 + g and m0 + g + 8 at k = k0 + 2t and k0 + 2t + 8 of A, column n0 + g at the
// same k of B; the accumulator layout is that of gemm.
template <int NTILE, int NTN, int NW = 8, bool BLK = false, typename AV, typename BV>
__device__ __forceinline__ void gemm16(float (&acc)[NTILE][4], const AV& A, const BV& B, int K,
                                       int warp, int lane) {
  using M = TileMap<NTILE, NTN, NW, BLK>;
  constexpr int NA = BLK ? M::WM : NTILE;
  constexpr bool kShareB = !BLK && (NW % NTN) == 0;
  constexpr int NB = BLK ? M::WN : (kShareB ? 1 : NTILE);
  const int g = lane >> 2, t2 = 2 * (lane & 3);
  for (int k0 = 0; k0 < K; k0 += 16) {
    uint32_t a[NA][4], b[NB][2];
#pragma unroll
    for (int ia = 0; ia < NA; ++ia) {
      int m0, n0;
      M::at(warp, BLK ? ia * M::WN : ia, m0, n0);
      a[ia][0] = A.pc(m0 + g, k0 + t2);
      a[ia][1] = A.pc(m0 + g + 8, k0 + t2);
      a[ia][2] = A.pc(m0 + g, k0 + t2 + 8);
      a[ia][3] = A.pc(m0 + g + 8, k0 + t2 + 8);
    }
#pragma unroll
    for (int ib = 0; ib < NB; ++ib) {
      int m0, n0;
      M::at(warp, ib, m0, n0);
      b[ib][0] = B.pr(k0 + t2, n0 + g);
      b[ib][1] = B.pr(k0 + t2 + 8, n0 + g);
    }
#pragma unroll
    for (int ti = 0; ti < NTILE; ++ti) {
      const int ia = BLK ? ti / M::WN : ti;
      const int ib = BLK ? ti % M::WN : (kShareB ? 0 : ti);
      mma_bf16_16x8x16(acc[ti], a[ia], b[ib]);
    }
  }
}

// gemm16 for BF16 inputs (the forward's operand precision), gemm (TF32) for FP32 inputs.
template <bool B16, int NTILE, int NTN, int NW = 8, bool BLK = false, typename AV, typename BV>
__device__ __forceinline__ void gemmx(float (&acc)[NTILE][4], const AV& A, const BV& B, int K,
                                      int warp, int lane) {
  if constexpr (B16)
    gemm16<NTILE, NTN, NW, BLK>(acc, A, B, K, warp, lane);
  else
    gemm<NTILE, NTN, NW, BLK>(acc, A, B, K, warp, lane);
}

template <int NTILE>
__device__ __forceinline__ void zero(float (&acc)[NTILE][4]) {
#pragma unroll
  for (int ti = 0; ti < NTILE; ++ti)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[ti][e] = 0.f;
}

// Calls f(row, col, value&) for every element this warp holds.
template <int NTILE, int NTN, int NW = 8, bool BLK = false, typename F>
__device__ __forceinline__ void each(float (&acc)[NTILE][4], int warp, int lane, F&& f) {
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int ti = 0; ti < NTILE; ++ti) {
    int m0, n0;
    TileMap<NTILE, NTN, NW, BLK>::at(warp, ti, m0, n0);
#pragma unroll
    for (int e = 0; e < 4; ++e) f(m0 + g + 8 * (e >> 1), n0 + 2 * t + (e & 1), acc[ti][e]);
  }
}

// vec[row] += sum over this warp's columns of w(row, col) acc(row, col) (4-lane reduction,
// then one shared-memory atomic per row segment).
template <int NTILE, int NTN, int NW = 8, bool BLK = false, typename W>
__device__ __forceinline__ void row_dot(const float (&acc)[NTILE][4], const W& w, float* vec,
                                        int warp, int lane) {
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int ti = 0; ti < NTILE; ++ti) {
    int m0, n0;
    TileMap<NTILE, NTN, NW, BLK>::at(warp, ti, m0, n0);
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int r = m0 + g + 8 * hr, c = n0 + 2 * t;
      float s = acc[ti][2 * hr] * w(r, c) + acc[ti][2 * hr + 1] * w(r, c + 1);
      s += __shfl_xor_sync(0xffffffffu, s, 1);
      s += __shfl_xor_sync(0xffffffffu, s, 2);
      if (t == 0) atomicAdd(&vec[r], s);
    }
  }
}

}  // namespace mt
}  // namespace sfg
