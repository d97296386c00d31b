// solve_tc.cuh -- the chunk's unit-lower-triangular inverse T = (I + A)^{-1}
// (64 x 64, FP32 in shared memory) for the tensor-core kernels.
//
// The Attention Gym page describes the fused kernels' solve as hierarchical
// over 16x16 blocks.  Here:
//  1. the four 16x16 diagonal blocks are inverted by right-looking forward
//     substitution, one thread per block column (the dependency chain is one
//     FMA per row);
//  2. the off-diagonal blocks follow from T_10 = -T_11 A_10 T_00, first inside
//     each 32x32 half, then for the 32x32 lower-left block, with the 16x8x8
//     products on the warp-level TF32 tensor-core MMA (FP32 accumulate).
// Matrices use leading dimension SOLVE_LD (68 floats: conflict-free A-operand
// fragment loads).
#pragma once

#include <stdint.h>

namespace sfg {

constexpr int SOLVE_LD = 68;

__device__ __forceinline__ uint32_t f2tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}

// d += a * b, one m16n8k8 TF32 tile (FP32 accumulate).
__device__ __forceinline__ void mma_tf32_16x8x8(float (&d)[4], const uint32_t (&a)[4],
                                                const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// One warp: C0[0:16, 0:8] = alpha * A0[0:16, 0:K] B0[0:K, 0:8], where A0, B0, C0
// point at the sub-matrix origins (row-major FP32, leading dimension SOLVE_LD).
__device__ __forceinline__ void warp_tile_tf32(const float* A0, const float* B0, float* C0, int K,
                                               float alpha, int lane) {
  const int g = lane >> 2, t = lane & 3;
  float d[4] = {0.f, 0.f, 0.f, 0.f};
  for (int k = 0; k < K; k += 8) {
    const uint32_t a[4] = {f2tf32(A0[g * SOLVE_LD + k + t]), f2tf32(A0[(g + 8) * SOLVE_LD + k + t]),
                           f2tf32(A0[g * SOLVE_LD + k + t + 4]),
                           f2tf32(A0[(g + 8) * SOLVE_LD + k + t + 4])};
    const uint32_t b[2] = {f2tf32(B0[(k + t) * SOLVE_LD + g]), f2tf32(B0[(k + t + 4) * SOLVE_LD + g])};
    mma_tf32_16x8x8(d, a, b);
  }
  C0[g * SOLVE_LD + 2 * t] = alpha * d[0];
  C0[g * SOLVE_LD + 2 * t + 1] = alpha * d[1];
  C0[(g + 8) * SOLVE_LD + 2 * t] = alpha * d[2];
  C0[(g + 8) * SOLVE_LD + 2 * t + 1] = alpha * d[3];
}

// T = (I + A)^{-1}.  A: strictly lower 64x64 (entries on/above the diagonal are
// not read).  T: fully written (zeros above the diagonal).  X: 32 x SOLVE_LD
// FP32 scratch.  Called by `nthr` >= 128 threads (tid in [0, nthr)); warps 0-3
// run the tensor-core merges.  bar() synchronises exactly those threads.
template <typename Bar>
__device__ void solve64_tc(const float* A, float* T, float* X, int tid, int nthr, Bar bar) {
  const int warp = tid >> 5, lane = tid & 31;
  if (tid < 64) {
    const int b = tid >> 4, m = tid & 15, base = 16 * b;
    float acc[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = (i == m) ? 1.f : 0.f;
#pragma unroll
    for (int j = 0; j < 15; ++j) {
      const float x = acc[j];
#pragma unroll
      for (int i = j + 1; i < 16; ++i) acc[i] -= A[(base + i) * SOLVE_LD + base + j] * x;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) T[(base + i) * SOLVE_LD + base + m] = acc[i];
  } else {
    // zero the six 16x16 blocks above the block diagonal
    for (int idx = tid - 64; idx < 6 * 256; idx += nthr - 64) {
      const int blk = idx >> 8, e = idx & 255;
      const int br = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
      const int bc = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
      T[(16 * br + (e >> 4)) * SOLVE_LD + 16 * bc + (e & 15)] = 0.f;
    }
  }
  bar();
  // 32-level: in half p (rows/cols r0 = 32p), X_p = A_10 T_00 into X rows [16p, 16p+16),
  // then T_10 = -T_11 X_p.  Warp w: half p = w / 2, 8-column tile nt = w % 2.
  const int L = SOLVE_LD;
  if (warp < 4) {
    const int p = warp >> 1, nt = warp & 1, r0 = 32 * p;
    warp_tile_tf32(A + (r0 + 16) * L + r0, T + r0 * L + r0 + 8 * nt, X + 16 * p * L + 8 * nt, 16,
                   1.f, lane);
  }
  bar();
  if (warp < 4) {
    const int p = warp >> 1, nt = warp & 1, r0 = 32 * p;
    warp_tile_tf32(T + (r0 + 16) * L + r0 + 16, X + 16 * p * L + 8 * nt,
                   T + (r0 + 16) * L + r0 + 8 * nt, 16, -1.f, lane);
  }
  bar();
  // 64-level: X = A[32:64, 0:32] T[0:32, 0:32]; then T[32:64, 0:32] = -T[32:64, 32:64] X.
  // Eight 16x8 tiles (mt in {0,1}, nt in {0..3}), two per warp.
  if (warp < 4) {
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const int tile = 2 * warp + s, mt = tile >> 2, nt = tile & 3;
      warp_tile_tf32(A + (32 + 16 * mt) * L, T + 8 * nt, X + 16 * mt * L + 8 * nt, 32, 1.f, lane);
    }
  }
  bar();
  if (warp < 4) {
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const int tile = 2 * warp + s, mt = tile >> 2, nt = tile & 3;
      warp_tile_tf32(T + (32 + 16 * mt) * L + 32, X + 8 * nt, T + (32 + 16 * mt) * L + 8 * nt, 32,
                     -1.f, lane);
    }
  }
  bar();
}

// In-place variant: AT holds A (strictly lower) on entry and T on exit.  Each
// stage overwrites only blocks of A that no later stage reads: the diagonal
// blocks after every thread has its column in registers, A_10 of each 32x32
// half after X_p = A_10 T_00, and A[32:64, 0:32] after the 64-level X.
template <typename Bar>
__device__ void solve64_tc_inplace(float* AT, float* X, int tid, int nthr, Bar bar) {
  const int warp = tid >> 5, lane = tid & 31;
  const int L = SOLVE_LD;
  // diagonal blocks: warp b (< 4) inverts block b, lane m (and m + 16, redundantly) owns column m
  float acc[16];
  const int m = lane & 15, base = 16 * (warp & 3);
  if (warp < 4) {
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = (i == m) ? 1.f : 0.f;
#pragma unroll
    for (int j = 0; j < 15; ++j) {
      const float x = acc[j];
#pragma unroll
      for (int i = j + 1; i < 16; ++i) acc[i] -= AT[(base + i) * L + base + j] * x;
    }
  }
  bar();
  if (warp < 4) {
    if (lane < 16) {
#pragma unroll
      for (int i = 0; i < 16; ++i) AT[(base + i) * L + base + m] = acc[i];
    } else {
      // zero the six 16x16 blocks above the block diagonal (64 threads)
      for (int idx = warp * 16 + lane - 16; idx < 6 * 256; idx += 64) {
        const int blk = idx >> 8, e = idx & 255;
        const int br = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
        const int bc = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
        AT[(16 * br + (e >> 4)) * L + 16 * bc + (e & 15)] = 0.f;
      }
    }
  }
  bar();
  if (warp < 4) {
    const int p = warp >> 1, nt = warp & 1, r0 = 32 * p;
    warp_tile_tf32(AT + (r0 + 16) * L + r0, AT + r0 * L + r0 + 8 * nt, X + 16 * p * L + 8 * nt,
                   16, 1.f, lane);
  }
  bar();
  if (warp < 4) {
    const int p = warp >> 1, nt = warp & 1, r0 = 32 * p;
    warp_tile_tf32(AT + (r0 + 16) * L + r0 + 16, X + 16 * p * L + 8 * nt,
                   AT + (r0 + 16) * L + r0 + 8 * nt, 16, -1.f, lane);
  }
  bar();
  const int nw = nthr >> 5;
  for (int tile = warp; tile < 8; tile += nw) {
    const int mt = tile >> 2, nt = tile & 3;
    warp_tile_tf32(AT + (32 + 16 * mt) * L, AT + 8 * nt, X + 16 * mt * L + 8 * nt, 32, 1.f, lane);
  }
  bar();
  for (int tile = warp; tile < 8; tile += nw) {
    const int mt = tile >> 2, nt = tile & 3;
    warp_tile_tf32(AT + (32 + 16 * mt) * L + 32, X + 8 * nt, AT + (32 + 16 * mt) * L + 8 * nt, 32,
                   -1.f, lane);
  }
  bar();
}

}  // namespace sfg
