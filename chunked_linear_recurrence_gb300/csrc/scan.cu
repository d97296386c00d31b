// scan.cu -- exclusive scan of segment maps (Attention Gym "Linear Attention",
// section "Context Parallelism": a prefix scan over the [bias; transition]
// summaries recovers every range's entry state; Megatron-LM PR "Mamba2
// state-passing context parallelism": exclusive causal scan of (S_ext, a_block)).
//
//   entry_0 = S0,  entry_{j+1} = entry_j P_j + S_ext_j,  final = entry_R
//
// and its reverse, for the state cotangents of the backward (whose per-segment map is
// dS_entry = dS_exit P^T + C): the segments are walked from the last one and P enters
// transposed, exit_{R-1} = dS_final, exit_{j-1} = exit_j P_j^T + C_j.
//
// Rows of the state are independent under right-multiplication by P, so the
// scan is split over (head, block of RB rows); each CTA keeps its rows in
// shared memory and walks the R segments in order.  FP32 throughout.
#include "common.cuh"
#include "scan.cuh"

namespace sfg {

template <int D, int RB, bool REV>
__global__ void __launch_bounds__(D) state_scan_kernel(int R, int H, const float* __restrict__ P,
                                                       const float* __restrict__ E,
                                                       const float* __restrict__ S0,
                                                       float* __restrict__ entry,
                                                       float* __restrict__ final_state) {
  __shared__ float cur[RB][D];
  const int c = threadIdx.x;                 // column owned by this thread
  const int h = blockIdx.y, r0 = blockIdx.x * RB;
  const size_t SZ = (size_t)D * D;
#pragma unroll
  for (int r = 0; r < RB; ++r)
    cur[r][c] = S0 ? S0[(size_t)h * SZ + (size_t)(r0 + r) * D + c] : 0.f;
  __syncthreads();
  for (int jj = 0; jj < R; ++jj) {
    const int j = REV ? R - 1 - jj : jj;
    const size_t base = ((size_t)j * H + h) * SZ;
    float acc[RB];
#pragma unroll
    for (int r = 0; r < RB; ++r) {
      entry[base + (size_t)(r0 + r) * D + c] = cur[r][c];
      acc[r] = E[base + (size_t)(r0 + r) * D + c];
    }
    const float* Pj = P + base;
#pragma unroll 4
    for (int m = 0; m < D; ++m) {
      const float pm = REV ? Pj[(size_t)c * D + m] : Pj[(size_t)m * D + c];
#pragma unroll
      for (int r = 0; r < RB; ++r) acc[r] += cur[r][m] * pm;
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < RB; ++r) cur[r][c] = acc[r];
    __syncthreads();
  }
  if (final_state)
#pragma unroll
    for (int r = 0; r < RB; ++r) final_state[(size_t)h * SZ + (size_t)(r0 + r) * D + c] = cur[r][c];
}

template <bool REV>
static cudaError_t launch_scan_t(int R, int H, int D, const float* P, const float* E,
                                 const float* S0, float* entry, float* final_state,
                                 cudaStream_t st) {
  constexpr int RB = 8;
  if (D == 64)
    state_scan_kernel<64, RB, REV><<<dim3(64 / RB, H), 64, 0, st>>>(R, H, P, E, S0, entry,
                                                                    final_state);
  else if (D == 128)
    state_scan_kernel<128, RB, REV><<<dim3(128 / RB, H), 128, 0, st>>>(R, H, P, E, S0, entry,
                                                                       final_state);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t launch_state_scan(int R, int H, int D, const float* P, const float* E,
                              const float* S0, float* entry, float* final_state, cudaStream_t st) {
  return launch_scan_t<false>(R, H, D, P, E, S0, entry, final_state, st);
}

cudaError_t launch_state_scan_reverse(int R, int H, int D, const float* P, const float* C,
                                      const float* dSf, float* exits, float* d_initial,
                                      cudaStream_t st) {
  return launch_scan_t<true>(R, H, D, P, C, dSf, exits, d_initial, st);
}

}  // namespace sfg
