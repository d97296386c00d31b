// scan.cuh -- launcher of the segment-map exclusive scan.
#pragma once
#include <cuda_runtime.h>

namespace sfg {
cudaError_t launch_state_scan(int R, int H, int D, const float* P, const float* E,
                              const float* S0, float* entry, float* final_state, cudaStream_t st);
// Reverse scan of cotangent maps: exits[R-1] = dSf, exits[j-1] = exits[j] P_j^T + C_j,
// d_initial = exits[0] P_0^T + C_0.
cudaError_t launch_state_scan_reverse(int R, int H, int D, const float* P, const float* C,
                                      const float* dSf, float* exits, float* d_initial,
                                      cudaStream_t st);
}
