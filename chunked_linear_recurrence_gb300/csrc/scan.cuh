// scan.cuh -- launcher of the segment-map exclusive scan.
#pragma once
#include <cuda_runtime.h>

namespace sfg {
cudaError_t launch_state_scan(int R, int H, int D, const float* P, const float* E,
                              const float* S0, float* entry, float* final_state, cudaStream_t st);
}
