// fwd_tc.cuh -- launcher of the tensor-core (tcgen05 / TMEM / TMA) forward for
// BF16 q/k/v with K = V = 128.
#pragma once
#include <cuda_runtime.h>

#include "simt_chunk.cuh"

namespace sfg {
// True when this build contains the tensor-core forward.
bool tc_fwd_available();
// status: device int the kernel sets to a nonzero code when a bounded wait expires.
cudaError_t launch_tc_fwd(const ChainParams& p, int* status, cudaStream_t st);
}  // namespace sfg
