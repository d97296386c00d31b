// fwd_tc.cu -- tensor-core forward (placeholder until the kernel lands).
#include "fwd_tc.cuh"

namespace sfg {
bool tc_fwd_available() { return false; }
cudaError_t launch_tc_fwd(const ChainParams&, int*, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace sfg
