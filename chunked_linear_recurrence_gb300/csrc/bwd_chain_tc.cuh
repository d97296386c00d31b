// bwd_chain_tc.cuh -- the BF16 head-size-128 backward's reverse cotangent chain on tcgen05
// (bwd_chain_tc.cu).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "chunk_record.cuh"
#include "simt_chunk.cuh"

namespace sfg {

// The reverse cotangent chain of every (sequence, head) over the chunk records `fac`
// ([slots,H] of REC_BYTES: Ahat, (-W)^T and the decays of chunk_record.cuh): writes each
// chunk's exit cotangent to p.tape (BF16 swizzled tiles) and the sequence-start cotangent to
// p.ds0 (when non-NULL).  BF16, K = V = 128.
cudaError_t launch_tc_bwd_chain(const ChainParams& p, const float* fac, cudaStream_t st);
// Qg = scale diag(e^gamma) Q into every chunk record of `fac` (the records the state replay
// kept have no Qg).
cudaError_t launch_tc_bwd_qg(const ChainParams& p, float* fac, int64_t slots, cudaStream_t st);

}  // namespace sfg
