// bwd_chain_tc.cuh -- the BF16 head-size-128 backward's per-chunk factor record and the
// reverse cotangent chain on tcgen05 (bwd_chain_tc.cu).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "simt_chunk.cuh"

namespace sfg {

// Factor record of one chunk-head (written by mma_bwd_factor_kernel<128>, rows past the
// sequence end zero), BF16 tiles in the 128-byte-swizzled panel layout of tc_ptx.cuh:
constexpr uint32_t FB_AQK = 0;        // scale Aqk [64 i][64 j]  (Aqk = Gamma o Q K^T, lower)
constexpr uint32_t FB_NW = 8192;      // -W [64 i][128 k]       (two panels of 8 KB)
constexpr uint32_t FB_QG = 24576;     // scale diag(e^gamma) Q [64 i][128 k]
constexpr uint32_t FB_VEC = 40960;    // FP32: e^{gamma_C - gamma_j} [64], then e^{gamma_C}
constexpr uint32_t FB_BYTES = 41472;

// The reverse cotangent chain of every (sequence, head) over the factors `fac`: writes each
// chunk's exit cotangent to p.tape (BF16 swizzled tiles) and the sequence-start cotangent to
// p.ds0 (when non-NULL).  BF16, K = V = 128.
cudaError_t launch_tc_bwd_chain(const ChainParams& p, const float* fac, cudaStream_t st);

}  // namespace sfg
