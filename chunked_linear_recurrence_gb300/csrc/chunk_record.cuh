// chunk_record.cuh -- the per-chunk factor record of the tensor-core kernels (BF16 inputs,
// K = V = 128): made by the split forward's preparation CTAs (and, in the state replay,
// kept per chunk-head for the backward's reverse chain) or by the backward's factor kernel.
// BF16 tiles in the 128-byte-swizzled panel layout of tc_ptx.cuh, then FP32 decays.
#pragma once
#include <stdint.h>

namespace sfg {

constexpr uint32_t R_W = 0;           // (-W)^T [128 k][64 i], one panel, 16 KB
constexpr uint32_t R_T1 = 16384;      // T' = T diag(beta) [64 i][64 j], 8 KB
constexpr uint32_t R_AH = 24576;      // Ahat = M o Gamma o Q K^T [64 i][64 j], 8 KB
constexpr uint32_t R_VEC = 32768;     // the decay vectors (FP32), at these offsets:
constexpr uint32_t V_DEC = 0;         //   e^{gamma_C - gamma_j}, j < 64
constexpr uint32_t V_EG = 256;        //   e^{gamma_i}, i < 64
constexpr uint32_t V_GC = 512;        //   e^{gamma_C}
constexpr uint32_t REC_BYTES = 33792;
static_assert(REC_BYTES % 16 == 0 && V_GC + 4 <= REC_BYTES - R_VEC, "record layout");

// The backward's copy of a record appends Qg = scale diag(e^gamma) Q [64 i][128 k] (two
// panels of 8 KB), the B operand of the reverse chain's dS += dO^T Qg.
constexpr uint32_t R_QG = REC_BYTES;
constexpr uint32_t REC2_BYTES = R_QG + 16384;
static_assert(R_QG % 1024 == 0, "record layout");

}  // namespace sfg
