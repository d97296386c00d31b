// fwd_tc.cuh -- launcher of the tensor-core (tcgen05 / TMEM / TMA) chunk kernel for
// BF16 q/k/v with K = V = 128.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "simt_chunk.cuh"

namespace sfg {

// FWD: outputs + final state.  SUMMARY: per (range, head) the affine map's S_ext and
// P (p.bounds, p.N = number of ranges, results in p.E / p.P).  REPLAY: chunk-entry
// states into p.ckpt (the backward's state replay).
enum { TC_MODE_FWD = 0, TC_MODE_SUMMARY = 1, TC_MODE_REPLAY = 2 };

// True when this build can encode TMA descriptors (the tensor-core kernel is usable).
bool tc_fwd_available();
// TMA descriptor of a [rows, H, 128] BF16 tensor viewed as (128, H, rows), box 64 x 1 x 64,
// 128-byte swizzle (one head's 64-token chunk, in two 64-column panels).
bool make_bf16_map(CUtensorMap* m, const void* base, int rows, int H);
// status: device int the kernel sets to a nonzero code when a bounded wait expires.
cudaError_t launch_tc(const ChainParams& p, int mode, int* status, cudaStream_t st);

}  // namespace sfg
