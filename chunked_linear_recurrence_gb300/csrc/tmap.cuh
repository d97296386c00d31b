// tmap.cuh -- TMA tensor maps of the BF16 token-major tensors ([rows, H, 128]).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

namespace sfg {

// True when the driver entry point that encodes TMA descriptors is available (the tensor-core
// kernels are usable).  The environment variable SF_GDN_DISABLE_TMA_ENCODER (set to anything
// but "0" before the first call) makes it report false.
bool tc_fwd_available();
// TMA descriptor of a [rows, H, 128] BF16 tensor viewed as (128, H, rows), box 64 x 1 x 64,
// 128-byte swizzle (one head's 64-token chunk, in two 64-column panels).
bool make_bf16_map(CUtensorMap* m, const void* base, int rows, int H);
// The same tensor viewed as (64, rows, 2, H) with box 64 x 64 x 2 x 1: one copy moves a
// head's 64-token chunk as both 64-column panels (panel 1 right after panel 0, 8 KB apart).
// Coordinates (0, first row, 0, head).
bool make_bf16_map_4d(CUtensorMap* m, const void* base, int rows, int H);

}  // namespace sfg
