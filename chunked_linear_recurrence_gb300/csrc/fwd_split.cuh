// fwd_split.cuh -- launcher of the split forward (preparation CTAs feeding state-chain CTAs
// through an L2-resident ring) for dense BF16 q/k/v with K = V = 128.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>

#include "simt_chunk.cuh"

namespace sfg {

// Workspace bytes the split forward needs for N sequences of H heads (status word included).
size_t split_fwd_workspace(int N, int H);
// Dense (p.cu == NULL) or packed (p.cu != NULL, p.B == 1) inputs, p.T > 0.  ws: workspace
// of split_fwd_workspace(p.N, p.H) bytes whose first 256 bytes are not used; status: the
// device status word.  With p.ckpt != NULL the launch is the backward's state replay: every
// chunk's entry state is written to p.ckpt ([slots,H] tiles of 32 KB, slots as
// chunk_slot_base: BF16 [128 v][128 k] in the 128-byte-swizzled panel layout of tc_ptx.cuh)
// and p.out / p.final_state may be NULL.
cudaError_t launch_split_fwd(const ChainParams& p, void* ws, int* status, cudaStream_t st);

// Workspace bytes of the segment summaries for R token ranges of H heads.
size_t split_summary_workspace(int R, int H);
// Segment summaries of p.N = R token ranges p.bounds ([R,2]) of the dense rows (p.B, p.T > 0)
// into p.P ([R,H,K,K]) and p.E ([R,H,V,K]) on the split kernel: each chunk's record is
// prepared once and read by two chain CTAs, one from S0 = 0 with the value term (E), one
// from S0 = I without it (P).  ws: split_summary_workspace(R, H) bytes, first 256 unused.
cudaError_t launch_split_summary(const ChainParams& p, void* ws, int* status, cudaStream_t st);

// Failure-detection tests: the next split launch on the calling host thread never publishes
// record `item` (production order) and gives every bounded wait `wait_limit_cycles` clock
// cycles, so that a wait runs out and the kernel takes its abort path (one shot).
void inject_split_timeout(long long item, long long wait_limit_cycles);

}  // namespace sfg
