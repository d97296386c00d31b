/*
 * sf_gdn.h -- C ABI of the chunk-parallel gated delta rule for GB300 (sm_103a).
 *
 * The operation (Attention Gym, "Linear Attention" page, section "Gated Delta
 * Rule"): for every sequence n and value head h, with state S [V,K] carried in
 * FP32 from an initial state (zero when none is given), each token applies
 *
 *     decayed  = exp(gate) * S                 (gate: natural log, scalar)
 *     residual = beta * (v - decayed @ k)
 *     S        = decayed + outer(residual, k)
 *     out      = scale * S @ q                 (the query reads the UPDATED state)
 *
 * The kernels compute it chunk-parallel in 64-token chunks (StateFlow paper,
 * section 2.2, Eq. 2: Pre / ST / Out); chunking changes only the order of the
 * floating-point operations, not the result.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  * Every tensor pointer is a DEVICE pointer owned by the caller.  The library
 *    allocates no device or host memory in any entry point; scratch comes from
 *    the caller's `workspace` (size from the matching *_workspace query), or,
 *    for sf_gdn_chunk_bwd_noalloc only, from a fixed array built into the
 *    library.
 *  * Layouts are contiguous, row-major:
 *        q, k    [B, T, HK, K]     v, out, d_out  [B, T, H, V]
 *        gate, beta, dgate, dbeta  [B, T, H]  (FP32)
 *        states  [N, H, V, K] (FP32; V-major: S @ k is a [V] vector)
 *        cu_seqlens  int32 [N+1] or NULL
 *  * Grouped query/key heads (Attention Gym chunk_gdn parameter table): HK
 *    divides H and value head h reads query/key head h / (H / HK), i.e. each
 *    block of H / HK consecutive value heads shares one query/key head; dq and
 *    dk of a shared head are the sums over its block.  HK = H is the plain case.
 *  * q/k/v (and out, d_out, dq, dk, dv) share one dtype: SF_BF16 or SF_F32.
 *    gate, beta and every state are FP32; all recurrence math is FP32.
 *  * Supported head sizes: K == V, either 64 or 128 (else SF_ERR_UNSUPPORTED).
 *    Element offsets must fit in int32 (B*T*H*max(K,V) < 2^31), else
 *    SF_ERR_UNSUPPORTED.  Base pointers of q, k, v, out must be 16-byte aligned.
 *  * Packed varlen (Attention Gym chunk_gdn contract): with cu_seqlens != NULL,
 *    B must be 1 and N = number of sequences; sequence n owns token rows
 *    [cu_seqlens[n], cu_seqlens[n+1]).  Offsets start at 0, never decrease and
 *    may end before T; rows at or past cu_seqlens[N] are inactive: never read
 *    as part of a sequence, never written.  Repeated offsets are empty
 *    sequences whose state passes through unchanged.  Each sequence is chunked
 *    from its own first token, so its last chunk may be partial.  These device
 *    values are the caller's responsibility on the hot path; kernels clamp
 *    them into [0, B*T] so that a bad offset cannot make them access memory
 *    out of bounds, and sf_validate_cu_seqlens checks them synchronously.
 *  * Every call is asynchronous on `stream` (NULL = legacy default stream) and
 *    never synchronises the host.  Host-visible argument errors are reported
 *    before anything is launched.  Nothing falls back to another
 *    implementation: an unsupported request returns SF_ERR_UNSUPPORTED.
 *  * The workspace's first 256 bytes hold a device status word.  A kernel
 *    whose internal wait exceeds its time limit writes SF_ERR_TIMEOUT there
 *    and returns; sf_workspace_status reads (and clears) it.  The next word
 *    records where the first expired wait was (a diagnostic: bit 30 set, the
 *    block index in bits 12-29, the warp in bits 6-11, the awaited barrier in
 *    bits 0-5); it is left for the caller to read and clear.
 *  * sf_last_error() describes the last non-SF_OK status of the calling host
 *    thread.
 */
#ifndef SF_GDN_H
#define SF_GDN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; declared here so the header needs no CUDA headers. */
typedef struct CUstream_st *sf_stream_t;

typedef enum {
  SF_OK = 0,
  SF_ERR_INVALID_ARG = 1,   /* NULL pointer, bad size or alignment, inconsistent shape */
  SF_ERR_UNSUPPORTED = 2,   /* valid request outside what the kernels implement */
  SF_ERR_WORKSPACE = 3,     /* workspace NULL or smaller than the query returned */
  SF_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
  SF_ERR_TIMEOUT = 5        /* a kernel's bounded internal wait expired (status word) */
} sf_status;

typedef enum { SF_F32 = 0, SF_BF16 = 1 } sf_dtype;

/* Problem shape.  N = number of sequences: B when cu_seqlens is NULL, else
 * len(cu_seqlens) - 1 (and then B must be 1).  scale <= 0 selects 1/sqrt(K).
 * H = value heads (v, gate, beta, states); HK = query/key heads, which must
 * divide H (0 means HK = H, so a zero-initialised shape keeps every head). */
typedef struct {
  int B, T, H, K, V, N;
  sf_dtype dtype;
  float scale;
  int HK;
} sf_gdn_shape;

/* Description of the calling thread's last error (never NULL). */
const char *sf_last_error(void);

/* Library version string, e.g. "sf_gdn 0.1 sm_103a". */
const char *sf_version(void);

/* ------------------------------------------------------------------------
 * Forward: chunk_gdn.  Attention Gym "Linear Attention", chunk_gdn API entry
 * (inputs, initial_state, cu_seqlens, scale, output_final_state); StateFlow
 * section 3.1, Eq. 4-5 (the output state of a chunk is the next chunk's input
 * state).
 *
 *   initial_state  [N,H,V,K] FP32, or NULL for zeros
 *   out            [B,T,H,V] in the q/k/v dtype (inactive rows untouched)
 *   final_state    [N,H,V,K] FP32; required iff output_final_state != 0
 *
 * Returns SF_ERR_INVALID_ARG for NULL/misaligned pointers or inconsistent
 * shapes (HK not dividing H among them), SF_ERR_UNSUPPORTED for head sizes
 * other than 64/128, K != V or int32 overflow, SF_ERR_WORKSPACE when
 * ws_bytes < sf_gdn_fwd_workspace().
 * ---------------------------------------------------------------------- */
size_t sf_gdn_fwd_workspace(const sf_gdn_shape *shape);
sf_status sf_gdn_chunk_fwd(const sf_gdn_shape *shape, const void *q, const void *k,
                           const void *v, const float *gate, const float *beta,
                           const float *initial_state, const int32_t *cu_seqlens,
                           int output_final_state, void *out, float *final_state,
                           void *workspace, size_t ws_bytes, sf_stream_t stream);

/* ------------------------------------------------------------------------
 * Paged-cache prefill (Attention Gym "Linear Attention", paged_chunk_gdn): the
 * forward, advancing a pool of recurrent states in place.
 *   state_cache    [num_slots,H,V,K] FP32, read and written in place
 *   state_indices  int32 [N] device: sequence n starts from slot
 *                  state_indices[n] and leaves its final state there.  Indices
 *                  must be unique among the positive ones (caller's
 *                  responsibility); an index <= 0 (or >= num_slots) marks
 *                  padding: zero output rows, the cache untouched.
 *   has_initial_state  uint8 [N] device or NULL (all 1): 0 starts the
 *                  sequence from zero without reading the slot, and the slot
 *                  is overwritten (also for an empty sequence)
 *   out            [B,T,H,V]; rows past cu_seqlens[N] untouched
 * Shapes, dtypes, workspace (sf_gdn_fwd_workspace) and errors as
 * sf_gdn_chunk_fwd, whose initial/final state arguments the cache replaces.
 * ---------------------------------------------------------------------- */
sf_status sf_gdn_paged_chunk_fwd(const sf_gdn_shape *shape, const void *q, const void *k,
                                 const void *v, const float *gate, const float *beta,
                                 float *state_cache, int num_slots,
                                 const int32_t *state_indices,
                                 const uint8_t *has_initial_state,
                                 const int32_t *cu_seqlens, void *out, void *workspace,
                                 size_t ws_bytes, sf_stream_t stream);

/* ------------------------------------------------------------------------
 * Segment summary.  Attention Gym "Linear Attention", section "Context
 * Parallelism": every token step is affine in the V-major state, so a token
 * range maps its entry state to S_out = S_in @ P + S_ext; Megatron-LM PR
 * "Mamba2 state-passing context parallelism" uses the scalar special case
 * S_out = a_block * S_in + S_ext.  q is not needed (the map ignores it).
 *
 *   bounds  int32 [R,2] device: (start, stop) flattened token rows
 *           (row = b*T + t); a range must lie inside one batch row and may
 *           be empty (identity map).  It is chunked from its own start.
 *   P       [R,H,K,K] FP32      S_ext  [R,H,V,K] FP32
 * A range that is out of [0, B*T], reversed, or crosses a batch row gets NaN
 * in its P and S_ext (the kernels read nothing outside the inputs).
 * shape->N, shape->scale and cu_seqlens are not used.
 * ---------------------------------------------------------------------- */
size_t sf_gdn_summary_workspace(const sf_gdn_shape *shape, int R);
sf_status sf_gdn_segment_summary(const sf_gdn_shape *shape, const void *k, const void *v,
                                 const float *gate, const float *beta,
                                 const int32_t *bounds, int R, float *P, float *S_ext,
                                 void *workspace, size_t ws_bytes, sf_stream_t stream);

/* ------------------------------------------------------------------------
 * Exclusive scan of segment maps (same section: a prefix scan over the
 * summaries recovers each range's true entry state):
 *     entry_0 = S0,   entry_{j+1} = entry_j @ P_j + S_ext_j,   final = entry_R
 *   P [R,H,K,K], S_ext [R,H,V,K], S0 [H,V,K] or NULL (zeros),
 *   entry_states [R,H,V,K], final_state [H,V,K] or NULL.  All FP32.
 * K == V in {64,128}.  Needs no workspace.
 * ---------------------------------------------------------------------- */
sf_status sf_state_scan(int R, int H, int K, int V, const float *P, const float *S_ext,
                        const float *S0, float *entry_states, float *final_state,
                        sf_stream_t stream);

/* ------------------------------------------------------------------------
 * Reverse segment summary: the backward counterpart of the segment summary
 * (same section: the backward carries the state cotangent from the end of
 * the sequence to its start, and each token's adjoint is affine in it).  For
 * consecutive segments of one token stream, the cotangent at a segment's
 * start is
 *     dS_entry = dS_exit @ P^T + C
 * with P the segment's forward transition (sf_gdn_segment_summary) and C the
 * cotangent its own output gradients produce at its start when nothing flows
 * in at its end.  This entry point computes C.
 *
 *   shape          B = 1 (rows flattened), T = rows, N = R segments,
 *                  HK query/key heads as everywhere
 *   seg_offsets    int32 [R+1] device, the cu_seqlens convention: segment r
 *                  owns rows [seg_offsets[r], seg_offsets[r+1])
 *   q, k [1,T,HK,K]; gate, beta [1,T,H]; d_out [1,T,H,V] (q/k dtype)
 *   C              [R,H,V,K] FP32
 * C depends on neither the values nor the forward states.  Supported: BF16
 * with K = V in {64,128}; F32 with K = V = 64.
 * ---------------------------------------------------------------------- */
size_t sf_gdn_reverse_summary_workspace(const sf_gdn_shape *shape);
sf_status sf_gdn_segment_reverse_summary(const sf_gdn_shape *shape, const void *q,
                                         const void *k, const float *gate, const float *beta,
                                         const void *d_out, const int32_t *seg_offsets,
                                         float *C, void *workspace, size_t ws_bytes,
                                         sf_stream_t stream);

/* ------------------------------------------------------------------------
 * Reverse exclusive scan of the cotangent maps, from the last segment to the
 * first:
 *     exit_{R-1} = dS_final,   exit_{j-1} = exit_j @ P_j^T + C_j,
 *     d_initial  = exit_0 @ P_0^T + C_0
 *   P [R,H,K,K], C [R,H,V,K], dS_final [H,V,K] or NULL (zeros),
 *   exit_cotangents [R,H,V,K] (the cotangent at each segment's end),
 *   d_initial [H,V,K] or NULL.  All FP32.  K == V in {64,128}.  No workspace.
 * With the entry states of sf_state_scan and these exit cotangents, the
 * packed backward over the segments (initial_state = entry states,
 * d_final_state = exit cotangents) gives every gradient of the single pass.
 * ---------------------------------------------------------------------- */
sf_status sf_state_scan_reverse(int R, int H, int K, int V, const float *P, const float *C,
                                const float *dS_final, float *exit_cotangents,
                                float *d_initial, sf_stream_t stream);

/* ------------------------------------------------------------------------
 * Backward of sf_gdn_chunk_fwd (StateFlow section 3.1, Eq. 6-7: the
 * input-state gradient of chunk i+1 is the output-state gradient of chunk i;
 * section 3.4.2, Eq. 18: state replay, output gradient, backward state
 * transition, preparation gradient).  Gradients of
 *     L = <d_out, out> + <d_final_state, final_state>
 * with respect to every input:
 *   d_out          [B,T,H,V] q/k/v dtype (rows past cu_seqlens[N] ignored)
 *   d_final_state  [N,H,V,K] FP32 or NULL (zeros)
 *   dq, dk [B,T,HK,K], dv [B,T,H,V] in the q/k/v dtype; dgate, dbeta [B,T,H]
 *   FP32; d_initial_state [N,H,V,K] FP32 or NULL (not computed).
 * Inactive rows of the gradients are not written.
 * Supported: BF16 with K=V in {64,128}; F32 with K=V=64.
 * ---------------------------------------------------------------------- */
size_t sf_gdn_bwd_workspace(const sf_gdn_shape *shape);
sf_status sf_gdn_chunk_bwd(const sf_gdn_shape *shape, const void *q, const void *k,
                           const void *v, const float *gate, const float *beta,
                           const float *initial_state, const int32_t *cu_seqlens,
                           const void *d_out, const float *d_final_state, void *dq,
                           void *dk, void *dv, float *dgate, float *dbeta,
                           float *d_initial_state, void *workspace, size_t ws_bytes,
                           sf_stream_t stream);

/* ------------------------------------------------------------------------
 * Backward without a workspace.  The pages have no counterpart of this entry
 * point; it exists for callers that cannot allocate device memory where they
 * need gradients -- host runtimes that freeze their allocator after warm-up
 * (a late allocation is refused or breaks their accounting), embedders that
 * own all device memory themselves and hand none to libraries.  Same arguments
 * and results as sf_gdn_chunk_bwd, minus the workspace: the scratch (chunk
 * checkpoints and cotangent tape) is a fixed device array of
 * SF_BWD_NOALLOC_SCRATCH_BYTES built into the library, present on every GPU
 * that loads it until the process exits.  No CUDA, library or other
 * allocating routine is called.
 *  * Limit: shapes whose sf_gdn_bwd_workspace() exceeds
 *    SF_BWD_NOALLOC_SCRATCH_BYTES return SF_ERR_UNSUPPORTED.  For BF16 at
 *    K = V = 128 the scratch is 115,712 bytes per chunk-head (heads x
 *    B x ceil(T/64) dense, heads x (ceil(T/64) + N) packed) and 540,672 bytes
 *    per (sequence, head) pair, up to 64 pairs, for the record ring of the
 *    state replay: one sequence of 2 heads fits up to T = 8896.
 *  * The first call on a device looks up the array's device address for that
 *    device (cudaGetSymbolAddress, with the device current); make that first
 *    call before any stream capture.
 *  * Every call shares the one array: calls whose work overlaps on the GPU
 *    (other streams, other host threads) race on it.  Nothing in it has to
 *    start at zero; each call writes every scratch value before reading it.
 *  * The array's first word is the call's device status word (the workspace
 *    status word of the other entry points): a bounded internal wait that ran
 *    out leaves SF_ERR_TIMEOUT there.  sf_gdn_chunk_bwd_noalloc_status reads
 *    it for the current device, clears it and returns it.
 * ---------------------------------------------------------------------- */
#define SF_BWD_NOALLOC_SCRATCH_BYTES (32ull << 20)
sf_status sf_gdn_chunk_bwd_noalloc(const sf_gdn_shape *shape, const void *q, const void *k,
                                   const void *v, const float *gate, const float *beta,
                                   const float *initial_state, const int32_t *cu_seqlens,
                                   const void *d_out, const float *d_final_state, void *dq,
                                   void *dk, void *dv, float *dgate, float *dbeta,
                                   float *d_initial_state, sf_stream_t stream);

/* Synchronises `stream`, reads the status word of sf_gdn_chunk_bwd_noalloc's
 * built-in scratch on the current device, clears it and returns it (SF_OK when
 * no kernel reported a timeout since the last read).  Like the entry point it
 * allocates nothing; the pages have no counterpart of it either. */
sf_status sf_gdn_chunk_bwd_noalloc_status(sf_stream_t stream);

/* ------------------------------------------------------------------------
 * Helpers (not on the hot path).
 * ---------------------------------------------------------------------- */
/* Synchronous check of device cu_seqlens [N+1]: starts at 0, never decreases,
 * ends at or before T.  Returns SF_OK or SF_ERR_INVALID_ARG (with a message). */
sf_status sf_validate_cu_seqlens(const int32_t *cu_seqlens, int N, int T, sf_stream_t stream);

/* Synchronises `stream`, reads the workspace status word, clears it and returns
 * it (SF_OK when no kernel reported a timeout). */
sf_status sf_workspace_status(void *workspace, sf_stream_t stream);

/* Failure-detection testing only (not for production use; the pages have no
 * counterpart).  The next call on the calling host thread that runs the BF16
 * K = V = 128 tensor-core kernel (forward, paged forward, segment summary or
 * the backward's state replay) never publishes the chunk record with index
 * `record` in the kernel's production order, and every bounded internal wait
 * of that launch gives up after `wait_limit_cycles` SM clock cycles (>= 1e6)
 * instead of about 2 s.  The waiting CTA raises the kernel's abort flag, every
 * CTA leaves after its own copies and products have completed, and the status
 * word reads SF_ERR_TIMEOUT; the call itself still returns SF_OK (the failure
 * is on the device).  Later launches are normal.  One shot; returns
 * SF_ERR_INVALID_ARG for a negative record or a limit below 1e6. */
sf_status sf_testing_inject_timeout(long long record, long long wait_limit_cycles);

#ifdef __cplusplus
}
#endif
#endif /* SF_GDN_H */
