// api.cu -- the C ABI (include/sf_gdn.h): argument checks, workspace layout and
// kernel dispatch.  No entry point allocates memory or synchronises the host
// (except the two documented synchronous helpers at the end).
#if __has_include(<nvtx3/nvToolsExt.h>)
#include <nvtx3/nvToolsExt.h>
#define SF_HAVE_NVTX 1
#endif

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <string>

#include "../../include/sf_gdn.h"
#include "api_internal.cuh"
#include "common.cuh"
#include "fwd_split.cuh"
#include "tmap.cuh"
#include "scan.cuh"
#include "simt_chunk.cuh"

namespace {

thread_local std::string g_last_error = "no error";

sf_status fail(sf_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

}  // namespace

sf_status sfg::report(sf_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

namespace {

// An NVTX range around each compute entry point, so that timelines (Nsight Systems, ncu's
// range filters) show the library's calls; without a tool attached it does nothing.
// (Without the NVTX headers it compiles to nothing.)
struct Range {
#ifdef SF_HAVE_NVTX
  explicit Range(const char* name) { nvtxRangePushA(name); }
  ~Range() { nvtxRangePop(); }
#else
  explicit Range(const char*) {}
#endif
  Range(const Range&) = delete;
  Range& operator=(const Range&) = delete;
};

sf_status cuda_fail(cudaError_t e, const char* where) {
  return fail(SF_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

constexpr size_t kStatusBytes = 256;

// BF16 with K = V = 128 runs only on the tensor-core kernels, which need TMA descriptors;
// without the driver's encoder that request is unsupported (nothing else serves it).
constexpr const char* kNoTmaEncoder =
    "BF16 with K = V = 128 needs the tensor-core kernels, but the driver entry point "
    "cuTensorMapEncodeTiled is unavailable (or disabled by SF_GDN_DISABLE_TMA_ENCODER)";

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Host-visible checks shared by every token-stream entry point.
sf_status check_shape(const sf_gdn_shape* s, bool packed, bool need_n, const char* fn) {
  if (!s) return fail(SF_ERR_INVALID_ARG, "%s: shape is NULL", fn);
  if (s->B < 1 || s->T < 0 || s->H < 1 || s->K < 1 || s->V < 1)
    return fail(SF_ERR_INVALID_ARG, "%s: need B>=1, T>=0, H>=1, K>=1, V>=1 (got B=%d T=%d H=%d K=%d V=%d)",
                fn, s->B, s->T, s->H, s->K, s->V);
  if (s->dtype != SF_F32 && s->dtype != SF_BF16)
    return fail(SF_ERR_INVALID_ARG, "%s: dtype must be SF_F32 or SF_BF16", fn);
  if (s->HK < 0 || s->H % (s->HK > 0 ? s->HK : s->H))
    return fail(SF_ERR_INVALID_ARG, "%s: query/key heads HK = %d must divide H = %d", fn, s->HK,
                s->H);
  if (s->K != s->V || (s->K != 64 && s->K != 128))
    return fail(SF_ERR_UNSUPPORTED, "%s: head sizes K == V in {64, 128} only (got K=%d V=%d)", fn,
                s->K, s->V);
  const long long elems = (long long)s->B * s->T * s->H * s->K;
  if (elems >= (1LL << 31))
    return fail(SF_ERR_UNSUPPORTED, "%s: tensors need int64 element offsets (%lld elements)", fn,
                elems);
  if (need_n) {
    if (packed) {
      if (s->B != 1) return fail(SF_ERR_INVALID_ARG, "%s: cu_seqlens requires B == 1", fn);
      if (s->N < 1) return fail(SF_ERR_INVALID_ARG, "%s: cu_seqlens requires N >= 1", fn);
    } else if (s->N != s->B) {
      return fail(SF_ERR_INVALID_ARG, "%s: without cu_seqlens N must equal B (N=%d B=%d)", fn,
                  s->N, s->B);
    }
  }
  return SF_OK;
}

int eff_hk(const sf_gdn_shape* s) { return s->HK > 0 ? s->HK : s->H; }

float eff_scale(const sf_gdn_shape* s) {
  return s->scale > 0.f ? s->scale : 1.0f / std::sqrt((float)s->K);
}

int64_t bwd_slots(const sf_gdn_shape* s, bool packed) {
  const int64_t per = (s->T + sfg::CHUNK - 1) / sfg::CHUNK;
  return packed ? per + s->N : (int64_t)s->N * per;
}

size_t round_up(size_t x) { return (x + 255) & ~(size_t)255; }

// Bytes of one chunk-head's entry state (replay checkpoint) or exit cotangent (tape): BF16
// with K = V = 128 keeps them as the BF16 swizzled tiles the tensor-core gradient kernel reads
// (32 KB), the other kernels as FP32 [V,K].
size_t state_tile_bytes(const sf_gdn_shape* s) {
  if (s->dtype == SF_BF16 && s->K == 128 && s->V == 128) return 128 * 128 * 2;
  return (size_t)s->K * s->V * sizeof(float);
}

// Backward workspace: status word | chunk-entry states | exit cotangents ([slots,H] of
// state_tile_bytes each) | BF16 only: per-chunk factors [slots,H] and, for head size 128, the
// split forward's ring (state replay) | grouped heads only: the per-value-head parts of dq
// and dk (FP32 [B,T,H,K] each).
struct BwdLayout {
  size_t one, fac, split, gqa, total;
};

BwdLayout bwd_layout(const sf_gdn_shape* shape) {
  BwdLayout l{0, 0, 0, 0, kStatusBytes};
  if (!shape || shape->K < 1 || shape->H < 1 || shape->T < 0) return l;
  // dense inputs need N * ceil(T/64) slots with N == B; packed ones (B == 1) at most
  // ceil(T/64) + N (every sequence's last chunk may be partial), which also covers the
  // dense B == N == 1
  const int64_t per = (shape->T + sfg::CHUNK - 1) / sfg::CHUNK;
  const int64_t n = shape->N > 0 ? shape->N : shape->B;
  const int64_t slots = shape->B == 1 ? per + n : (int64_t)shape->B * per;
  l.one = round_up((size_t)slots * shape->H * state_tile_bytes(shape));
  if (shape->dtype == SF_BF16 && (shape->K == 64 || shape->K == 128))
    l.fac = round_up((size_t)slots * shape->H * sfg::mma_bwd_fac_bytes(shape->K));
  if (shape->dtype == SF_BF16 && shape->K == 128 && shape->V == 128)
    l.split = sfg::split_fwd_workspace((int)n, shape->H);
  if (shape->HK > 0 && shape->HK < shape->H)
    l.gqa = round_up((size_t)shape->B * shape->T * shape->H * shape->K * sizeof(float));
  l.total = kStatusBytes + 2 * l.one + l.fac + l.split + 2 * l.gqa;
  return l;
}

}  // namespace

extern "C" {

const char* sf_last_error(void) { return g_last_error.c_str(); }

const char* sf_version(void) { return "sf_gdn 0.1 sm_103a"; }

size_t sf_gdn_fwd_workspace(const sf_gdn_shape* shape) {
  // BF16 with K = V = 128 may run on the split forward, which passes chunk records
  // between its CTAs through a ring in the workspace.
  if (shape && shape->dtype == SF_BF16 && shape->K == 128 && shape->V == 128)
    return sfg::split_fwd_workspace(shape->N > 0 ? shape->N : shape->B, shape->H > 0 ? shape->H : 1);
  return kStatusBytes;
}

}  // extern "C"

namespace {

// The forward shared by sf_gdn_chunk_fwd and sf_gdn_paged_chunk_fwd (pool != NULL: the
// entry and final states are slots of the paged cache).
sf_status chunk_fwd(const char* fn, const sf_gdn_shape* shape, const void* q, const void* k,
                    const void* v, const float* gate, const float* beta,
                    const float* initial_state, const int32_t* cu_seqlens, float* final_state,
                    void* out, float* pool, int num_slots, const int32_t* state_indices,
                    const uint8_t* has_initial_state, void* workspace, size_t ws_bytes,
                    sf_stream_t stream) {
  const Range range(fn);
  sf_status st = check_shape(shape, cu_seqlens != nullptr, true, fn);
  if (st != SF_OK) return st;
  if (shape->T > 0 && (!q || !k || !v || !gate || !beta || !out))
    return fail(SF_ERR_INVALID_ARG, "%s: q, k, v, gate, beta and out must be non-NULL", fn);
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return fail(SF_ERR_INVALID_ARG, "%s: q, k, v and out must be 16-byte aligned", fn);
  if (!workspace || ws_bytes < sf_gdn_fwd_workspace(shape))
    return fail(SF_ERR_WORKSPACE, "%s: workspace needs %zu bytes", fn, sf_gdn_fwd_workspace(shape));
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const bool bf16 = shape->dtype == SF_BF16;
  const int D = shape->K;
  sfg::ChainParams p{};
  p.q = q; p.k = k; p.v = v; p.g = gate; p.beta = beta; p.s0 = initial_state;
  p.cu = cu_seqlens; p.out = out; p.final_state = final_state;
  p.pool = pool; p.num_slots = num_slots; p.state_idx = state_indices;
  p.has_init = has_initial_state;
  p.B = shape->B; p.T = shape->T; p.H = shape->H; p.N = shape->N; p.scale = eff_scale(shape);
  p.HK = eff_hk(shape);
  if (bf16 && D == 128 && shape->T > 0 && !sfg::tc_fwd_available())
    return fail(SF_ERR_UNSUPPORTED, "%s: %s", fn, kNoTmaEncoder);
  cudaError_t e;
  if (bf16 && D == 128 && shape->T > 0)
    e = sfg::launch_split_fwd(p, workspace, reinterpret_cast<int*>(workspace), cs);
  else  // (T = 0: no token is read or written, only the states move; any dtype's kernel does)
    e = sfg::launch_simt_chain(p, sfg::MODE_FWD, bf16 && shape->T > 0, D, shape->N, cs);
  if (e != cudaSuccess) return cuda_fail(e, fn);
  return SF_OK;
}

}  // namespace

extern "C" {

sf_status sf_gdn_chunk_fwd(const sf_gdn_shape* shape, const void* q, const void* k, const void* v,
                           const float* gate, const float* beta, const float* initial_state,
                           const int32_t* cu_seqlens, int output_final_state, void* out,
                           float* final_state, void* workspace, size_t ws_bytes,
                           sf_stream_t stream) {
  const char* fn = "sf_gdn_chunk_fwd";
  if (output_final_state && !final_state)
    return fail(SF_ERR_INVALID_ARG, "%s: output_final_state requires final_state", fn);
  return chunk_fwd(fn, shape, q, k, v, gate, beta, initial_state, cu_seqlens,
                   output_final_state ? final_state : nullptr, out, nullptr, 0, nullptr, nullptr,
                   workspace, ws_bytes, stream);
}

sf_status sf_gdn_paged_chunk_fwd(const sf_gdn_shape* shape, const void* q, const void* k,
                                 const void* v, const float* gate, const float* beta,
                                 float* state_cache, int num_slots, const int32_t* state_indices,
                                 const uint8_t* has_initial_state, const int32_t* cu_seqlens,
                                 void* out, void* workspace, size_t ws_bytes, sf_stream_t stream) {
  const char* fn = "sf_gdn_paged_chunk_fwd";
  if (!state_cache || !state_indices || num_slots < 1)
    return fail(SF_ERR_INVALID_ARG, "%s: state_cache, state_indices and num_slots >= 1 needed", fn);
  if (!aligned16(state_cache))
    return fail(SF_ERR_INVALID_ARG, "%s: state_cache must be 16-byte aligned", fn);
  return chunk_fwd(fn, shape, q, k, v, gate, beta, nullptr, cu_seqlens, nullptr, out, state_cache,
                   num_slots, state_indices, has_initial_state, workspace, ws_bytes, stream);
}

size_t sf_gdn_summary_workspace(const sf_gdn_shape* shape, int R) {
  // BF16 with K = V = 128 runs on the split kernel (records pass through a ring)
  if (shape && shape->dtype == SF_BF16 && shape->K == 128 && shape->V == 128 && R > 0)
    return sfg::split_summary_workspace(R, shape->H > 0 ? shape->H : 1);
  return kStatusBytes;
}

sf_status sf_gdn_segment_summary(const sf_gdn_shape* shape, const void* k, const void* v,
                                 const float* gate, const float* beta, const int32_t* bounds,
                                 int R, float* P, float* S_ext, void* workspace, size_t ws_bytes,
                                 sf_stream_t stream) {
  const char* fn = "sf_gdn_segment_summary";
  const Range range(fn);
  sf_status st = check_shape(shape, false, false, fn);
  if (st != SF_OK) return st;
  if (R < 0) return fail(SF_ERR_INVALID_ARG, "%s: R must be >= 0", fn);
  if (R == 0) return SF_OK;
  if (shape->T < 1) return fail(SF_ERR_INVALID_ARG, "%s: T must be >= 1", fn);
  if (!k || !v || !gate || !beta || !bounds || !P || !S_ext)
    return fail(SF_ERR_INVALID_ARG, "%s: k, v, gate, beta, bounds, P, S_ext must be non-NULL", fn);
  if (!aligned16(k) || !aligned16(v))
    return fail(SF_ERR_INVALID_ARG, "%s: k and v must be 16-byte aligned", fn);
  if (!workspace || ws_bytes < sf_gdn_summary_workspace(shape, R))
    return fail(SF_ERR_WORKSPACE, "%s: workspace needs %zu bytes", fn,
                sf_gdn_summary_workspace(shape, R));
  sfg::ChainParams p{};
  p.k = k; p.v = v; p.g = gate; p.beta = beta; p.bounds = bounds; p.P = P; p.E = S_ext;
  p.B = shape->B; p.T = shape->T; p.H = shape->H; p.N = R; p.scale = 1.f;
  p.HK = eff_hk(shape);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const bool bf16 = shape->dtype == SF_BF16;
  if (bf16 && shape->K == 128 && !sfg::tc_fwd_available())
    return fail(SF_ERR_UNSUPPORTED, "%s: %s", fn, kNoTmaEncoder);
  cudaError_t e;
  if (bf16 && shape->K == 128)
    e = sfg::launch_split_summary(p, workspace, reinterpret_cast<int*>(workspace), cs);
  else
    e = sfg::launch_simt_chain(p, sfg::MODE_SUMMARY, bf16, shape->K, R, cs);
  if (e != cudaSuccess) return cuda_fail(e, fn);
  return SF_OK;
}

sf_status sf_state_scan(int R, int H, int K, int V, const float* P, const float* S_ext,
                        const float* S0, float* entry_states, float* final_state,
                        sf_stream_t stream) {
  const char* fn = "sf_state_scan";
  const Range range(fn);
  if (R < 0 || H < 1) return fail(SF_ERR_INVALID_ARG, "%s: need R>=0 and H>=1", fn);
  if (K != V || (K != 64 && K != 128))
    return fail(SF_ERR_UNSUPPORTED, "%s: K == V in {64, 128} only", fn);
  if (R > 0 && (!P || !S_ext || !entry_states))
    return fail(SF_ERR_INVALID_ARG, "%s: P, S_ext and entry_states must be non-NULL", fn);
  if (R == 0 && !final_state) return SF_OK;
  cudaError_t e = sfg::launch_state_scan(R, H, K, P, S_ext, S0, entry_states, final_state,
                                         reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, fn);
  return SF_OK;
}

size_t sf_gdn_bwd_workspace(const sf_gdn_shape* shape) { return bwd_layout(shape).total; }

// Reverse summary workspace: status word | exit cotangents of every chunk (the reverse
// chain's tape, [slots,H] of state_tile_bytes) | BF16 only: per-chunk factors [slots,H].
// Slots as the packed backward: ceil(T/64) + R.
struct RevLayout {
  size_t tape, fac, total;
};

RevLayout rev_layout(const sf_gdn_shape* shape) {
  RevLayout l{0, 0, kStatusBytes};
  if (!shape || shape->K < 1 || shape->H < 1 || shape->T < 0 || shape->N < 0) return l;
  const int64_t slots = (shape->T + sfg::CHUNK - 1) / sfg::CHUNK + shape->N;
  l.tape = round_up((size_t)slots * shape->H * state_tile_bytes(shape));
  if (shape->dtype == SF_BF16 && (shape->K == 64 || shape->K == 128))
    l.fac = round_up((size_t)slots * shape->H * sfg::mma_bwd_fac_bytes(shape->K));
  l.total = kStatusBytes + l.tape + l.fac;
  return l;
}

size_t sf_gdn_reverse_summary_workspace(const sf_gdn_shape* shape) {
  return rev_layout(shape).total;
}

sf_status sf_gdn_segment_reverse_summary(const sf_gdn_shape* shape, const void* q, const void* k,
                                         const float* gate, const float* beta, const void* d_out,
                                         const int32_t* seg_offsets, float* C, void* workspace,
                                         size_t ws_bytes, sf_stream_t stream) {
  const char* fn = "sf_gdn_segment_reverse_summary";
  const Range range(fn);
  sf_status st = check_shape(shape, true, true, fn);
  if (st != SF_OK) return st;
  const bool bf16 = shape->dtype == SF_BF16;
  const int D = shape->K;
  if (!bf16 && D != 64)
    return fail(SF_ERR_UNSUPPORTED, "%s: FP32 inputs support K = V = 64 only", fn);
  if (!seg_offsets || !C)
    return fail(SF_ERR_INVALID_ARG, "%s: seg_offsets and C must be non-NULL", fn);
  if (shape->T > 0 && (!q || !k || !gate || !beta || !d_out))
    return fail(SF_ERR_INVALID_ARG, "%s: q, k, gate, beta and d_out must be non-NULL", fn);
  const RevLayout lay = rev_layout(shape);
  if (!workspace || ws_bytes < lay.total)
    return fail(SF_ERR_WORKSPACE, "%s: workspace needs %zu bytes", fn, lay.total);
  char* ws = reinterpret_cast<char*>(workspace);
  sfg::ChainParams p{};
  p.q = q; p.k = k; p.g = gate; p.beta = beta; p.cu = seg_offsets; p.dout = d_out;
  p.dsf = nullptr;        // nothing flows in at a segment's end
  p.ds0 = C;              // the cotangent the chain leaves at the segment's start
  p.tape = reinterpret_cast<float*>(ws + kStatusBytes);
  p.fac = lay.fac ? reinterpret_cast<float*>(ws + kStatusBytes + lay.tape) : nullptr;
  p.status = reinterpret_cast<int*>(workspace);
  p.B = shape->B; p.T = shape->T; p.H = shape->H; p.N = shape->N; p.scale = eff_scale(shape);
  p.HK = eff_hk(shape);
  const int64_t slots = bwd_slots(shape, true);
  cudaError_t e = sfg::launch_simt_bwd(p, bf16, D, slots, reinterpret_cast<cudaStream_t>(stream),
                                       /*chain_only=*/true);
  if (e != cudaSuccess) return cuda_fail(e, fn);
  return SF_OK;
}

sf_status sf_state_scan_reverse(int R, int H, int K, int V, const float* P, const float* C,
                                const float* dS_final, float* exit_cotangents, float* d_initial,
                                sf_stream_t stream) {
  const char* fn = "sf_state_scan_reverse";
  const Range range(fn);
  if (R < 0 || H < 1) return fail(SF_ERR_INVALID_ARG, "%s: need R>=0 and H>=1", fn);
  if (K != V || (K != 64 && K != 128))
    return fail(SF_ERR_UNSUPPORTED, "%s: K == V in {64, 128} only", fn);
  if (R > 0 && (!P || !C || !exit_cotangents))
    return fail(SF_ERR_INVALID_ARG, "%s: P, C and exit_cotangents must be non-NULL", fn);
  if (R == 0 && !d_initial) return SF_OK;
  cudaError_t e = sfg::launch_state_scan_reverse(R, H, K, P, C, dS_final, exit_cotangents,
                                                 d_initial, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, fn);
  return SF_OK;
}

sf_status sf_gdn_chunk_bwd(const sf_gdn_shape* shape, const void* q, const void* k, const void* v,
                           const float* gate, const float* beta, const float* initial_state,
                           const int32_t* cu_seqlens, const void* d_out, const float* d_final_state,
                           void* dq, void* dk, void* dv, float* dgate, float* dbeta,
                           float* d_initial_state, void* workspace, size_t ws_bytes,
                           sf_stream_t stream) {
  const char* fn = "sf_gdn_chunk_bwd";
  const Range range(fn);
  const bool packed = cu_seqlens != nullptr;
  sf_status st = check_shape(shape, packed, true, fn);
  if (st != SF_OK) return st;
  const bool bf16 = shape->dtype == SF_BF16;
  const int D = shape->K;
  if (!bf16 && D != 64)
    return fail(SF_ERR_UNSUPPORTED, "%s: FP32 inputs support K = V = 64 only", fn);
  if (shape->T > 0 && (!q || !k || !v || !gate || !beta || !d_out || !dq || !dk || !dv || !dgate ||
                       !dbeta))
    return fail(SF_ERR_INVALID_ARG, "%s: inputs and gradient outputs must be non-NULL", fn);
  const size_t need = sf_gdn_bwd_workspace(shape);
  if (!workspace || ws_bytes < need)
    return fail(SF_ERR_WORKSPACE, "%s: workspace needs %zu bytes", fn, need);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const int64_t slots = bwd_slots(shape, packed);
  const BwdLayout lay = bwd_layout(shape);
  const size_t one = lay.one;
  char* ws = reinterpret_cast<char*>(workspace);
  sfg::ChainParams p{};
  p.q = q; p.k = k; p.v = v; p.g = gate; p.beta = beta; p.s0 = initial_state; p.cu = cu_seqlens;
  p.ckpt = reinterpret_cast<float*>(ws + kStatusBytes);
  p.tape = reinterpret_cast<float*>(ws + kStatusBytes + one);
  p.dout = d_out; p.dsf = d_final_state; p.dq = dq; p.dk = dk; p.dv = dv; p.dg = dgate;
  p.dbeta = dbeta; p.ds0 = d_initial_state;
  p.status = reinterpret_cast<int*>(workspace);
  p.fac = lay.fac ? reinterpret_cast<float*>(ws + kStatusBytes + 2 * one) : nullptr;
  p.B = shape->B; p.T = shape->T; p.H = shape->H; p.N = shape->N; p.scale = eff_scale(shape);
  p.HK = eff_hk(shape);
  // grouped heads: the gradient kernels write per-value-head FP32 parts, summed below
  float* gq = nullptr;
  float* gk = nullptr;
  if (lay.gqa) {
    gq = reinterpret_cast<float*>(ws + kStatusBytes + 2 * one + lay.fac + lay.split);
    gk = reinterpret_cast<float*>(reinterpret_cast<char*>(gq) + lay.gqa);
    p.dq = gq;
    p.dk = gk;
    p.dqk_f32 = 1;
  }
  if (bf16 && D == 128 && shape->T > 0 && !sfg::tc_fwd_available())
    return fail(SF_ERR_UNSUPPORTED, "%s: %s", fn, kNoTmaEncoder);
  cudaError_t e;
  if (bf16 && D == 128 && shape->T > 0) {
    char* split = ws + kStatusBytes + 2 * one + lay.fac;
    e = sfg::launch_split_fwd(p, split, reinterpret_cast<int*>(workspace), cs);
    p.fac_ready = 1;    // the replay kept every chunk's record in p.fac
    // the replay's ring is free once it has run: the fused backward's tape counts
    if (!packed && lay.split >= ((size_t)shape->N * shape->H + 1) * 128)
      p.sync = reinterpret_cast<uint32_t*>(split);
  } else if (shape->T > 0) {
    e = sfg::launch_simt_chain(p, sfg::MODE_REPLAY, bf16, D, shape->N, cs);
  } else {
    e = cudaSuccess;   // no chunk: nothing to replay
  }
  if (e != cudaSuccess) return cuda_fail(e, fn);
  e = sfg::launch_simt_bwd(p, bf16, D, slots, cs);
  if (e != cudaSuccess) return cuda_fail(e, fn);
  if (lay.gqa) {
    const int64_t rows = (int64_t)shape->B * shape->T;
    e = sfg::launch_group_sum(gq, dq, bf16, rows, shape->H, p.HK, D, cu_seqlens, shape->N, cs);
    if (e == cudaSuccess)
      e = sfg::launch_group_sum(gk, dk, bf16, rows, shape->H, p.HK, D, cu_seqlens, shape->N, cs);
    if (e != cudaSuccess) return cuda_fail(e, fn);
  }
  return SF_OK;
}

sf_status sf_validate_cu_seqlens(const int32_t* cu_seqlens, int N, int T, sf_stream_t stream) {
  const char* fn = "sf_validate_cu_seqlens";
  if (!cu_seqlens || N < 1 || T < 0) return fail(SF_ERR_INVALID_ARG, "%s: bad arguments", fn);
  std::string host((size_t)(N + 1) * sizeof(int32_t), '\0');
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(&host[0], cu_seqlens, host.size(), cudaMemcpyDeviceToHost, cs);
  if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
  if (e != cudaSuccess) return cuda_fail(e, fn);
  const int32_t* c = reinterpret_cast<const int32_t*>(host.data());
  if (c[0] != 0) return fail(SF_ERR_INVALID_ARG, "%s: cu_seqlens[0] = %d, expected 0", fn, c[0]);
  for (int i = 0; i < N; ++i)
    if (c[i + 1] < c[i])
      return fail(SF_ERR_INVALID_ARG, "%s: cu_seqlens decreases at %d (%d -> %d)", fn, i, c[i],
                  c[i + 1]);
  if (c[N] > T) return fail(SF_ERR_INVALID_ARG, "%s: cu_seqlens[N] = %d exceeds T = %d", fn, c[N], T);
  return SF_OK;
}

sf_status sf_testing_inject_timeout(long long record, long long wait_limit_cycles) {
  if (record < 0 || wait_limit_cycles < 1000000)
    return fail(SF_ERR_INVALID_ARG,
                "sf_testing_inject_timeout: need record >= 0 and wait_limit_cycles >= 1e6");
  sfg::inject_split_timeout(record, wait_limit_cycles);
  return SF_OK;
}

sf_status sf_workspace_status(void* workspace, sf_stream_t stream) {
  const char* fn = "sf_workspace_status";
  if (!workspace) return fail(SF_ERR_INVALID_ARG, "%s: workspace is NULL", fn);
  int word = 0;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(&word, workspace, sizeof(int), cudaMemcpyDeviceToHost, cs);
  if (e == cudaSuccess) e = cudaMemsetAsync(workspace, 0, sizeof(int), cs);
  if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
  if (e != cudaSuccess) return cuda_fail(e, fn);
  if (word != 0) return fail((sf_status)word, "%s: a kernel reported status %d", fn, word);
  return SF_OK;
}

}  // extern "C"
