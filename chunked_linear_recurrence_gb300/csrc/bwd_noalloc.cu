// bwd_noalloc.cu -- the backward without a caller workspace.
//
// sf_gdn_chunk_bwd needs scratch (the chunk-entry state checkpoints and the
// state-cotangent tape) that the caller allocates.  Some callers cannot
// allocate at the point where they need gradients: host runtimes whose
// allocator is frozen after warm-up (a new device allocation there would be
// refused or would break their memory accounting), and embedders that own
// every byte of device memory and have no allocator to hand to a library.
// This entry point serves them: its scratch is a fixed array compiled into the
// library (SF_BWD_NOALLOC_SCRATCH_BYTES on every GPU that loads it, held until
// the process exits), and it calls no allocating routine of CUDA, of the
// library or of anyone else.
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/sf_gdn.h"
#include "api_internal.cuh"

namespace {

// Device-side scratch shared by every call of sf_gdn_chunk_bwd_noalloc.
static __device__ __align__(256) unsigned char g_bwd_scratch[SF_BWD_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_bwd_scratch on the current device.  In host code the
// symbol is only a host-side stand-in, so the address is looked up once per
// device (with that device current) and cached.
cudaError_t scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_bwd_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" sf_status sf_gdn_chunk_bwd_noalloc(
    const sf_gdn_shape* shape, const void* q, const void* k, const void* v, const float* gate,
    const float* beta, const float* initial_state, const int32_t* cu_seqlens, const void* d_out,
    const float* d_final_state, void* dq, void* dk, void* dv, float* dgate, float* dbeta,
    float* d_initial_state, sf_stream_t stream) {
  if (!shape) return sfg::report(SF_ERR_INVALID_ARG, "sf_gdn_chunk_bwd_noalloc: shape is NULL");
  const size_t need = sf_gdn_bwd_workspace(shape);
  if (need > (size_t)SF_BWD_NOALLOC_SCRATCH_BYTES)
    return sfg::report(SF_ERR_UNSUPPORTED,
                       "sf_gdn_chunk_bwd_noalloc: this shape needs %zu bytes of scratch, more than "
                       "the %llu of the built-in array; call sf_gdn_chunk_bwd with a workspace",
                       need, (unsigned long long)SF_BWD_NOALLOC_SCRATCH_BYTES);
  void* scratch = nullptr;
  const cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess)
    return sfg::report(SF_ERR_CUDA, "sf_gdn_chunk_bwd_noalloc: scratch address: %s",
                       cudaGetErrorString(e));
  // The checkpoints and the tape are written before they are read within one
  // call, so nothing in the array has to start at zero.
  return sf_gdn_chunk_bwd(shape, q, k, v, gate, beta, initial_state, cu_seqlens, d_out,
                          d_final_state, dq, dk, dv, dgate, dbeta, d_initial_state, scratch,
                          (size_t)SF_BWD_NOALLOC_SCRATCH_BYTES, stream);
}

// The array's first word is the status word of the kernels that ran on it (a bounded wait
// that ran out writes SF_ERR_TIMEOUT there).  Read it back on `stream` and clear it.
extern "C" sf_status sf_gdn_chunk_bwd_noalloc_status(sf_stream_t stream) {
  const char* fn = "sf_gdn_chunk_bwd_noalloc_status";
  void* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess)
    return sfg::report(SF_ERR_CUDA, "%s: scratch address: %s", fn, cudaGetErrorString(e));
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  int word = 0;
  e = cudaMemcpyAsync(&word, scratch, sizeof(int), cudaMemcpyDeviceToHost, cs);
  if (e == cudaSuccess) e = cudaMemsetAsync(scratch, 0, sizeof(int), cs);
  if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
  if (e != cudaSuccess) return sfg::report(SF_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(e));
  if (word != 0) return sfg::report((sf_status)word, "%s: a kernel reported status %d", fn, word);
  return SF_OK;
}
