// group_sum.cu -- the backward's last step for grouped query/key heads.
//
// With HK query/key heads over H value heads (value head h reads query/key head
// h / (H / HK); Attention Gym "Linear Attention", chunk_gdn parameter table), the
// gradient of a shared query or key head is the sum of what its block of H / HK value
// heads pushes back into it.  The gradient kernels leave those per-value-head parts in
// FP32 [rows, H, D]; this kernel adds each block in a fixed order (the result does not
// depend on scheduling) and writes [rows, HK, D] in the q/k dtype, active rows only.
#include <cuda_bf16.h>

#include "common.cuh"
#include "simt_chunk.cuh"

namespace sfg {
namespace {

template <typename Tout>
__global__ void __launch_bounds__(256) group_sum_kernel(const float* __restrict__ acc,
                                                        Tout* __restrict__ out, int64_t rows,
                                                        int H, int HK, int D,
                                                        const int32_t* __restrict__ cu, int N) {
  // active rows: [0, cu[N]) for packed sequences (clamped into [0, rows]), else all
  int64_t active = rows;
  if (cu) {
    const int64_t e = cu[N];
    active = e < 0 ? 0 : (e < rows ? e : rows);
  }
  const int G = H / HK, D4 = D / 4;
  const int64_t total = active * HK * D4;           // float4 groups of the output
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int c = (int)(idx % D4) * 4;
    const int64_t rh = idx / D4;
    const int hk = (int)(rh % HK);
    const int64_t r = rh / HK;
    const float* a = acc + ((size_t)r * H + (size_t)hk * G) * D + c;
    float4 s = *reinterpret_cast<const float4*>(a);
    for (int j = 1; j < G; ++j) {
      const float4 x = *reinterpret_cast<const float4*>(a + (size_t)j * D);
      s.x += x.x; s.y += x.y; s.z += x.z; s.w += x.w;
    }
    Tout* o = out + ((size_t)r * HK + hk) * D + c;
    o[0] = from_f<Tout>(s.x);
    o[1] = from_f<Tout>(s.y);
    o[2] = from_f<Tout>(s.z);
    o[3] = from_f<Tout>(s.w);
  }
}

}  // namespace

cudaError_t launch_group_sum(const float* acc, void* out, bool bf16, int64_t rows, int H, int HK,
                             int D, const int32_t* cu, int N, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  if (HK < 1 || H % HK || D % 4) return cudaErrorInvalidValue;
  const int64_t total = rows * HK * (D / 4);
  const int64_t want = (total + 255) / 256;
  const unsigned grid = (unsigned)(want < 152 * 16 ? want : 152 * 16);
  if (bf16)
    group_sum_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(
        acc, reinterpret_cast<__nv_bfloat16*>(out), rows, H, HK, D, cu, N);
  else
    group_sum_kernel<float><<<grid, 256, 0, st>>>(acc, reinterpret_cast<float*>(out), rows, H, HK,
                                                  D, cu, N);
  return cudaGetLastError();
}

}  // namespace sfg
