// tmap.cu -- TMA tensor maps of the BF16 token-major tensors, encoded through the driver
// entry point that the runtime hands out (no link-time dependency on libcuda).
#include <cudaTypedefs.h>

#include <cstdlib>
#include <mutex>

#include "tmap.cuh"

namespace sfg {
namespace {

constexpr int D = 128;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    // A host-side switch to report the encoder as absent, so that the status a caller gets
    // without it (SF_ERR_UNSUPPORTED, nothing launched) can be checked on any machine.
    const char* off = std::getenv("SF_GDN_DISABLE_TMA_ENCODER");
    if (off && off[0] && off[0] != '0') return;
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

}  // namespace

bool tc_fwd_available() { return encode_fn() != nullptr; }

bool make_bf16_map(CUtensorMap* m, const void* base, int rows, int H) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
  cuuint32_t box[3] = {64, 1, 64};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_bf16_map_4d(CUtensorMap* m, const void* base, int rows, int H) {
  auto enc = encode_fn();
  if (!enc) return false;
  // (64 columns, rows, 2 column panels, heads): the panel dimension sits between the rows
  // and the heads in memory, so one box of 64 x 64 x 2 x 1 lands as two 64-row panels
  cuuint64_t dims[4] = {64, (cuuint64_t)rows, 2, (cuuint64_t)H};
  cuuint64_t strides[3] = {(cuuint64_t)H * D * 2, 128, (cuuint64_t)D * 2};
  cuuint32_t box[4] = {64, 64, 2, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace sfg
