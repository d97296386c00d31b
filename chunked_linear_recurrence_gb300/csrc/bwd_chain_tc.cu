// bwd_chain_tc.cu -- the backward's reverse state-cotangent chain for BF16 inputs with
// K = V = 128 on tcgen05 (the body is chain_tc.cuh), and the kernel that adds Qg to the
// chunk records the state replay kept.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>

#include "bwd_chain_tc.cuh"
#include "chain_tc.cuh"
#include "tmap.cuh"

namespace sfg {
namespace {

using namespace chaintc;

// Qg = scale diag(e^gamma) Q of every chunk-head into its record (gamma: the in-chunk
// cumulative gate; rows past the sequence end zero).  One CTA of 256 threads per (slot, head),
// slots walked with a grid stride until the first empty one; thread t takes row t / 4 and
// columns [32 (t mod 4), + 32).
__global__ void __launch_bounds__(256) qg_kernel(const ChainParams p, uint8_t* fac, int64_t slots) {
  __shared__ float se[64];
  const int tid = threadIdx.x, lane = tid & 31, h = blockIdx.y, H = p.H;
  const int hk = qk_head(h, H, p.HK);
  const __nv_bfloat16* q = reinterpret_cast<const __nv_bfloat16*>(p.q);
  for (int64_t slot = blockIdx.x; slot < slots; slot += gridDim.x) {
    int n = -1;
    int64_t bos = 0, eos = 0, ci = 0;
    if (!locate_chunk(slot, p.B, p.T, p.cu, p.N, n, bos, eos, ci)) break;
    const int64_t c0 = bos + ci * CHUNK;
    const int L = (int)((eos - c0) < CHUNK ? (eos - c0) : CHUNK);
    if (tid < 32) {
      const int e0 = 2 * lane, e1 = e0 + 1;
      const float g0 = e0 < L ? p.g[(size_t)(c0 + e0) * H + h] : 0.f;
      const float g1 = e1 < L ? p.g[(size_t)(c0 + e1) * H + h] : 0.f;
      float sum = g0 + g1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float t = __shfl_up_sync(0xffffffffu, sum, o);
        if (lane >= o) sum += t;
      }
      const float excl = sum - (g0 + g1);
      se[e0] = p.scale * expf(excl + g0);
      se[e1] = p.scale * expf(excl + g0 + g1);
    }
    __syncthreads();
    const int i = tid >> 2, c = 32 * (tid & 3);
    uint8_t* tile = fac + ((size_t)slot * H + h) * REC2_BYTES + R_QG;
    const float f = se[i];
    const uint4* src = reinterpret_cast<const uint4*>(q + ((size_t)(c0 + i) * p.HK + hk) * D + c);
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
      const uint4 v4 = i < L ? src[cc] : make_uint4(0, 0, 0, 0);
      const uint32_t va[4] = {v4.x, v4.y, v4.z, v4.w};
      float x[8];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 fv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&va[e]));
        x[2 * e] = f * fv.x;
        x[2 * e + 1] = f * fv.y;
      }
      st_row8_bf16(tile, i, c + 8 * cc, PANEL, x);
    }
    __syncthreads();   // se is rewritten by the next chunk
  }
}

__global__ void __launch_bounds__(NT, 1)
    tc_bwd_chain_kernel(const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mdo,
                        const ChainParams p, const float* fac) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  chain_cta<false>(&mk, &mdo, p, fac, (int)blockIdx.x, nullptr, sm);
}

}  // namespace

cudaError_t launch_tc_bwd_qg(const ChainParams& p, float* fac, int64_t slots, cudaStream_t st) {
  if (slots <= 0 || (int64_t)p.B * p.T == 0) return cudaSuccess;
  qg_kernel<<<dim3((unsigned)slot_grid(p, slots), p.H), 256, 0, st>>>(
      p, reinterpret_cast<uint8_t*>(fac), slots);
  return cudaGetLastError();
}

cudaError_t launch_tc_bwd_chain(const ChainParams& p, const float* fac, cudaStream_t st) {
  const int chains = p.N * p.H;
  if (chains <= 0) return cudaSuccess;
  CUtensorMap mk, mdo;
  const int rows = p.B * p.T;
  if (rows > 0) {
    if (!make_bf16_map(&mk, p.k, rows, p.HK) || !make_bf16_map(&mdo, p.dout, rows, p.H))
      return cudaErrorInvalidValue;
  } else {
    memset(&mk, 0, sizeof(mk));   // no chunk: the maps are never used
    memset(&mdo, 0, sizeof(mdo));
  }
  auto kern = tc_bwd_chain_kernel;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  kern<<<chains, NT, SMEM_ALLOC, st>>>(mk, mdo, p, fac);
  return cudaGetLastError();
}

}  // namespace sfg
