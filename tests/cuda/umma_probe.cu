// umma_probe.cu -- test-only: one tcgen05.mma sequence D = A * B (M = 128) with
// the operand layouts and descriptor builders the library's tensor-core kernels
// use, so that each layout can be checked against a host matmul.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../chunked_linear_recurrence_gb300/csrc/tc_ptx.cuh"

using namespace sfg::tc;

__global__ void probe_kernel(int N, int K, int a_mn, int b_mn, int neg,
                             const __nv_bfloat16* __restrict__ A,   // [128][K] row-major
                             const __nv_bfloat16* __restrict__ B,   // [K][N] row-major
                             float* __restrict__ Dout) {            // [128][N]
  extern __shared__ uint8_t raw[];
  uint8_t* sm = raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
  const int M = 128;
  const uint32_t a_ps = a_mn ? K * 128 : M * 128;     // panel stride of the A tile
  const uint32_t b_ps = b_mn ? K * 128 : N * 128;
  uint8_t* ta = sm;
  uint8_t* tb = sm + 2 * 32768;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + 4 * 32768);
  uint32_t* slot = reinterpret_cast<uint32_t*>(bar + 1);
  const int tid = threadIdx.x;
  // stage A: K-major tile [m][k]; MN-major tile [k][m]
  for (int idx = tid; idx < M * K / 8; idx += blockDim.x) {
    int r, c;
    float x[8];
    if (!a_mn) { r = idx / (K / 8); c = (idx % (K / 8)) * 8;
      for (int e = 0; e < 8; ++e) x[e] = __bfloat162float(A[r * K + c + e]); }
    else { r = idx / (M / 8); c = (idx % (M / 8)) * 8;      // r = k, c = m
      for (int e = 0; e < 8; ++e) x[e] = __bfloat162float(A[(c + e) * K + r]); }
    st_row8_bf16(ta, r, c, a_ps, x);
  }
  for (int idx = tid; idx < N * K / 8; idx += blockDim.x) {
    int r, c;
    float x[8];
    if (!b_mn) { r = idx / (K / 8); c = (idx % (K / 8)) * 8;  // r = n, c = k
      for (int e = 0; e < 8; ++e) x[e] = __bfloat162float(B[(c + e) * N + r]); }
    else { r = idx / (N / 8); c = (idx % (N / 8)) * 8;        // r = k, c = n
      for (int e = 0; e < 8; ++e) x[e] = __bfloat162float(B[r * N + c + e]); }
    st_row8_bf16(tb, r, c, b_ps, x);
  }
  if (tid == 0) { mbar_init(bar, 1); fence_mbar_init(); }
  if (tid < 32) { tmem_alloc(slot, 256); tmem_relinquish(); }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *slot;
  if (tid == 0) {
    const uint32_t id = idesc_bf16(M, N, a_mn, b_mn, neg);
    for (int kk = 0; kk < K / 16; ++kk) {
      const int k = kk * 16;
      const uint32_t aa = smem_u32(ta) + (a_mn ? k * 128 : (k >> 6) * a_ps + (k & 63) * 2);
      const uint32_t bb = smem_u32(tb) + (b_mn ? k * 128 : (k >> 6) * b_ps + (k & 63) * 2);
      mma_bf16(tm, sdesc_sw128(aa, a_mn ? a_ps : 0, 1024), sdesc_sw128(bb, b_mn ? b_ps : 0, 1024),
               id, kk > 0);
    }
    mma_commit(bar);
  }
  const bool ok = mbar_wait(bar, 0);
  tc_fence_after();
  const int w = tid >> 5, lane = tid & 31, row = w * 32 + lane;
  if (ok) {
    for (int c0 = 0; c0 < N; c0 += 32) {
      float x[32];
      tmem_ld32(tm + ((uint32_t)(w * 32) << 16) + c0, x);
      tmem_ld_wait();
      for (int e = 0; e < 32; ++e) Dout[row * N + c0 + e] = x[e];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (tid < 32) { tc_fence_after(); tmem_dealloc(tm, 256); }
}

extern "C" int umma_probe(int N, int K, int a_mn, int b_mn, int neg, const void* A, const void* B,
                          float* D) {
  if ((N != 64 && N != 128) || (K != 64 && K != 128)) return -1;
  const int smem = 4 * 32768 + 64 + 1024;
  cudaFuncSetAttribute(probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  probe_kernel<<<1, 128, smem>>>(N, K, a_mn, b_mn, neg, (const __nv_bfloat16*)A,
                                 (const __nv_bfloat16*)B, D);
  return (int)cudaDeviceSynchronize();
}

// ---- the tensor-core kernels' 64x64 unit-lower-triangular inverse
#include "../../chunked_linear_recurrence_gb300/csrc/solve_tc.cuh"

struct ProbeBar {
  __device__ __forceinline__ void operator()() const { __syncthreads(); }
};

__global__ void solve_probe_kernel(const float* __restrict__ A, float* __restrict__ T) {
  __shared__ float sA[64 * sfg::SOLVE_LD], sT[64 * sfg::SOLVE_LD], sX[32 * sfg::SOLVE_LD];
  for (int i = threadIdx.x; i < 64 * 64; i += blockDim.x)
    sA[(i >> 6) * sfg::SOLVE_LD + (i & 63)] = A[i];
  __syncthreads();
  sfg::solve64_tc(sA, sT, sX, threadIdx.x, blockDim.x, ProbeBar());
  for (int i = threadIdx.x; i < 64 * 64; i += blockDim.x) T[i] = sT[(i >> 6) * sfg::SOLVE_LD + (i & 63)];
}

__global__ void solve_inplace_probe_kernel(const float* __restrict__ A, float* __restrict__ T) {
  __shared__ float sAT[64 * sfg::SOLVE_LD], sX[32 * sfg::SOLVE_LD];
  for (int i = threadIdx.x; i < 64 * 64; i += blockDim.x)
    sAT[(i >> 6) * sfg::SOLVE_LD + (i & 63)] = A[i];
  __syncthreads();
  sfg::solve64_tc_inplace(sAT, sX, threadIdx.x, blockDim.x, ProbeBar());
  for (int i = threadIdx.x; i < 64 * 64; i += blockDim.x) T[i] = sAT[(i >> 6) * sfg::SOLVE_LD + (i & 63)];
}

extern "C" int solve_probe(const float* A, float* T, int nthreads, int inplace) {
  if (inplace)
    solve_inplace_probe_kernel<<<1, nthreads>>>(A, T);
  else
    solve_probe_kernel<<<1, nthreads>>>(A, T);
  return (int)cudaDeviceSynchronize();
}

// ---- A operand from TMEM (BF16 pairs packed per 32-bit column), B from shared memory
__global__ void probe_ta_kernel(int N, int K, int b_mn, int neg, const __nv_bfloat16* __restrict__ A,
                                const __nv_bfloat16* __restrict__ B, float* __restrict__ Dout) {
  extern __shared__ uint8_t raw[];
  uint8_t* sm = raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
  const uint32_t b_ps = b_mn ? K * 128 : N * 128;
  uint8_t* tb = sm;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + 2 * 32768);
  uint32_t* slot = reinterpret_cast<uint32_t*>(bar + 1);
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31, row = w * 32 + lane;
  for (int idx = tid; idx < N * K / 8; idx += blockDim.x) {
    int r, c;
    float x[8];
    if (!b_mn) { r = idx / (K / 8); c = (idx % (K / 8)) * 8;
      for (int e = 0; e < 8; ++e) x[e] = __bfloat162float(B[(c + e) * N + r]); }
    else { r = idx / (N / 8); c = (idx % (N / 8)) * 8;
      for (int e = 0; e < 8; ++e) x[e] = __bfloat162float(B[r * N + c + e]); }
    st_row8_bf16(tb, r, c, b_ps, x);
  }
  if (tid == 0) { mbar_init(bar, 1); fence_mbar_init(); }
  if (tid < 32) { tmem_alloc(slot, 512); tmem_relinquish(); }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *slot;
  const uint32_t lanes = (uint32_t)(w * 32) << 16;
  for (int c0 = 0; c0 < K / 2; c0 += 16) {          // row `row` of A -> columns 256 + c
    uint32_t u[16];
    for (int e = 0; e < 16; ++e)
      u[e] = pack_bf16x2(__bfloat162float(A[row * K + 2 * (c0 + e)]),
                         __bfloat162float(A[row * K + 2 * (c0 + e) + 1]));
    tmem_st16(tm + lanes + 256 + c0, u);
  }
  tmem_st_wait();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0) {
    const uint32_t id = idesc_bf16(128, N, false, b_mn, neg);
    for (int kk = 0; kk < K / 16; ++kk) {
      const int k = kk * 16;
      const uint32_t bb = smem_u32(tb) + (b_mn ? k * 128 : (k >> 6) * b_ps + (k & 63) * 2);
      mma_bf16_ta(tm, tm + 256 + kk * 8, sdesc_sw128(bb, b_mn ? b_ps : 0, 1024), id, kk > 0);
    }
    mma_commit(bar);
  }
  const bool ok = mbar_wait(bar, 0);
  tc_fence_after();
  if (ok) {
    for (int c0 = 0; c0 < N; c0 += 32) {
      float x[32];
      tmem_ld32(tm + lanes + c0, x);
      tmem_ld_wait();
      for (int e = 0; e < 32; ++e) Dout[row * N + c0 + e] = x[e];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (tid < 32) { tc_fence_after(); tmem_dealloc(tm, 512); }
}

extern "C" int umma_probe_ta(int N, int K, int b_mn, int neg, const void* A, const void* B, float* D) {
  if ((N != 64 && N != 128) || (K != 64 && K != 128)) return -1;
  const int smem = 2 * 32768 + 64 + 1024;
  cudaFuncSetAttribute(probe_ta_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  probe_ta_kernel<<<1, 128, smem>>>(N, K, b_mn, neg, (const __nv_bfloat16*)A,
                                    (const __nv_bfloat16*)B, D);
  return (int)cudaDeviceSynchronize();
}
