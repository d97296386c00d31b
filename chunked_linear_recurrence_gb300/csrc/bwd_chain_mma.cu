// bwd_chain_mma.cu -- the backward's reverse state-cotangent chain for BF16 inputs on the
// warp-level tensor cores (mma.sync m16n8k8, TF32 operands, FP32 carry).
//
// StateFlow section 3.1, Eq. 6-7: the cotangent of a chunk's entry state is the cotangent
// of the previous chunk's exit state; walking a sequence backwards, per chunk with exit
// cotangent dSn:
//     dDelta   = scale Aqk^T dO + diag(dec) K dSn^T
//     dS_entry = e^{gamma_C} dSn + scale dO^T diag(e^gamma) Q - dDelta^T W
// (the chunk algebra of common.cuh, differentiated).  Two kernels:
//   * mma_bwd_factor_kernel, fully parallel over chunks, computes each chunk's Aqk and W
//     (the [K;Q] K^T contractions, the triangular solve) once;
//   * mma_bwd_chain_kernel walks each (sequence, head) chain backwards, tiled along V
//     (StateFlow section 3.4.1, Eq. 16: rows of the cotangent evolve independently given
//     the chunk factors), with the cotangent rows FP32 in shared memory.  Each chunk's
//     exit cotangent goes to the tape for the token-gradient kernel (head size 128: as the
//     BF16 swizzled tile that kernel's tensor cores read; 64: FP32 [V,K]); the cotangent
//     at the sequence start is d_initial_state.
#include <type_traits>

#include "bwd_chain_tc.cuh"
#include "chunk_record.cuh"
#include "common.cuh"
#include "mma_tiles.cuh"
#include "simt_chunk.cuh"
#include "solve_tc.cuh"
#include "tc_ptx.cuh"

namespace sfg {
namespace {

using namespace mt;
constexpr int NTB = 256;   // 8 warps
// Leading dimensions (floats) of the FP32 tiles: 4 mod 32, so that the mma fragment loads
// (8 rows x 4 columns per instruction) fall on distinct banks.
constexpr int C_LD6 = 68;
template <int D>
__host__ __device__ constexpr int c_ldd() { return D + 4; }

// Two floats as a BF16 pair (the lower index in the low half).
__device__ __forceinline__ uint32_t tc_pack(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

struct CtaBarB {
  __device__ __forceinline__ void operator()() const { __syncthreads(); }
};

}  // namespace

// Per-chunk factors of the backward chain, rows past the sequence end zero: head size 64:
// fac[(slot * H + h)] = { Aqk [64][64], W [64][D], e^gamma [64], dec [64] } (FP32); head
// size 128: the backward's chunk record of chunk_record.cuh (Ahat, (-W)^T, the decays and
// Qg; T' unused).
template <int D>
__host__ __device__ constexpr size_t fac_bytes() {
  return D == 128 ? (size_t)REC2_BYTES : 4 * (64 * 64 + 64 * D + 128);
}

// As mt::each, two adjacent columns at a time: f(row, col, x[col], x[col + 1]).
template <int NTILE, int NTN, int NW, bool BLK, typename F>
__device__ __forceinline__ void each_pair(float (&acc)[NTILE][4], int warp, int lane, F&& f) {
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int ti = 0; ti < NTILE; ++ti) {
    int m0, n0;
    TileMap<NTILE, NTN, NW, BLK>::at(warp, ti, m0, n0);
    f(m0 + g, n0 + 2 * t, acc[ti][0], acc[ti][1]);
    f(m0 + g + 8, n0 + 2 * t, acc[ti][2], acc[ti][3]);
  }
}

// One chunk (backward slot `slot`); false when the slot holds no chunk.
template <int D>
__device__ __forceinline__ bool factor_chunk(const ChainParams& p, float* fac, int64_t slot) {
  constexpr int LDI = D + 8, LD6 = C_LD6, NTD = D / 8, TD = 4 * NTD / 8;
  extern __shared__ float sm[];
  float* sA = sm;                 // A = diag(beta) Ak, then scratch of the solve
  float* sT = sA + 64 * LD6;
  float* sX = sT + 64 * LD6;      // solve scratch (1024 floats)
  float* sg = sX + 64 * LD6;
  float* sb = sg + 64;
  float* sgam = sb + 64;
  float* sbeg = sgam + 64;
  __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(sbeg + 64);
  __nv_bfloat16* sK = sQ + 64 * LDI;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, h = blockIdx.y, H = p.H;
  const int hk = qk_head(h, H, p.HK);
  const float scale = p.scale;
  int n;
  int64_t bos, eos, ci;
  if (!locate_chunk(slot, p.B, p.T, p.cu, p.N, n, bos, eos, ci)) return false;
  const int64_t c0 = bos + ci * CHUNK;
  const int L = (int)((eos - c0) < CHUNK ? (eos - c0) : CHUNK);
  const __nv_bfloat16* q = (const __nv_bfloat16*)p.q;
  const __nv_bfloat16* k = (const __nv_bfloat16*)p.k;
  for (int idx = tid; idx < 64 * D; idx += NTB) {
    const int i = idx / D, c = idx % D;
    const size_t off = ((size_t)(c0 + i) * p.HK + hk) * D + c;
    const __nv_bfloat16 z = __float2bfloat16_rn(0.f);
    sQ[i * LDI + c] = (i < L) ? q[off] : z;
    sK[i * LDI + c] = (i < L) ? k[off] : z;
  }
  if (tid < 64) {
    const size_t off = (size_t)(c0 + tid) * H + h;
    sg[tid] = (tid < L) ? p.g[off] : 0.f;
    sb[tid] = (tid < L) ? p.beta[off] : 0.f;
  }
  __syncthreads();
  if (tid < 32) warp_cumsum64(sg, sgam, tid);
  __syncthreads();
  float* out = fac + (size_t)(slot * H + h) * (fac_bytes<D>() / 4);
  float* oAqk = out;
  float* oW = out + 64 * 64;
  float* ovec = oW + 64 * D;
  uint8_t* ob = reinterpret_cast<uint8_t*>(out);   // head size 128: the BF16 tile layout
  if (tid < 64) {
    const float eg = expf(sgam[tid]);
    sbeg[tid] = sb[tid] * eg;
    if constexpr (D == 128) {
      float* fv = reinterpret_cast<float*>(ob + R_VEC);
      fv[V_DEC / 4 + tid] = expf(sgam[63] - sgam[tid]);
      fv[V_EG / 4 + tid] = eg;
      if (tid == 0) fv[V_GC / 4] = expf(sgam[63]);
    } else {
      ovec[tid] = eg;
      ovec[64 + tid] = expf(sgam[63] - sgam[tid]);
    }
  }
  const auto Kv = view(sK, LDI, 1);
  {
    float a1[4][4], a2[4][4];
    zero(a1);
    zero(a2);
    // BF16 inputs on BF16 mma: the products are exact, the sums FP32
    gemm16<4, 8, 8, true>(a1, rm(sK, LDI), cm(sK, LDI), D, warp, lane);
    gemm16<4, 8, 8, true>(a2, rm(sQ, LDI), cm(sK, LDI), D, warp, lane);
    each<4, 8, 8, true>(a1, warp, lane, [&](int i, int j, float& x) {
      sA[i * LD6 + j] = (j < i) ? sb[i] * expf(sgam[i] - sgam[j]) * x : 0.f;
    });
    if constexpr (D == 128) {
      each_pair<4, 8, 8, true>(a2, warp, lane, [&](int i, int j, float x0, float x1) {
        const float y0 = (j <= i) ? expf(sgam[i] - sgam[j]) * x0 : 0.f;
        const float y1 = (j + 1 <= i) ? expf(sgam[i] - sgam[j + 1]) * x1 : 0.f;
        *reinterpret_cast<uint32_t*>(ob + R_AH + tc::sw128_off(i, j, 8192)) =
            tc::pack_bf16x2(y0, y1);
      });
    } else {
      each<4, 8, 8, true>(a2, warp, lane, [&](int i, int j, float& x) {
        oAqk[i * 64 + j] = (j <= i) ? expf(sgam[i] - sgam[j]) * x : 0.f;
      });
    }
  }
  __syncthreads();
  if constexpr (D == 128) {
    // Qg = scale diag(e^gamma) Q, eight columns (16 bytes) per store
    for (int idx = tid; idx < 64 * 16; idx += NTB) {
      const int i = idx >> 4, c = (idx & 15) * 8;
      const float f = scale * expf(sgam[i]);
      float x[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = f * __bfloat162float(sQ[i * LDI + c + e]);
      tc::st_row8_bf16(ob + R_QG, i, c, 8192, x);
    }
  }
  static_assert(LD6 == SOLVE_LD, "solve layout");
  solve64_tc(sA, sT, sX, tid, NTB, CtaBarB());   // merges on TF32 mma, as in the forward
  {
    float acc[TD][4];
    zero(acc);
    gemm<TD, NTD, 8, true>(acc, cols_scaled(view(sT, LD6, 1), sbeg), Kv, 64, warp, lane);
    if constexpr (D == 128) {
      // (-W)^T [128 k][64 i]: element (i, c) of W at row c, column i
      each_pair<TD, NTD, 8, true>(acc, warp, lane, [&](int i, int c, float x0, float x1) {
        *reinterpret_cast<__nv_bfloat16*>(ob + R_W + tc::sw128_off(c, i, 16384)) =
            __float2bfloat16_rn(-x0);
        *reinterpret_cast<__nv_bfloat16*>(ob + R_W + tc::sw128_off(c + 1, i, 16384)) =
            __float2bfloat16_rn(-x1);
      });
    } else {
      each<TD, NTD, 8, true>(acc, warp, lane, [&](int i, int c, float& x) { oW[i * D + c] = x; });
    }
  }
  return true;
}

// Slots blockIdx.x, blockIdx.x + gridDim.x, ... until the first empty one.
template <int D>
__global__ void __launch_bounds__(NTB) mma_bwd_factor_kernel(const ChainParams p, float* fac,
                                                             int64_t slots) {
  for (int64_t slot = blockIdx.x; slot < slots; slot += gridDim.x) {
    if (!factor_chunk<D>(p, fac, slot)) break;
    __syncthreads();   // shared memory is rewritten by the next chunk
  }
}

// 16-byte asynchronous copy global -> shared; src_bytes = 0 fills the 16 bytes with zeros.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Shared-memory operands of one chunk of the reverse chain (two of them: the next chunk's
// arrive while the current one is used).
template <int D, int BV>
struct ChainBuf {
  static constexpr int LDI = D + 8, LDO = BV + 8;
  static constexpr size_t Q = 0;                                   // [64][LDI] bf16
  static constexpr size_t K = Q + 2 * 64 * LDI;                    // [64][LDI] bf16
  static constexpr size_t W = K + 2 * 64 * LDI;                    // [64][c_ldd] f32
  static constexpr size_t AQK = W + 4 * 64 * c_ldd<D>();           // [64][C_LD6] f32
  static constexpr size_t DO = AQK + 4 * 64 * C_LD6;               // [64][LDO] bf16
  static constexpr size_t VEC = DO + 2 * 64 * LDO;                 // e^gamma [64], dec [64]
  static constexpr size_t BYTES = VEC + 4 * 128;
  static_assert(K % 16 == 0 && W % 16 == 0 && AQK % 16 == 0 && DO % 16 == 0 && VEC % 16 == 0 &&
                    BYTES % 16 == 0,
                "16-byte copies");
};

// Reverse chain: grid (D / BV, H, N); CTA (rv, h, n) owns cotangent rows [BV rv, BV rv + BV).
template <int D, int BV>
__global__ void __launch_bounds__(NTB) mma_bwd_chain_kernel(const ChainParams p, const float* fac) {
  using B = ChainBuf<D, BV>;
  // dS rows: 8 mod 32 floats, for the conflict-free 8-byte BF16-pair loads of dS K^T
  constexpr int LDS = D + 8, LD6 = C_LD6, LDI = B::LDI, LDO = B::LDO, LDW = c_ldd<D>();
  constexpr int MB = BV / 16;                 // 16-row bands of the cotangent tile
  constexpr int T64 = MB * 8 / 8;             // tiles per warp of a BV x 64 output
  constexpr int TDD = MB * (D / 8) / 8;       // tiles per warp of a BV x D output
  static_assert(MB * 8 % 8 == 0 && MB * (D / 8) % 8 == 0, "tiles per warp");
  extern __shared__ __align__(16) float sm[];
  float* dS = sm;                             // [BV][LDS] running cotangent rows
  float* dDT = dS + BV * LDS;                 // [BV][LD6] dDelta^T
  uint8_t* bufs = reinterpret_cast<uint8_t*>(dDT + BV * LD6);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.y, n = blockIdx.z, r0 = blockIdx.x * BV, H = p.H;
  const int hk = qk_head(h, H, p.HK);
  const float scale = p.scale;
  const __nv_bfloat16* q = (const __nv_bfloat16*)p.q;
  const __nv_bfloat16* k = (const __nv_bfloat16*)p.k;
  const __nv_bfloat16* dO = (const __nv_bfloat16*)p.dout;
  int64_t bos, eos;
  seq_span(n, p.B, p.T, p.cu, bos, eos);
  const int64_t nc = n_chunks(eos - bos);
  const int64_t slot0 = chunk_slot_base(n, p.B, p.T, p.cu);

  // chunk ci's operands into buffer `buf` (one commit group)
  auto stage = [&](int64_t ci, int buf) {
    uint8_t* base = bufs + (size_t)buf * B::BYTES;
    const int64_t c0 = bos + ci * CHUNK;
    const int L = (int)((eos - c0) < CHUNK ? (eos - c0) : CHUNK);
    const float* f = fac + ((size_t)(slot0 + ci) * H + h) * (fac_bytes<D>() / 4);
    constexpr int QP = D / 8;                 // 16-byte pieces per q/k row
    for (int idx = tid; idx < 64 * QP; idx += NTB) {
      const int i = idx / QP, c = (idx % QP) * 8;
      const size_t off = ((size_t)(c0 + (i < L ? i : 0)) * p.HK + hk) * D + c;
      const int nb = i < L ? 16 : 0;
      cp_async16(base + B::Q + 2 * (i * LDI + c), q + off, nb);
      cp_async16(base + B::K + 2 * (i * LDI + c), k + off, nb);
    }
    constexpr int WP = D / 4;                 // 16-byte pieces per W row
    for (int idx = tid; idx < 64 * WP; idx += NTB) {
      const int i = idx / WP, c = (idx % WP) * 4;
      cp_async16(base + B::W + 4 * (i * LDW + c), f + 64 * 64 + i * D + c, 16);
    }
    for (int idx = tid; idx < 64 * 16; idx += NTB) {
      const int i = idx >> 4, c = (idx & 15) * 4;
      cp_async16(base + B::AQK + 4 * (i * LD6 + c), f + i * 64 + c, 16);
    }
    constexpr int OP = BV / 8;                // 16-byte pieces per dO row segment
    for (int idx = tid; idx < 64 * OP; idx += NTB) {
      const int i = idx / OP, c = (idx % OP) * 8;
      const size_t off = ((size_t)(c0 + (i < L ? i : 0)) * H + h) * D + r0 + c;
      cp_async16(base + B::DO + 2 * (i * LDO + c), dO + off, i < L ? 16 : 0);
    }
    if (tid < 32) cp_async16(base + B::VEC + 16 * tid, f + 64 * 64 + 64 * D + 4 * tid, 16);
    cp_async_commit();
  };

  for (int idx = tid; idx < BV * D; idx += NTB) {
    const int r = idx / D, c = idx % D;
    dS[r * LDS + c] = p.dsf ? p.dsf[(((size_t)n * H + h) * D + r0 + r) * D + c] : 0.f;
  }
  if (nc > 0) stage(nc - 1, 0);
  for (int64_t ci = nc - 1; ci >= 0; --ci) {
    const int buf = (int)((nc - 1 - ci) & 1);
    const size_t slot = (size_t)(slot0 + ci);
    __syncthreads();                          // the other buffer's last reader is done
    if (ci > 0) {
      stage(ci - 1, buf ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();                          // this chunk's operands have landed
    const uint8_t* base = bufs + (size_t)buf * B::BYTES;
    const __nv_bfloat16* sQ = reinterpret_cast<const __nv_bfloat16*>(base + B::Q);
    const __nv_bfloat16* sK = reinterpret_cast<const __nv_bfloat16*>(base + B::K);
    const float* sW = reinterpret_cast<const float*>(base + B::W);
    const float* sAqk = reinterpret_cast<const float*>(base + B::AQK);
    const __nv_bfloat16* sdO = reinterpret_cast<const __nv_bfloat16*>(base + B::DO);
    const float* seg = reinterpret_cast<const float*>(base + B::VEC);
    const float* sdec = seg + 64;
    const auto dOT = view(sdO, 1, LDO);       // dO^T (v, i)
    if constexpr (D == 128) {
      // the tensor-core gradient kernel's operand: rows r0 .. r0 + BV - 1 of a BF16
      // [128 v][128 k] tile in the 128-byte-swizzled panel layout (16-byte chunk c of row v
      // of panel k / 64 at ((c ^ (v mod 8)) << 4))
      uint8_t* dst = reinterpret_cast<uint8_t*>(p.tape) + (slot * H + h) * (size_t)(D * D * 2);
      for (int idx = tid; idx < BV * 16; idx += NTB) {
        const int r = idx >> 4, pc = idx & 15, v = r0 + r, c = pc & 7;
        const float* x = dS + r * LDS + 8 * pc;
        const uint4 val = make_uint4(tc_pack(x[0], x[1]), tc_pack(x[2], x[3]), tc_pack(x[4], x[5]),
                                     tc_pack(x[6], x[7]));
        *reinterpret_cast<uint4*>(dst + (pc >> 3) * 16384 + v * 128 + ((c ^ (v & 7)) << 4)) = val;
      }
    } else {
      float4* dst = reinterpret_cast<float4*>(p.tape + (slot * H + h) * D * D + (size_t)r0 * D);
      for (int idx = tid; idx < BV * D / 4; idx += NTB) {
        const int r = idx / (D / 4), c = (idx % (D / 4)) * 4;
        dst[idx] = make_float4(dS[r * LDS + c], dS[r * LDS + c + 1], dS[r * LDS + c + 2],
                               dS[r * LDS + c + 3]);
      }
    }
    const float gC = seg[63];                 // e^{gamma_C}
    // dDelta^T [v][j] = scale (dO^T Aqk)[v][j] + dec_j (dS K^T)[v][j]
    {
      float a1[T64][4], a2[T64][4];
      zero(a1);
      zero(a2);
      gemm<T64, 8, 8, true>(a1, dOT, view(sAqk, LD6, 1), 64, warp, lane);
      // (k = D: BF16 operand pairs, the forward's tensor-core precision)
      gemm16<T64, 8, 8, true>(a2, rm(dS, LDS), cm(sK, LDI), D, warp, lane);
      each<T64, 8, 8, true>(a2, warp, lane, [&](int, int j, float& x) { x *= sdec[j]; });
#pragma unroll
      for (int ti = 0; ti < T64; ++ti)
#pragma unroll
        for (int e = 0; e < 4; ++e) a1[ti][e] = scale * a1[ti][e] + a2[ti][e];
      each<T64, 8, 8, true>(a1, warp, lane, [&](int v, int j, float& x) { dDT[v * LD6 + j] = x; });
    }
    __syncthreads();
    // dS <- e^{gamma_C} dS + scale (dO^T diag(e^gamma)) Q - dDelta^T W
    {
      float a3[TDD][4], a4[TDD][4];
      zero(a3);
      zero(a4);
      gemm<TDD, D / 8, 8, true>(a3, cols_scaled(dOT, seg), view(sQ, LDI, 1), 64, warp, lane);
      gemm<TDD, D / 8, 8, true>(a4, view(dDT, LD6, 1), view(sW, LDW, 1), 64, warp, lane);
#pragma unroll
      for (int ti = 0; ti < TDD; ++ti)
#pragma unroll
        for (int e = 0; e < 4; ++e) a3[ti][e] = scale * a3[ti][e] - a4[ti][e];
      each<TDD, D / 8, 8, true>(a3, warp, lane, [&](int v, int c, float& x) {
        dS[v * LDS + c] = gC * dS[v * LDS + c] + x;
      });
    }
  }
  __syncthreads();
  if (p.ds0)
    for (int idx = tid; idx < BV * D; idx += NTB) {
      const int r = idx / D, c = idx % D;
      p.ds0[(((size_t)n * H + h) * D + r0 + r) * D + c] = dS[r * LDS + c];
    }
}

size_t mma_bwd_fac_bytes(int D) { return D == 128 ? fac_bytes<128>() : fac_bytes<64>(); }

template <int D>
static cudaError_t launch_chain_d(const ChainParams& p, float* fac, int64_t slots, cudaStream_t st) {
  constexpr int BV = 32;
  {
    const size_t smem = sizeof(float) * (3 * 64 * C_LD6 + 4 * 64) + 2 * 2 * 64 * (D + 8);
    auto kern = mma_bwd_factor_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (slots > 0) kern<<<dim3((unsigned)slot_grid(p, slots), p.H), NTB, smem, st>>>(p, fac, slots);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  const size_t smem = sizeof(float) * (BV * (D + 8) + BV * C_LD6) + 2 * ChainBuf<D, BV>::BYTES;
  auto kern = mma_bwd_chain_kernel<D, BV>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<dim3(D / BV, p.H, p.N), NTB, smem, st>>>(p, fac);
  return cudaGetLastError();
}

cudaError_t launch_mma_bwd_chain(const ChainParams& p, float* fac, int D, int64_t slots,
                                 cudaStream_t st) {
  if (D == 128) {
    // the chunk records: kept by the state replay, else made here; then the reverse chain
    // on tcgen05 (bwd_chain_tc.cu)
    cudaError_t e;
    if (!p.fac_ready) {
      const size_t smem = sizeof(float) * (3 * 64 * C_LD6 + 4 * 64) + 2 * 2 * 64 * (128 + 8);
      auto kern = mma_bwd_factor_kernel<128>;
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      if (slots > 0) kern<<<dim3((unsigned)slot_grid(p, slots), p.H), NTB, smem, st>>>(p, fac, slots);
    } else {
      launch_tc_bwd_qg(p, fac, slots, st);   // the replay's records lack only Qg
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    return launch_tc_bwd_chain(p, fac, st);
  }
  if (D == 64) return launch_chain_d<64>(p, fac, slots, st);
  return cudaErrorInvalidValue;
}

}  // namespace sfg
