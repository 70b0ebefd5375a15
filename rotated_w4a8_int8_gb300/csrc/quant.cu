// Kernels 1 and 2 of the ConvRot W4A8 layer and their C-ABI entry points.
//
//   convrot_prepare_weight: NVFP4 decode -> ConvRot256 rotation (FP32) -> row S8
//   convrot_quant_act:      (SwiGLU ->) ConvRot256 rotation (FP32) -> row S8
//
// Both follow the ComfyUI Turing Utils page (comfy.icu), node list, entry
// "Load ConvRot DiT and Load ConvRot CLIP also accept ComfyUI-native nvfp4
// layers": paired ConvRot256 on activations and decoded NVFP4 weights, both
// operands zero-padded to whole 256-blocks, FP32 rotation, row-scaled S8 with
// a rounded FP32 scale reciprocal.  SwiGLU follows the MiniMax-H3 explainer
// (modelpad.app), MLP section: gate, value = chunk(2); swish(gate) * value.
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>

#include "../../include/convrot.h"
#include "rotate_quant.cuh"

namespace convrot {

// ------------------------------------------------------------------ loaders
enum : int { DT_BF16 = 0, DT_FP16 = 1, DT_FP32 = 2 };

template <int DT>
__device__ __forceinline__ float load_scalar(const void* row, int k) {
  if constexpr (DT == DT_BF16) {
    const uint16_t b = static_cast<const uint16_t*>(row)[k];
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
  } else if constexpr (DT == DT_FP16) {
    return __half2float(static_cast<const __half*>(row)[k]);
  } else {
    return static_cast<const float*>(row)[k];
  }
}

__device__ __forceinline__ void unpack_bf16x2(uint32_t w, float& lo, float& hi) {
  lo = __uint_as_float(w << 16);
  hi = __uint_as_float(w & 0xffff0000u);
}

__device__ __forceinline__ void unpack_f16x2(uint32_t w, float& lo, float& hi) {
  __half2 h = *reinterpret_cast<__half2*>(&w);
  float2 f = __half22float2(h);
  lo = f.x;
  hi = f.y;
}

// 16 consecutive elements x[c0 .. c0+15] of one row, zero beyond K.
template <int DT, bool VEC>
__device__ __forceinline__ void load16(const void* row, int c0, int K, float (&v)[16]) {
  if (c0 >= K) {
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = 0.f;
    return;
  }
  if (VEC && c0 + 16 <= K) {
    if constexpr (DT == DT_FP32) {
      const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(row) + c0);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        float4 f = __ldg(p + u);
        v[4 * u] = f.x; v[4 * u + 1] = f.y; v[4 * u + 2] = f.z; v[4 * u + 3] = f.w;
      }
    } else {
      const uint4* p = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(row) + c0);
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        uint4 w = __ldg(p + u);
        uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if constexpr (DT == DT_BF16) unpack_bf16x2(ws[j], v[8 * u + 2 * j], v[8 * u + 2 * j + 1]);
          else unpack_f16x2(ws[j], v[8 * u + 2 * j], v[8 * u + 2 * j + 1]);
        }
      }
    }
    return;
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = (c0 + i < K) ? load_scalar<DT>(row, c0 + i) : 0.f;
}

// E4M3 ("FN") byte -> float, through the hardware FP8 -> FP16 conversion (exact).
__device__ __forceinline__ float e4m3_to_float(uint8_t b) {
  uint32_t h2;
  const uint16_t pair = b;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(pair));
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  return __low2float(h);
}

// 16 decoded NVFP4 elements of chunk c0/16, WITHOUT the tensor scale:
// u = E2M1 * E4M3, exact in FP32.  Elements >= K (serialised padding or
// beyond the stored row) are zero.
__device__ __forceinline__ void load16_nvfp4(const uint8_t* prow, const uint8_t* srow, int c0,
                                             int K, float (&u)[16]) {
  if (c0 >= K) {
#pragma unroll
    for (int i = 0; i < 16; ++i) u[i] = 0.f;
    return;
  }
  const uint2 pk = __ldg(reinterpret_cast<const uint2*>(prow + (c0 >> 1)));
  const float half_scale = e4m3_to_float(__ldg(srow + (c0 >> 4))) * 0.5f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint32_t word = (i < 8) ? pk.x : pk.y;
    const uint32_t nib = (word >> (4 * (i & 7))) & 0xFu;
    // twice the E2M1 magnitude of codes 0..7 is 0,1,2,3,4,6,8,12 (one nibble each)
    const uint32_t mag2 = (0xC8643210u >> ((nib & 7u) * 4u)) & 0xFu;
    float val = static_cast<float>(mag2) * half_scale;
    if (nib & 8u) val = -val;
    u[i] = (c0 + i < K) ? val : 0.f;
  }
}

// ------------------------------------------------------------------ kernels
// Kernel 2: one CTA per token row.  Thread t: slot = t / 16 rotates blocks
// slot, slot + S, slot + 2S, ... (at most NBMAX of them).
template <int DT, bool SWIGLU, int NBMAX, bool VEC>
__global__ void __launch_bounds__(kMaxThreads)
quant_act_kernel(const void* __restrict__ x, int64_t ld_x, int K, int nblocks, int S,
                 void* __restrict__ q, int f16_codes, int64_t ld_q, float* __restrict__ scale) {
  __shared__ __align__(16) float smem[(kMaxThreads / 16) * kSlotFloats];
  __shared__ float red[kMaxThreads / 32];
  const int row = blockIdx.x;
  const int slot = threadIdx.x >> 4, lane16 = threadIdx.x & 15;
  const size_t esize = (DT == DT_FP32) ? 4 : 2;
  const char* xrow = static_cast<const char*>(x) + static_cast<size_t>(row) * ld_x * esize;
  float* my = smem + slot * kSlotFloats;

  float v[NBMAX][16];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < NBMAX; ++i) {
    const int blk = slot + S * i;
    const bool active = (slot < S) && (blk < nblocks);
    if (active) {
      const int c0 = blk * kBlock + 16 * lane16;
      if constexpr (SWIGLU) {
        float g[16], val[16];
        load16<DT, VEC>(xrow, c0, K, g);
        load16<DT, VEC>(xrow + static_cast<size_t>(K) * esize, c0, K, val);
#pragma unroll
        for (int e = 0; e < 16; ++e) v[i][e] = __fmul_rn(__fdiv_rn(g[e], 1.0f + expf(-g[e])), val[e]);
      } else {
        load16<DT, VEC>(xrow, c0, K, v[i]);
      }
    }
    rotate_block(v[i], my, lane16, active);
    if (active) {
#pragma unroll
      for (int e = 0; e < 16; ++e) amax = fmaxf(amax, fabsf(v[i][e]));
    }
  }
  const RowQuant rq(cta_absmax(amax, red));
  if (threadIdx.x == 0) scale[row] = rq.s;
  const size_t qsize = f16_codes ? 2 : 1;
  void* qrow = static_cast<char*>(q) + static_cast<size_t>(row) * ld_q * qsize;
#pragma unroll
  for (int i = 0; i < NBMAX; ++i) {
    const int blk = slot + S * i;
    if (slot < S && blk < nblocks) store_codes(qrow, f16_codes, blk, lane16, v[i], rq);
  }
}

// Kernel 1: one CTA per weight row; same block schedule as kernel 2.
template <int NBMAX>
__global__ void __launch_bounds__(kMaxThreads)
prepare_weight_kernel(const uint8_t* __restrict__ w_fp4, const uint8_t* __restrict__ w_sf,
                      const float* __restrict__ tscale, int K, int K_s, int nblocks, int S,
                      void* __restrict__ q, int f16_codes, int64_t ld_q, float* __restrict__ scale) {
  __shared__ __align__(16) float smem[(kMaxThreads / 16) * kSlotFloats];
  __shared__ float red[kMaxThreads / 32];
  const int row = blockIdx.x;
  const int slot = threadIdx.x >> 4, lane16 = threadIdx.x & 15;
  const uint8_t* prow = w_fp4 + static_cast<size_t>(row) * (K_s >> 1);
  const uint8_t* srow = w_sf + static_cast<size_t>(row) * (K_s >> 4);
  const float t = __ldg(tscale);
  float* my = smem + slot * kSlotFloats;

  float v[NBMAX][16];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < NBMAX; ++i) {
    const int blk = slot + S * i;
    const bool active = (slot < S) && (blk < nblocks);
    if (active) load16_nvfp4(prow, srow, blk * kBlock + 16 * lane16, K, v[i]);
    rotate_block(v[i], my, lane16, active);
    if (active) {
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        v[i][e] = __fmul_rn(v[i][e], t);           // rotated weight in FP32
        amax = fmaxf(amax, fabsf(v[i][e]));
      }
    }
  }
  const RowQuant rq(cta_absmax(amax, red));
  if (threadIdx.x == 0) scale[row] = rq.s;
  const size_t qsize = f16_codes ? 2 : 1;
  void* qrow = static_cast<char*>(q) + static_cast<size_t>(row) * ld_q * qsize;
#pragma unroll
  for (int i = 0; i < NBMAX; ++i) {
    const int blk = slot + S * i;
    if (slot < S && blk < nblocks) store_codes(qrow, f16_codes, blk, lane16, v[i], rq);
  }
}

// ------------------------------------------------------------------ launch geometry
struct RowGeometry {
  int nblocks, nbmax, S, threads;
};

// At most 32 slots (512 threads) per row; each slot rotates ceil(nblocks/32)
// blocks, held in registers (NBMAX = 1, 2, 4 or 8 -> K_p <= 65536).
static bool row_geometry(int K_p, RowGeometry* g) {
  g->nblocks = K_p / kBlock;
  const int nb = (g->nblocks + 31) / 32;
  if (nb > 8) return false;
  g->nbmax = nb <= 1 ? 1 : nb <= 2 ? 2 : nb <= 4 ? 4 : 8;
  g->S = (g->nblocks + nb - 1) / nb;
  g->threads = ((16 * g->S + 31) / 32) * 32;
  return true;
}

template <int DT, bool SWIGLU, bool VEC>
static cudaError_t launch_act_dt(const RowGeometry& g, int M, const void* x, int64_t ld_x, int K,
                                 void* q, int f16, int64_t ld_q, float* scale, cudaStream_t st) {
  dim3 grid(M), block(g.threads);
  switch (g.nbmax) {
    case 1: quant_act_kernel<DT, SWIGLU, 1, VEC><<<grid, block, 0, st>>>(x, ld_x, K, g.nblocks, g.S, q, f16, ld_q, scale); break;
    case 2: quant_act_kernel<DT, SWIGLU, 2, VEC><<<grid, block, 0, st>>>(x, ld_x, K, g.nblocks, g.S, q, f16, ld_q, scale); break;
    case 4: quant_act_kernel<DT, SWIGLU, 4, VEC><<<grid, block, 0, st>>>(x, ld_x, K, g.nblocks, g.S, q, f16, ld_q, scale); break;
    default: quant_act_kernel<DT, SWIGLU, 8, VEC><<<grid, block, 0, st>>>(x, ld_x, K, g.nblocks, g.S, q, f16, ld_q, scale); break;
  }
  return cudaGetLastError();
}

template <int DT>
static cudaError_t launch_act(const RowGeometry& g, int M, const void* x, int64_t ld_x, int K,
                              bool swiglu, bool vec, void* q, int f16, int64_t ld_q, float* scale,
                              cudaStream_t st) {
  if (swiglu) {
    return vec ? launch_act_dt<DT, true, true>(g, M, x, ld_x, K, q, f16, ld_q, scale, st)
               : launch_act_dt<DT, true, false>(g, M, x, ld_x, K, q, f16, ld_q, scale, st);
  }
  return vec ? launch_act_dt<DT, false, true>(g, M, x, ld_x, K, q, f16, ld_q, scale, st)
             : launch_act_dt<DT, false, false>(g, M, x, ld_x, K, q, f16, ld_q, scale, st);
}

}  // namespace convrot

using namespace convrot;

extern "C" int convrot_quant_act(const void* x, convrot_dtype x_dtype, int64_t ld_x, int M, int K,
                                 int swiglu, void* a_q, convrot_codes fmt, int64_t ld_aq,
                                 float* a_scale, cudaStream_t stream) {
  if (M < 0 || K <= 0) return CONVROT_ERR_INVALID_ARG;
  if (x_dtype != CONVROT_BF16 && x_dtype != CONVROT_FP16 && x_dtype != CONVROT_FP32)
    return CONVROT_ERR_UNSUPPORTED;
  if (fmt != CONVROT_CODES_S8 && fmt != CONVROT_CODES_F16) return CONVROT_ERR_UNSUPPORTED;
  const int K_p = convrot_padded_k(K);
  if (K_p > CONVROT_MAX_KP) return CONVROT_ERR_UNSUPPORTED;
  const int64_t k_in = swiglu ? 2 * static_cast<int64_t>(K) : K;
  if (ld_x < k_in || ld_aq < K_p) return CONVROT_ERR_INVALID_ARG;
  if (M == 0) return CONVROT_OK;
  if (!x || !a_q || !a_scale) return CONVROT_ERR_INVALID_ARG;
  const size_t esize = x_dtype == CONVROT_FP32 ? 4 : 2;
  if (reinterpret_cast<uintptr_t>(x) % esize) return CONVROT_ERR_MISALIGNED;
  if (fmt == CONVROT_CODES_F16 && reinterpret_cast<uintptr_t>(a_q) % 2) return CONVROT_ERR_MISALIGNED;
  if (reinterpret_cast<uintptr_t>(a_scale) % 4) return CONVROT_ERR_MISALIGNED;
  // vector path: every row start and the value half (SwiGLU) 16-byte aligned
  const bool vec = (reinterpret_cast<uintptr_t>(x) % 16 == 0) &&
                   ((ld_x * static_cast<int64_t>(esize)) % 16 == 0) &&
                   (!swiglu || (static_cast<int64_t>(K) * esize) % 16 == 0);
  RowGeometry g;
  if (!row_geometry(K_p, &g)) return CONVROT_ERR_UNSUPPORTED;
  const int f16 = fmt == CONVROT_CODES_F16;
  cudaError_t e;
  switch (x_dtype) {
    case CONVROT_BF16: e = launch_act<DT_BF16>(g, M, x, ld_x, K, swiglu != 0, vec, a_q, f16, ld_aq, a_scale, stream); break;
    case CONVROT_FP16: e = launch_act<DT_FP16>(g, M, x, ld_x, K, swiglu != 0, vec, a_q, f16, ld_aq, a_scale, stream); break;
    default: e = launch_act<DT_FP32>(g, M, x, ld_x, K, swiglu != 0, vec, a_q, f16, ld_aq, a_scale, stream); break;
  }
  return e == cudaSuccess ? CONVROT_OK : CONVROT_ERR_CUDA;
}

extern "C" int convrot_prepare_weight(const uint8_t* w_fp4, const uint8_t* w_sf,
                                      const float* w_tensor_scale, int N, int K, void* w_q,
                                      convrot_codes fmt, int64_t ld_wq, float* w_scale,
                                      cudaStream_t stream) {
  if (N < 0 || K <= 0) return CONVROT_ERR_INVALID_ARG;
  if (fmt != CONVROT_CODES_S8 && fmt != CONVROT_CODES_F16) return CONVROT_ERR_UNSUPPORTED;
  const int K_p = convrot_padded_k(K);
  if (K_p > CONVROT_MAX_KP) return CONVROT_ERR_UNSUPPORTED;
  if (ld_wq < K_p) return CONVROT_ERR_INVALID_ARG;
  if (N == 0) return CONVROT_OK;
  if (!w_fp4 || !w_sf || !w_tensor_scale || !w_q || !w_scale) return CONVROT_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(w_fp4) % 8 || reinterpret_cast<uintptr_t>(w_tensor_scale) % 4 ||
      reinterpret_cast<uintptr_t>(w_scale) % 4)
    return CONVROT_ERR_MISALIGNED;
  if (fmt == CONVROT_CODES_F16 && reinterpret_cast<uintptr_t>(w_q) % 2) return CONVROT_ERR_MISALIGNED;
  RowGeometry g;
  if (!row_geometry(K_p, &g)) return CONVROT_ERR_UNSUPPORTED;
  const int K_s = ((K + 15) / 16) * 16;
  const int f16 = fmt == CONVROT_CODES_F16;
  dim3 grid(N), block(g.threads);
  switch (g.nbmax) {
    case 1: prepare_weight_kernel<1><<<grid, block, 0, stream>>>(w_fp4, w_sf, w_tensor_scale, K, K_s, g.nblocks, g.S, w_q, f16, ld_wq, w_scale); break;
    case 2: prepare_weight_kernel<2><<<grid, block, 0, stream>>>(w_fp4, w_sf, w_tensor_scale, K, K_s, g.nblocks, g.S, w_q, f16, ld_wq, w_scale); break;
    case 4: prepare_weight_kernel<4><<<grid, block, 0, stream>>>(w_fp4, w_sf, w_tensor_scale, K, K_s, g.nblocks, g.S, w_q, f16, ld_wq, w_scale); break;
    default: prepare_weight_kernel<8><<<grid, block, 0, stream>>>(w_fp4, w_sf, w_tensor_scale, K, K_s, g.nblocks, g.S, w_q, f16, ld_wq, w_scale); break;
  }
  return cudaGetLastError() == cudaSuccess ? CONVROT_OK : CONVROT_ERR_CUDA;
}
