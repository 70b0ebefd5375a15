// NVFP4 weight input of the rotation kernels: the loads of one thread's 32
// packed elements and their exact decode to FP32 pairs in the pass-1 layout
// of rotate_block.  NVFP4 as the ComfyUI Turing Utils page (comfy.icu) reads
// it in its NVFP4 loader entry: E2M1 element codes, one E4M3 scale per 16
// elements, one FP32 tensor scale (applied by the caller).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>

#include "rotate_quant.cuh"

namespace convrot {

// NVFP4: two E2M1 codes (one byte, element 2j in the low nibble) -> FP16x2,
// through the hardware FP4 conversion (exact).
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

// Two E4M3 ("FN") scale bytes -> two floats (exact).
__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t two) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(two));
  return __half22float2(*reinterpret_cast<__half2*>(&h2));
}

// Pass-1 pairs of a weight block chunk: the 32 decoded NVFP4 elements
// [c0, c0 + 32) WITHOUT the tensor scale, u = E2M1 * E4M3 (exact in FP32);
// elements >= K are zero (serialised padding is ignored).
__device__ __forceinline__ void decode_nvfp4_pairs(uint2 w0, uint2 w1, uint16_t sc, int c0, int K,
                                                   float2 (&P)[16]) {
  // scales of row 2p (elements c0..c0+15) and row 2p+1 (c0+16..c0+31)
  const float2 scl = e4m3x2_to_float2(sc);
  uint32_t h0[8], h1[8];
  e2m1x8_to_f16x2(w0.x, *reinterpret_cast<uint32_t(*)[4]>(&h0[0]));
  e2m1x8_to_f16x2(w0.y, *reinterpret_cast<uint32_t(*)[4]>(&h0[4]));
  e2m1x8_to_f16x2(w1.x, *reinterpret_cast<uint32_t(*)[4]>(&h1[0]));
  e2m1x8_to_f16x2(w1.y, *reinterpret_cast<uint32_t(*)[4]>(&h1[4]));
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&h0[k]));   // row 2p: 2k, 2k+1
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&h1[k]));   // row 2p+1
    P[2 * k] = mul2(make_float2(a.x, b.x), scl);
    P[2 * k + 1] = mul2(make_float2(a.y, b.y), scl);
  }
  if (c0 + 32 > K) {                          // partial chunk: drop elements >= K
#pragma unroll
    for (int b = 0; b < 16; ++b) {
      if (c0 + b >= K) P[b].x = 0.f;
      if (c0 + 16 + b >= K) P[b].y = 0.f;
    }
  }
}

// Packed nibbles and the two block scales of the 32 elements [c0, c0 + 32);
// nothing past the stored row (K_s) is read.  W16: the 16 packed bytes are
// 16-byte aligned (row pitch K_s/2 a multiple of 16) and read at once.
template <bool W16>
__device__ __forceinline__ void load_nvfp4_raw(const uint8_t* prow, const uint8_t* srow, int c0,
                                               int K, int K_s, uint2& w0, uint2& w1, uint16_t& sc) {
  if (c0 >= K) {
    w0 = make_uint2(0u, 0u);
    w1 = make_uint2(0u, 0u);
    sc = 0;
    return;
  }
  const bool second = c0 + 16 < K_s;          // elements c0+16.. are stored
  if (W16 && second) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(prow + (c0 >> 1)));
    w0 = make_uint2(v.x, v.y);
    w1 = make_uint2(v.z, v.w);
  } else {
    w0 = __ldg(reinterpret_cast<const uint2*>(prow + (c0 >> 1)));
    w1 = second ? __ldg(reinterpret_cast<const uint2*>(prow + (c0 >> 1) + 8)) : make_uint2(0u, 0u);
  }
  // scale rows are K_s/16 bytes long (odd for some K): read the two bytes separately
  sc = static_cast<uint16_t>(__ldg(srow + (c0 >> 4)) |
                             (second ? static_cast<uint32_t>(__ldg(srow + (c0 >> 4) + 1)) << 8 : 0u));
}

}  // namespace convrot
