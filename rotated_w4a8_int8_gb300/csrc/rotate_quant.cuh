// Shared device code of the two ConvRot256 rotation + row-scaled S8 kernels.
//
// One CTA owns one row.  The padded row is split into 256-element blocks; a
// half-warp ("slot") of 16 threads rotates one block at a time.  The
// Sylvester Walsh-Hadamard matrix factorises as H_256 = H_16 (x) H_16 over
// the index j = 16 a + b, so the rotation runs in two register passes:
//   pass 1: thread a holds x[16a + 0..15] and transforms over b;
//   a swizzled shared-memory transpose inside the half-warp;
//   pass 2: thread b holds column b (x[16*0..15 + b]) and transforms over a.
// The result is scaled by 1/16, exactly.  After all blocks of the row are
// rotated (values stay in registers), the CTA reduces the row absmax, derives
// the FP32 scale and its FP32 reciprocal, and writes the S8 codes.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>

namespace convrot {

constexpr int kBlock = 256;
constexpr int kSlotFloats = kBlock + 16;   // +16 floats: adjacent slots use opposite bank halves
constexpr int kMaxThreads = 512;

// Unnormalised 16-point Walsh-Hadamard transform (Sylvester order), in place.
__device__ __forceinline__ void fwht16(float (&v)[16]) {
#pragma unroll
  for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if ((i & h) == 0) {
        const float p = v[i], q = v[i + h];
        v[i] = __fadd_rn(p, q);
        v[i + h] = __fsub_rn(p, q);
      }
    }
  }
}

// Offset (in floats) of element (a, b) of a block inside its slot region.
// Row a is 16 floats; its four 16-byte units are XOR-permuted by (a >> 1) & 3
// so that the float4 writes of pass 1 and the scalar column reads of pass 2
// are both free of bank conflicts.
__device__ __forceinline__ int swz(int a, int b) {
  return a * 16 + ((((b >> 2) ^ (a >> 1)) & 3) << 2) + (b & 3);
}

// Rotates one block: `v` holds this thread's pass-1 row (a = lane16) on entry
// and its pass-2 column (b = lane16) on exit, scaled by 1/16.  `slot_smem` is
// the half-warp's private region.  Must be called by all 32 lanes of the warp
// (`active` masks the work, not the barriers).
__device__ __forceinline__ void rotate_block(float (&v)[16], float* slot_smem, int lane16,
                                             bool active) {
  if (active) {
    fwht16(v);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      float4 w = make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
      *reinterpret_cast<float4*>(slot_smem + swz(lane16, 4 * u)) = w;
    }
  }
  __syncwarp();
  if (active) {
#pragma unroll
    for (int a = 0; a < 16; ++a) v[a] = slot_smem[swz(a, lane16)];
    fwht16(v);
#pragma unroll
    for (int a = 0; a < 16; ++a) v[a] = v[a] * 0.0625f;   // exact: power of two
  }
  __syncwarp();
}

// Row absmax over the CTA.  `red` holds one float per warp.
__device__ __forceinline__ float cta_absmax(float local, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) local = fmaxf(local, __shfl_xor_sync(0xffffffffu, local, o));
  const int warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  if ((threadIdx.x & 31) == 0) red[warp] = local;
  __syncthreads();
  float m = 0.f;
  for (int w = 0; w < nwarps; ++w) m = fmaxf(m, red[w]);
  return m;
}

// FP32 quantiser shared by both operands: s = fp32(amax / 127),
// r = fp32(1 / s), code = clamp(rint(fp32(v * r)), -127, 127).
struct RowQuant {
  float s, r;
  bool degenerate;
  __device__ __forceinline__ explicit RowQuant(float amax) {
    s = __fdiv_rn(amax, 127.0f);
    r = __frcp_rn(s);
    degenerate = (s == 0.0f) || isinf(r);
    if (degenerate) s = 0.0f;
  }
  __device__ __forceinline__ int code(float v) const {
    if (degenerate) return 0;
    int q = __float2int_rn(__fmul_rn(v, r));
    return max(-127, min(127, q));
  }
};

// Writes the 16 codes of this thread's pass-2 column of block `blk`:
// element 16 a + lane16 for a = 0..15.  For each a the 16 threads of a slot
// cover 16 consecutive codes.
__device__ __forceinline__ void store_codes(void* q_row, bool f16_codes, int blk, int lane16,
                                            const float (&v)[16], const RowQuant& rq) {
  const int base = blk * kBlock + lane16;
  if (f16_codes) {
    __half* q = static_cast<__half*>(q_row) + base;
#pragma unroll
    for (int a = 0; a < 16; ++a) q[16 * a] = __int2half_rn(rq.code(v[a]));
  } else {
    int8_t* q = static_cast<int8_t*>(q_row) + base;
#pragma unroll
    for (int a = 0; a < 16; ++a) q[16 * a] = static_cast<int8_t>(rq.code(v[a]));
  }
}

}  // namespace convrot
