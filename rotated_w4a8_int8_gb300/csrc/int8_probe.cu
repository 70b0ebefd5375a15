// Measurement aid, not part of the layer: the legacy warp-level INT8 tensor
// path (mma.sync m16n8k32, s8 x s8 -> s32) run from registers on every SM,
// so that the INT8 rate of this GPU is measured rather than assumed.  sm_103a
// has no 8-bit integer tcgen05 MMA; the layer's GEMM runs the FP16 tensor
// path on S8-valued operands instead, and its rate is reported beside this
// one and beside cuBLASLt's INT8 GEMM.
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/convrot.h"
#include "errors.h"

namespace convrot {

constexpr int kProbeWarps = 4;      // warps per CTA
constexpr int kProbeChains = 8;     // independent accumulators per warp (hides the MMA latency)

// Every MMA adds sum_k a * b over k < 32 to each accumulator element; with
// a = b = 1 in every byte that is 32, so after `iters` iterations each
// element holds 32 * iters, which the caller checks.
__global__ void __launch_bounds__(kProbeWarps * 32)
int8_mma_probe_kernel(uint32_t a_bytes, uint32_t b_bytes, int iters, int32_t* __restrict__ out) {
  int32_t acc[kProbeChains][4];
#pragma unroll
  for (int c = 0; c < kProbeChains; ++c)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[c][j] = 0;
  const uint32_t a0 = a_bytes, a1 = a_bytes, a2 = a_bytes, a3 = a_bytes, b0 = b_bytes, b1 = b_bytes;
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int c = 0; c < kProbeChains; ++c) {
      asm volatile(
          "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
          "{%0, %1, %2, %3};"
          : "+r"(acc[c][0]), "+r"(acc[c][1]), "+r"(acc[c][2]), "+r"(acc[c][3])
          : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
  }
  // one value per warp: the sum of its chains' first elements
  if ((threadIdx.x & 31) == 0) {
    int32_t s = 0;
#pragma unroll
    for (int c = 0; c < kProbeChains; ++c) s += acc[c][0];
    out[blockIdx.x * kProbeWarps + (threadIdx.x >> 5)] = s;
  }
}

}  // namespace convrot

extern "C" int convrot_int8_mma_probe(int blocks, int iters, int32_t* out, cudaStream_t stream) {
  // 32 * iters * kProbeChains must stay below 2^31
  if (blocks <= 0 || iters <= 0 || iters > (1 << 22) || !out) return CONVROT_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(out) % 4) return CONVROT_ERR_MISALIGNED;
  convrot::int8_mma_probe_kernel<<<blocks, convrot::kProbeWarps * 32, 0, stream>>>(0x01010101u, 0x01010101u, iters,
                                                                                   out);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? CONVROT_OK : convrot::record_cuda_error("int8_mma_probe launch", e);
}
