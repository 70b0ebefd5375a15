// Measurement aid, not part of the layer: the producer side of a GEMM that
// would decode, rotate and quantise the NVFP4 weight itself ("decode inside
// the GEMM") instead of reading the codes that convrot_prepare_weight wrote.
// The pages stage the weight work beside the GEMM (overlap), not inside it
// (ComfyUI Turing Utils page, comfy.icu, node list, the ConvRot loaders'
// NVFP4 entry); this kernel measures what the fused form would cost.
//
// The layer's GEMM computes each 256 x 256 output tile on a CTA pair; each CTA
// reads one 128-row half of the tile's B operand from shared memory, in the
// tensor core's K-major layout with the 128-byte swizzle, 64 K-columns per
// stage.  A fused producer has to write those codes there itself:
//  - the row scale s_w = max |rotated row| / 127 needs the whole rotated row
//    before any code exists, so a fused layer first runs a scales-only pass
//    (the caller passes the scales convrot_prepare_weight wrote; that pass's
//    own time comes on top);
//  - a code depends on its whole 256-deep rotation block, so the producer
//    fills four 64-deep K steps at once: a 64 KiB "super-stage", double
//    buffered;
//  - no 128 x K_p half-tile of codes fits in shared memory (1.3 MiB at
//    K_p = 5376), so a CTA rebuilds its half-tile for every 256-row strip of
//    tokens that meets it.
// This kernel runs that producer alone, one CTA per SM, over all work units
// of a GEMM with `m_strips` token strips (unit u: weight rows
// 128 * (u % n_halves) + [0, 128)): PW producer warps fill the super-stages
// and one consumer warp releases each as soon as it is full, an MMA that
// takes no time.  A fused GEMM can be no faster than its producer, so this
// kernel's time over a layer's schedule bounds such a GEMM from below.  For
// checking, the consumer copies the super-stages of one chosen unit to `dump`,
// un-swizzled, as FP16 codes.
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>

#include "../../include/convrot.h"
#include "errors.h"
#include "rotate_quant.cuh"
#include "nvfp4.cuh"

namespace crprobe {
using namespace convrot;

constexpr int ROWS = 128;                        // B rows per CTA: one half of a pair's 256-column tile
constexpr int SUB_BYTES = ROWS * 64 * 2;         // one 64-deep K step of FP16 codes: 16 KiB
constexpr int SUPER_BYTES = 4 * SUB_BYTES;       // one 256-deep rotation block: 64 KiB
constexpr int NSUPER = 2;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

constexpr size_t smem_bytes(int pw) {
  return size_t(NSUPER) * SUPER_BYTES + 1024 /*align*/ + size_t(pw) * 4 * kSlotBytes + 64 /*barriers*/;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// try_wait with a suspend-time hint: the waiting thread sleeps until the phase
// completes or kSuspendNs pass, instead of polling beside the producer warps
// (1% faster at 16 producer warps).  Raw input two blocks ahead instead of
// one measured 3% slower there (spills at 96 registers), 5% faster at 8.
constexpr uint32_t kSuspendNs = 20000;
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kSuspendNs)
      : "memory");
  return ok != 0;
}

// Bounded wait (lane 0 of the calling warp; the warp meets after it).  On a
// timeout it records `code` in *status, raises the CTA's abort flag and
// returns false; it also returns false once another warp has aborted.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, int code, volatile int* abort_flag,
                                          int* status) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0 && !mbar_try_wait(bar, parity)) {
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
      if (mbar_try_wait(bar, parity)) break;
      if ((it & 63u) == 0) {
        if (*abort_flag) { ok = 0; break; }
        if (globaltimer() - t0 > kWaitLimitNs) {
          atomicCAS(status, 0, code);
          *abort_flag = 1;
          ok = 0;
          break;
        }
      }
    }
  }
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Byte offset, inside a super-stage, of codes k and k+1 (k even, k < 256) of
// local row n: K step k / 64, row pitch 128 bytes, and the 16-byte chunk index
// XORed with n mod 8 (the 128-byte swizzle, in 1024-byte atoms).
__device__ __forceinline__ uint32_t code_offset(int n, int k) {
  const int kk = k & 63;
  return (k >> 6) * SUB_BYTES + n * 128 + ((((kk >> 3) ^ (n & 7))) << 4) + ((2 * kk) & 15);
}

// The codes of one rotated block of local row n: thread q (= lane8) holds the
// pairs at columns 2q, 2q+1 of every block row a, i.e. codes 16a + 2q and
// 16a + 2q + 1 (a = 2p from U[p].x, V[p].x; a = 2p + 1 from U[p].y, V[p].y).
// The slots of a warp take rows with distinct (n mod 8) / 2, so the 32 lanes'
// 4-byte stores fall on 32 distinct banks.
__device__ __forceinline__ void store_block_codes(char* super, int n, int lane8, const BlockCols& c) {
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    const int k = 32 * p + 2 * lane8;
    *reinterpret_cast<__half2*>(super + code_offset(n, k)) =
        __floats2half2_rn(rint_f<false>(c.U[p].x), rint_f<false>(c.V[p].x));
    *reinterpret_cast<__half2*>(super + code_offset(n, k + 16)) =
        __floats2half2_rn(rint_f<false>(c.U[p].y), rint_f<false>(c.V[p].y));
  }
}

enum : int { PROBE_WAIT_EMPTY = 1, PROBE_WAIT_FULL = 2 };

template <int PW, bool W16>
__global__ void __launch_bounds__((PW + 1) * 32, 1)
producer_probe_kernel(const uint8_t* __restrict__ w_fp4, const uint8_t* __restrict__ w_sf,
                      const float* __restrict__ tscale, const float* __restrict__ w_scale, int N, int K,
                      int K_s, int nblocks, int units, int n_halves, __half* __restrict__ dump,
                      int64_t ld_dump, int dump_unit, int* status) {
  static_assert(ROWS % (8 * PW) == 0, "each warp owns whole 8-row groups");
  constexpr int R = ROWS / (4 * PW);             // rows per slot per block (even)
  extern __shared__ __align__(16) char smem_raw[];
  char* smem = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  char* slots = smem + NSUPER * SUPER_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(slots + PW * 4 * kSlotBytes);
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + NSUPER);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * NSUPER);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NSUPER; ++i) {
      mbar_init(full0 + 8 * i, PW);
      mbar_init(empty0 + 8 * i, 1);
    }
    *abort_flag = 0;
  }
  __syncthreads();

  if (warp < PW) {
    // ---- producer: slot s4 of this warp owns rows 8 g + 2 s4 + (r & 1) of
    // the warp's 8-row groups g, r = 0 .. R-1
    const int s4 = lane >> 3, lane8 = lane & 7;
    char* my = slots + (warp * 4 + s4) * kSlotBytes;
    const float t16 = __ldg(tscale) * 0.0625f;     // t / 16 is exact
    uint32_t use = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
      const int n_base = (u % n_halves) * ROWS;
      int nl[R];
      float rr[R];
      const uint8_t* prow[R];
      const uint8_t* srow[R];
      bool valid[R];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        nl[r] = 8 * (warp * (R / 2) + (r >> 1)) + 2 * s4 + (r & 1);
        const int row = n_base + nl[r];
        valid[r] = row < N;
        const int rc = valid[r] ? row : 0;
        prow[r] = w_fp4 + static_cast<size_t>(rc) * (K_s >> 1);
        srow[r] = w_sf + static_cast<size_t>(rc) * (K_s >> 4);
        const float s = valid[r] ? __ldg(w_scale + rc) : 0.0f;
        rr[r] = s == 0.0f ? 0.0f : __frcp_rn(s);   // the quantiser's reciprocal of a stored scale
      }
      uint2 w0[R], w1[R];
      uint16_t sc[R];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        if (valid[r]) load_nvfp4_raw<W16>(prow[r], srow[r], 32 * lane8, K, K_s, w0[r], w1[r], sc[r]);
        else { w0[r] = w1[r] = make_uint2(0u, 0u); sc[r] = 0; }
      }
      bool ok = true;
      for (int b = 0; b < nblocks; ++b, ++use) {
        uint2 c0[R], c1[R];
        uint16_t cs[R];
#pragma unroll
        for (int r = 0; r < R; ++r) { c0[r] = w0[r]; c1[r] = w1[r]; cs[r] = sc[r]; }
        if (b + 1 < nblocks) {                     // next block's raw input, in flight during this one
#pragma unroll
          for (int r = 0; r < R; ++r)
            if (valid[r])
              load_nvfp4_raw<W16>(prow[r], srow[r], (b + 1) * kBlock + 32 * lane8, K, K_s, w0[r], w1[r], sc[r]);
        }
        const uint32_t buf = use & 1u, ph = (use >> 1) & 1u;
        if (!warp_wait(empty0 + 8 * buf, ph ^ 1u, PROBE_WAIT_EMPTY, abort_flag, status)) { ok = false; break; }
        char* super = smem + buf * SUPER_BYTES;
#pragma unroll
        for (int r = 0; r < R; ++r) {
          float2 P[16];
          decode_nvfp4_pairs(c0[r], c1[r], cs[r], b * kBlock + 32 * lane8, K, P);
          BlockCols c;
          rotate_block(P, c, my, lane8, true);
          scale_cols(c, t16);                      // rotated weight = fp32(z * t / 16)
          scale_cols(c, rr[r]);
          store_block_codes(super, nl[r], lane8, c);
        }
        // the tensor core reads shared memory through the async proxy
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(full0 + 8 * buf);
      }
      if (!ok) break;
    }
  } else if (warp == PW) {
    // ---- consumer: an MMA that takes no time
    uint32_t use = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
      const bool dumping = dump != nullptr && u == dump_unit;
      bool ok = true;
      for (int b = 0; b < nblocks; ++b, ++use) {
        const uint32_t buf = use & 1u, ph = (use >> 1) & 1u;
        if (!warp_wait(full0 + 8 * buf, ph, PROBE_WAIT_FULL, abort_flag, status)) { ok = false; break; }
        if (dumping) {
          const char* super = smem + buf * SUPER_BYTES;
          for (int i = lane; i < ROWS * (kBlock / 2); i += 32) {
            const int n = i / (kBlock / 2), k = 2 * (i % (kBlock / 2));
            *reinterpret_cast<__half2*>(dump + static_cast<size_t>(n) * ld_dump + b * kBlock + k) =
                *reinterpret_cast<const __half2*>(super + code_offset(n, k));
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * buf);
      }
      if (!ok) break;
    }
  }
}

template <int PW, bool W16>
static cudaError_t launch(int grid, const uint8_t* w_fp4, const uint8_t* w_sf, const float* t, const float* s,
                          int N, int K, int K_s, int nblocks, int units, int n_halves, __half* dump,
                          int64_t ld_dump, int dump_unit, int* status, cudaStream_t st) {
  auto k = producer_probe_kernel<PW, W16>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem_bytes(PW)));
  if (e != cudaSuccess) return e;
  k<<<grid, (PW + 1) * 32, smem_bytes(PW), st>>>(w_fp4, w_sf, t, s, N, K, K_s, nblocks, units, n_halves, dump,
                                                 ld_dump, dump_unit, status);
  return cudaGetLastError();
}

}  // namespace crprobe

extern "C" int convrot_decode_gemm_probe(const uint8_t* w_fp4, const uint8_t* w_sf, const float* w_tensor_scale,
                                         const float* w_scale, int N, int K, int m_strips, int producer_warps,
                                         void* dump, int64_t ld_dump, int dump_unit, int32_t* status,
                                         cudaStream_t stream) {
  using namespace crprobe;
  if (N <= 0 || K <= 0 || m_strips <= 0) return CONVROT_ERR_INVALID_ARG;
  if (producer_warps != 8 && producer_warps != 16) return CONVROT_ERR_UNSUPPORTED;
  const int K_p = convrot_padded_k(K);
  if (K_p > CONVROT_MAX_KP) return CONVROT_ERR_UNSUPPORTED;
  if (!w_fp4 || !w_sf || !w_tensor_scale || !w_scale || !status) return CONVROT_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(w_fp4) % 8 || reinterpret_cast<uintptr_t>(w_tensor_scale) % 4 ||
      reinterpret_cast<uintptr_t>(w_scale) % 4 || reinterpret_cast<uintptr_t>(status) % 4)
    return CONVROT_ERR_MISALIGNED;
  const int n_halves = (N + ROWS - 1) / ROWS;
  const long long units = static_cast<long long>(m_strips) * n_halves;
  if (units > 0x7fffffffLL) return CONVROT_ERR_UNSUPPORTED;
  if (dump) {
    if (ld_dump < K_p || dump_unit < 0 || dump_unit >= units) return CONVROT_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(dump) % 4 || ld_dump % 2) return CONVROT_ERR_MISALIGNED;
  }
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaMemsetAsync(status, 0, sizeof(int32_t), stream);
  if (e != cudaSuccess) return convrot::record_cuda_error("decode_gemm_probe setup", e);
  const int grid = static_cast<int>(units < sms ? units : sms);
  const int K_s = ((K + 15) / 16) * 16;
  const bool w16 = (reinterpret_cast<uintptr_t>(w_fp4) % 16 == 0) && ((K_s / 2) % 16 == 0);
  const int nblocks = K_p / CONVROT_BLOCK;
  const int u = static_cast<int>(units);
  __half* d = static_cast<__half*>(dump);
  if (producer_warps == 8)
    e = w16 ? launch<8, true>(grid, w_fp4, w_sf, w_tensor_scale, w_scale, N, K, K_s, nblocks, u, n_halves, d,
                              ld_dump, dump_unit, status, stream)
            : launch<8, false>(grid, w_fp4, w_sf, w_tensor_scale, w_scale, N, K, K_s, nblocks, u, n_halves, d,
                               ld_dump, dump_unit, status, stream);
  else
    e = w16 ? launch<16, true>(grid, w_fp4, w_sf, w_tensor_scale, w_scale, N, K, K_s, nblocks, u, n_halves, d,
                               ld_dump, dump_unit, status, stream)
            : launch<16, false>(grid, w_fp4, w_sf, w_tensor_scale, w_scale, N, K, K_s, nblocks, u, n_halves, d,
                                ld_dump, dump_unit, status, stream);
  return e == cudaSuccess ? CONVROT_OK : convrot::record_cuda_error("decode_gemm_probe launch", e);
}
