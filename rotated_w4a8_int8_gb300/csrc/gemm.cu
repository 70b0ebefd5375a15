// Kernel 3 of the ConvRot W4A8 layer: the row-scaled integer GEMM with its
// dequantising epilogue, and the C-ABI entry points convrot_gemm,
// convrot_gemm_i32 and convrot_device_error.
//
// What it computes (ComfyUI Turing Utils page on comfy.icu, node list, entry
// "Load ConvRot DiT ... nvfp4": "row-scaled INT8 Tensor Core GEMM", FP16 /
// BF16 / FP32 outputs, N tails; MiniMax-H3 explainer on modelpad.app: the
// rescale lives inside the matmul so the int32 intermediate never touches
// memory):
//     acc[m, n] = sum_k q_a[m, k] * q_w[n, k]            (exact int32)
//     y[m, n]   = fp32(acc) * s_a[m] * s_w[n]  -> out dtype
//
// GB300 design.  sm_103a has no 8-bit integer tcgen05 MMA, so the S8 codes
// arrive stored as FP16 integers and the product runs on tcgen05.mma
// kind::f16 with FP32 accumulation in tensor memory.  Products are at most
// 127^2 and a 512-deep partial sum at most 127^2 * 512 < 2^23, so every FP32
// partial sum is an exact integer.  The K loop is therefore cut into 512-wide
// chunks, each accumulated afresh in one of two TMEM buffers; epilogue warps
// convert each finished chunk to int32 (exact) and add it to per-thread int32
// registers while the tensor core fills the other buffer.
//
// CTA tile 128 x 256 (UMMA M=128, N=256, K=16), K step 64 (one 128-byte
// swizzled row per operand row), 4-stage TMA ring, persistent CTAs over a
// grouped tile order.  Warp 0: TMA producer.  Warp 1: TMEM owner and MMA
// issuer.  Warps 2..9: epilogue.  Every mbarrier wait is bounded: after about
// two seconds the waiting role records an error code, the CTA drains what it
// has in flight and returns.
#include <cstdint>
#include <cstdio>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "../../include/convrot.h"

namespace crgemm {

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int STAGES = 4;
constexpr int KCHUNK_STEPS = 8;                  // 8 * 64 = 512 K per exact FP32 chunk
constexpr int A_BYTES = BM * BK * 2;             // 16 KiB
constexpr int B_BYTES = BN * BK * 2;             // 32 KiB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int NUM_EPI_WARPS = 8;
constexpr int THREADS = 64 + NUM_EPI_WARPS * 32; // 320
constexpr int TMEM_COLS = 512;                   // two 256-column FP32 buffers
constexpr int GROUP_M = 16;                      // tile raster: 16 M-tiles share each B tile
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

enum ErrCode : int { ERR_NONE = 0, ERR_WAIT_FULL = 1, ERR_WAIT_EMPTY = 2, ERR_WAIT_ACC_FULL = 3,
                     ERR_WAIT_ACC_EMPTY = 4, ERR_WAIT_DRAIN = 5 };

__device__ int g_error = 0;   // first failure code of any GEMM launch (0 = none)

// ------------------------------------------------------------------ PTX helpers
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

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity.  Returns false (after
// recording `code`) if the phase does not complete within kWaitLimitNs or if
// another role of this CTA has already aborted.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int code,
                                          volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer() - t0 > kWaitLimitNs) {
        atomicCAS(&g_error, 0, code);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               ::"r"(bar) : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, FP16 inputs, FP32 accumulate.
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp receives
// row (lane base + i), columns col .. col+31.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile written by TMA
// with 128-byte swizzling: rows of 128 bytes, 8-row (1024-byte) swizzle atoms
// stacked along M/N (stride byte offset 1024), descriptor version 1, layout
// SWIZZLE_128B.  The leading byte offset is unused for this layout.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);       // start address
  d |= static_cast<uint64_t>(1) << 16;                       // leading byte offset (16 B, unused)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;               // stride byte offset
  d |= static_cast<uint64_t>(1) << 46;                       // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                       // SWIZZLE_128B
  return d;
}

// Instruction descriptor, kind::f16: D FP32, A and B FP16, both K-major,
// N = 256, M = 128.
constexpr uint32_t kIdesc = (1u << 4)                         // D format: F32
                            | (0u << 7) | (0u << 10)          // A, B: F16
                            | (0u << 15) | (0u << 16)         // K-major A and B
                            | (static_cast<uint32_t>(BN >> 3) << 17)
                            | (static_cast<uint32_t>(BM >> 4) << 24);

struct Params {
  int M, N, K_p;
  int num_m, num_n, num_tiles, k_steps;
  const float* a_scale;
  const float* w_scale;
  void* out;
  int64_t ld_out;
  int out_vec;      // 16-byte vector stores allowed (base and pitch aligned)
};

__device__ __forceinline__ void tile_coords(int tile, int num_m, int num_n, int& mb, int& nb) {
  const int per_group = GROUP_M * num_n;
  const int g = tile / per_group;
  const int first_m = g * GROUP_M;
  const int gsize = min(GROUP_M, num_m - first_m);
  const int r = tile - g * per_group;
  mb = first_m + r % gsize;
  nb = r / gsize;
}

// ------------------------------------------------------------------ epilogue stores
template <int OUT>
struct OutT;
template <> struct OutT<CONVROT_BF16> { using T = __nv_bfloat16; };
template <> struct OutT<CONVROT_FP16> { using T = __half; };
template <> struct OutT<CONVROT_FP32> { using T = float; };

template <int OUT>
__device__ __forceinline__ typename OutT<OUT>::T to_out(float y);
template <> __device__ __forceinline__ __nv_bfloat16 to_out<CONVROT_BF16>(float y) { return __float2bfloat16_rn(y); }
template <> __device__ __forceinline__ __half to_out<CONVROT_FP16>(float y) { return __float2half_rn(y); }
template <> __device__ __forceinline__ float to_out<CONVROT_FP32>(float y) { return y; }

// OUT = CONVROT_BF16 / FP16 / FP32, or -1 for raw int32 accumulators.
template <int OUT>
__global__ void __launch_bounds__(THREADS, 1)
gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
            const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  // barrier slots: full[4], empty[4], acc_full[2], acc_empty[2], drain
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + STAGES);
  const uint32_t accf0 = smem_u32(bars + 2 * STAGES), acce0 = smem_u32(bars + 2 * STAGES + 2);
  const uint32_t drain = smem_u32(bars + 2 * STAGES + 4);
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(bars + 2 * STAGES + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * STAGES + 6);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf0 + 8 * b, 1);
      mbar_init(acce0 + 8 * b, NUM_EPI_WARPS);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_a)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_b)) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_u32(const_cast<uint32_t*>(tmem_slot))), "r"(TMEM_COLS) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int k_steps = p.k_steps;
  const int chunks_per_tile = (k_steps + KCHUNK_STEPS - 1) / KCHUNK_STEPS;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      uint32_t issued_mask = 0, issued_phase = 0;   // last outstanding load per stage
      for (int tile = blockIdx.x; tile < p.num_tiles && ok; tile += gridDim.x) {
        int mb, nb;
        tile_coords(tile, p.num_m, p.num_n, mb, nb);
        for (int ks = 0; ks < k_steps; ++ks) {
          if (!mbar_wait(empty0 + 8 * stage, phase ^ 1u, ERR_WAIT_EMPTY, abort_flag)) { ok = false; break; }
          const uint32_t fb = full0 + 8 * stage;
          mbar_arrive_expect_tx(fb, STAGE_BYTES);
          const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
          tma_load_2d(sa, &tmap_a, fb, ks * BK, mb * BM);
          tma_load_2d(sa + A_BYTES, &tmap_b, fb, ks * BK, nb * BN);
          issued_mask |= 1u << stage;
          issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) {
        // let every load still in flight land before the CTA can exit
        for (int s = 0; s < STAGES; ++s)
          if (issued_mask & (1u << s)) {
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(full0 + 8 * s, (issued_phase >> s) & 1u) &&
                   globaltimer() - t0 < kWaitLimitNs) {}
          }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t chunk = 0;          // running chunk counter -> TMEM buffer and its phase
      bool ok = true;
      bool any = false;
      for (int tile = blockIdx.x; tile < p.num_tiles && ok; tile += gridDim.x) {
        for (int c = 0; c < chunks_per_tile && ok; ++c, ++chunk) {
          const uint32_t buf = chunk & 1u, use = chunk >> 1;
          if (!mbar_wait(acce0 + 8 * buf, (use & 1u) ^ 1u, ERR_WAIT_ACC_EMPTY, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + buf * BN;
          const int ks0 = c * KCHUNK_STEPS, ks1 = min(k_steps, ks0 + KCHUNK_STEPS);
          for (int ks = ks0; ks < ks1; ++ks) {
            if (!mbar_wait(full0 + 8 * stage, phase, ERR_WAIT_FULL, abort_flag)) { ok = false; break; }
            tc_fence_after();
            const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
            const uint64_t da = smem_desc_sw128(sa), db = smem_desc_sw128(sa + A_BYTES);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              // +32 bytes per K=16 step inside the 128-byte swizzled row
              tc_mma_f16(d_tmem, da + 2 * kk, db + 2 * kk, kIdesc, (ks > ks0 || kk > 0) ? 1u : 0u);
            }
            any = true;
            tc_commit(empty0 + 8 * stage);
            if (++stage == STAGES) { stage = 0; phase ^= 1u; }
          }
          if (ok) tc_commit(accf0 + 8 * buf);
        }
      }
      if (!ok && any) {
        // wait for the tensor core to finish everything issued before TMEM is freed
        tc_commit(drain);
        const uint64_t t0 = globaltimer();
        while (!mbar_try_wait(drain, 0) && globaltimer() - t0 < kWaitLimitNs) {}
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int ew = warp - 2;                  // 0..7
    const int quarter = warp & 3;             // TMEM lanes this warp may access
    const int col_half = ew >> 2;             // columns [0,128) or [128,256) of the tile
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    uint32_t chunk = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < p.num_tiles && ok; tile += gridDim.x) {
      int mb, nb;
      tile_coords(tile, p.num_m, p.num_n, mb, nb);
      int32_t acc[128];
#pragma unroll
      for (int j = 0; j < 128; ++j) acc[j] = 0;
      for (int c = 0; c < chunks_per_tile; ++c, ++chunk) {
        const uint32_t buf = chunk & 1u, use = chunk >> 1;
        // one lane polls, the warp follows: tcgen05.ld below needs a converged warp
        int got = 1;
        if (lane == 0) got = mbar_wait(accf0 + 8 * buf, use & 1u, ERR_WAIT_ACC_FULL, abort_flag) ? 1 : 0;
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) { ok = false; break; }
        tc_fence_after();
        const uint32_t t_base = tmem_base + lane_addr + buf * BN + col_half * 128;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(t_base + g * 32, r);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            // the FP32 value is an exact integer below 2^23: conversion is exact
            acc[g * 32 + j] += __float2int_rn(__uint_as_float(r[j]));
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acce0 + 8 * buf);
      }
      if (!ok) break;
      // ---- output: this thread owns row m, columns n0 .. n0+127
      const int m = mb * BM + quarter * 32 + lane;
      const int n0 = nb * BN + col_half * 128;
      if (m < p.M) {
        if constexpr (OUT < 0) {
          int32_t* orow = static_cast<int32_t*>(p.out) + static_cast<int64_t>(m) * p.ld_out;
#pragma unroll
          for (int j = 0; j < 128; ++j)
            if (n0 + j < p.N) orow[n0 + j] = acc[j];
        } else {
          using T = typename OutT<OUT>::T;
          constexpr int VEC = 16 / sizeof(T);
          const float sa = __ldg(p.a_scale + m);
          T* orow = static_cast<T*>(p.out) + static_cast<int64_t>(m) * p.ld_out;
#pragma unroll
          for (int j0 = 0; j0 < 128; j0 += VEC) {
            const int n = n0 + j0;
            if (p.out_vec && n + VEC <= p.N) {
              union { T v[VEC]; uint4 u; } pk;
#pragma unroll
              for (int j = 0; j < VEC; ++j) {
                const float y = __fmul_rn(__fmul_rn(static_cast<float>(acc[j0 + j]), sa),
                                          __ldg(p.w_scale + n + j));
                pk.v[j] = to_out<OUT>(y);
              }
              *reinterpret_cast<uint4*>(orow + n) = pk.u;
            } else {
#pragma unroll
              for (int j = 0; j < VEC; ++j) {
                if (n + j < p.N) {
                  const float y = __fmul_rn(__fmul_rn(static_cast<float>(acc[j0 + j]), sa),
                                            __ldg(p.w_scale + n + j));
                  orow[n + j] = to_out<OUT>(y);
                }
              }
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                 : "memory");
  }
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 2D map over an FP16 [rows][cols] matrix with pitch ld (elements), box
// [box_rows][64], 128-byte swizzle, zero fill outside the matrix.
static bool make_map(CUtensorMap* map, const void* base, int rows, int cols, int64_t ld, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

static int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

template <int OUT>
static cudaError_t launch(const CUtensorMap& ma, const CUtensorMap& mb, const Params& p, int grid,
                          cudaStream_t st) {
  static bool attr_set = false;   // per-process; same attribute value on every device
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(gemm_kernel<OUT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  gemm_kernel<OUT><<<grid, THREADS, SMEM_BYTES, st>>>(ma, mb, p);
  return cudaGetLastError();
}

static int validate_operands(const void* a_q, int64_t ld_aq, const void* w_q, int64_t ld_wq, int M,
                             int N, int K_p) {
  if (M < 0 || N < 0 || K_p <= 0 || K_p % CONVROT_BLOCK) return CONVROT_ERR_INVALID_ARG;
  if (K_p > CONVROT_MAX_KP) return CONVROT_ERR_UNSUPPORTED;
  if (ld_aq < K_p || ld_wq < K_p) return CONVROT_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return CONVROT_OK;
  if (!a_q || !w_q) return CONVROT_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(a_q) % 16 || reinterpret_cast<uintptr_t>(w_q) % 16 || ld_aq % 8 ||
      ld_wq % 8)
    return CONVROT_ERR_MISALIGNED;
  return CONVROT_OK;
}

static int run(int out_kind, const void* a_q, int64_t ld_aq, const float* a_scale, const void* w_q,
               int64_t ld_wq, const float* w_scale, int M, int N, int K_p, void* out, int64_t ld_out,
               size_t out_esize, cudaStream_t stream) {
  Params p;
  p.M = M;
  p.N = N;
  p.K_p = K_p;
  p.num_m = (M + BM - 1) / BM;
  p.num_n = (N + BN - 1) / BN;
  p.num_tiles = p.num_m * p.num_n;
  p.k_steps = K_p / BK;
  p.a_scale = a_scale;
  p.w_scale = w_scale;
  p.out = out;
  p.ld_out = ld_out;
  p.out_vec = (reinterpret_cast<uintptr_t>(out) % 16 == 0) && ((ld_out * static_cast<int64_t>(out_esize)) % 16 == 0);
  CUtensorMap ma, mb;
  if (!make_map(&ma, a_q, M, K_p, ld_aq, BM) || !make_map(&mb, w_q, N, K_p, ld_wq, BN))
    return CONVROT_ERR_CUDA;
  const int sms = sm_count();
  if (sms <= 0) return CONVROT_ERR_CUDA;
  const int grid = p.num_tiles < sms ? p.num_tiles : sms;
  cudaError_t e;
  switch (out_kind) {
    case CONVROT_BF16: e = launch<CONVROT_BF16>(ma, mb, p, grid, stream); break;
    case CONVROT_FP16: e = launch<CONVROT_FP16>(ma, mb, p, grid, stream); break;
    case CONVROT_FP32: e = launch<CONVROT_FP32>(ma, mb, p, grid, stream); break;
    default: e = launch<-1>(ma, mb, p, grid, stream); break;
  }
  return e == cudaSuccess ? CONVROT_OK : CONVROT_ERR_CUDA;
}

}  // namespace crgemm

using namespace crgemm;

extern "C" int convrot_gemm(const void* a_q, int64_t ld_aq, const float* a_scale, const void* w_q,
                            int64_t ld_wq, const float* w_scale, int M, int N, int K_p, void* out,
                            convrot_dtype out_dtype, int64_t ld_out, cudaStream_t stream) {
  if (out_dtype != CONVROT_BF16 && out_dtype != CONVROT_FP16 && out_dtype != CONVROT_FP32)
    return CONVROT_ERR_UNSUPPORTED;
  int st = validate_operands(a_q, ld_aq, w_q, ld_wq, M, N, K_p);
  if (st != CONVROT_OK) return st;
  if (ld_out < N) return CONVROT_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return CONVROT_OK;
  if (!a_scale || !w_scale || !out) return CONVROT_ERR_INVALID_ARG;
  const size_t es = out_dtype == CONVROT_FP32 ? 4 : 2;
  if (reinterpret_cast<uintptr_t>(out) % es || reinterpret_cast<uintptr_t>(a_scale) % 4 ||
      reinterpret_cast<uintptr_t>(w_scale) % 4)
    return CONVROT_ERR_MISALIGNED;
  return run(out_dtype, a_q, ld_aq, a_scale, w_q, ld_wq, w_scale, M, N, K_p, out, ld_out, es, stream);
}

extern "C" int convrot_gemm_i32(const void* a_q, int64_t ld_aq, const void* w_q, int64_t ld_wq, int M,
                                int N, int K_p, int32_t* acc, int64_t ld_acc, cudaStream_t stream) {
  int st = validate_operands(a_q, ld_aq, w_q, ld_wq, M, N, K_p);
  if (st != CONVROT_OK) return st;
  if (ld_acc < N) return CONVROT_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return CONVROT_OK;
  if (!acc) return CONVROT_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(acc) % 4) return CONVROT_ERR_MISALIGNED;
  return run(-1, a_q, ld_aq, nullptr, w_q, ld_wq, nullptr, M, N, K_p, acc, ld_acc, 4, stream);
}

extern "C" int convrot_device_error(cudaStream_t stream, int* code) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return CONVROT_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_error, sizeof(int)) != cudaSuccess) return CONVROT_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_error, &zero, sizeof(int)) != cudaSuccess) return CONVROT_ERR_CUDA;
  }
  if (code) *code = v;
  return v ? CONVROT_ERR_DEVICE_TIMEOUT : CONVROT_OK;
}
