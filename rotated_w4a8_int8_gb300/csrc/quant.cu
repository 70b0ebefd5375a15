// Kernels 1 and 2 of the ConvRot W4A8 layer and their C-ABI entry points.
//
//   convrot_prepare_weight: NVFP4 decode -> ConvRot256 rotation (FP32) -> row S8
//   convrot_quant_act:      (SwiGLU ->) (channel pre-scale ->) ConvRot256
//                           rotation (FP32) -> row S8
//
// Both follow the ComfyUI Turing Utils page (comfy.icu), node list, the entry
// on the ConvRot DiT / CLIP loaders reading native NVFP4 layers: paired
// ConvRot256 on activations and decoded NVFP4 weights, both operands
// zero-padded to whole 256-blocks, FP32 rotation, row-scaled S8 with a
// rounded FP32 scale reciprocal; pre-scales and SwiGLU before the rotation.
// SwiGLU follows the MiniMax-H3 explainer (modelpad.app), MLP section:
// gate, value = chunk(2); swish(gate) * value.
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>

#include "../../include/convrot.h"
#include "errors.h"
#include "rotate_quant.cuh"
#include "nvfp4.cuh"

// This file is compiled twice.  With CONVROT_QUANT_NORM = 0 it holds the
// kernels that write no code-norm bounds, the C-ABI entry points and the code
// widening; with CONVROT_QUANT_NORM = 1 only the kernels that also write the
// bounds and their launcher.  The bounds' sum of squares is a compile-time
// choice because, even when skipped at run time, it costs the register-bound
// weight kernel spills (a 30% slower kernel, measured) and the others time.
#ifndef CONVROT_QUANT_NORM
#define CONVROT_QUANT_NORM 0
#endif

namespace convrot {

// ------------------------------------------------------------------ loaders
enum : int { DT_BF16 = 0, DT_FP16 = 1, DT_FP32 = 2 };

// Raw storage words of the 32 elements [c0, c0 + 32) a thread owns in pass 1
// (rows 2p and 2p+1 of its block).  16-bit types: word k holds elements 2k,
// 2k+1; FP32: word k holds element k.
template <int DT>
struct Raw {
  static constexpr int N = (DT == DT_FP32) ? 32 : 16;
  uint32_t w[N];
};

template <int DT>
__device__ __forceinline__ uint32_t load_elem_bits(const char* row, int k) {
  if constexpr (DT == DT_FP32) return reinterpret_cast<const uint32_t*>(row)[k];
  else return reinterpret_cast<const uint16_t*>(row)[k];
}

// 32-byte read-only load (one full sector per thread).
__device__ __forceinline__ void ldg32B(const void* p, uint32_t* w) {
  asm("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
      : "l"(p));
}

// VEC: 0 = element loads, 1 = 16-byte loads, 2 = 32-byte loads (rows aligned
// to that size; a thread's 32 elements are contiguous).
template <int DT, int VEC>
__device__ __forceinline__ void load_raw(const char* row, int c0, int K, Raw<DT>& r) {
  if (c0 >= K) {
#pragma unroll
    for (int i = 0; i < Raw<DT>::N; ++i) r.w[i] = 0u;
    return;
  }
  if (VEC > 0 && c0 + 32 <= K) {
    constexpr int esz = (DT == DT_FP32) ? 4 : 2;
    const char* p = row + static_cast<size_t>(c0) * esz;
    if constexpr (VEC == 2) {
#pragma unroll
      for (int u = 0; u < Raw<DT>::N / 8; ++u) ldg32B(p + 32 * u, &r.w[8 * u]);
    } else {
#pragma unroll
      for (int u = 0; u < Raw<DT>::N / 4; ++u) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(p) + u);
        r.w[4 * u] = v.x; r.w[4 * u + 1] = v.y; r.w[4 * u + 2] = v.z; r.w[4 * u + 3] = v.w;
      }
    }
    return;
  }
  if constexpr (DT == DT_FP32) {
#pragma unroll
    for (int e = 0; e < 32; ++e) r.w[e] = (c0 + e < K) ? load_elem_bits<DT>(row, c0 + e) : 0u;
  } else {
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const uint32_t lo = (c0 + 2 * k < K) ? load_elem_bits<DT>(row, c0 + 2 * k) : 0u;
      const uint32_t hi = (c0 + 2 * k + 1 < K) ? load_elem_bits<DT>(row, c0 + 2 * k + 1) : 0u;
      r.w[k] = lo | (hi << 16);
    }
  }
}

// Element e (0..31) of a Raw as FP32.
template <int DT>
__device__ __forceinline__ float raw_elem(const Raw<DT>& r, int e) {
  if constexpr (DT == DT_FP32) {
    return __uint_as_float(r.w[e]);
  } else if constexpr (DT == DT_BF16) {
    const uint32_t w = r.w[e >> 1];
    return __uint_as_float((e & 1) ? (w & 0xffff0000u) : (w << 16));
  } else {
    const uint32_t w = r.w[e >> 1];
    return __half2float(__ushort_as_half(static_cast<unsigned short>((e & 1) ? (w >> 16) : (w & 0xffffu))));
  }
}

// Pass-1 pairs P[b] = (x[2p][b], x[2p+1][b]) = (elem b, elem 16 + b).
template <int DT>
__device__ __forceinline__ void pairs_from_raw(const Raw<DT>& r, float2 (&P)[16]) {
#pragma unroll
  for (int b = 0; b < 16; ++b) P[b] = make_float2(raw_elem<DT>(r, b), raw_elem<DT>(r, 16 + b));
}

// e^(-|g|) as 2^(-|g| log2 e) on the hardware base-2 exponential
// (ex2.approx.f32, not flushed: e stays subnormal, and g * e normal, for
// gates down to about -92).  Rounding the exponent -|g| log2 e costs up to
// about |g| * 2^-24 of relative error in e (a few ulp for ordinary gates, some
// tens near |g| = 88), on top of the instruction's own; a row's codes depend
// on h only up to its common scale.  Against the accurate expf the FFN-down
// SwiGLU kernel took 301.9 us instead of 313.9 us (same box, alternating
// order), and 522 of its 286 M codes moved by one.
__device__ __forceinline__ float exp_neg_abs(float g) {
  float r;
  asm("ex2.approx.f32 %0, %1;" : "=f"(r) : "f"(-fabsf(g) * 1.4426950408889634f));
  return r;
}

// Reciprocal of d in [1, 2] (MUFU, about 1 ulp).  Neither d nor 1/d is ever
// subnormal here, so flushing subnormals cannot change the result.
__device__ __forceinline__ float rcp_1to2(float d) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(d));
  return r;
}

// SwiGLU h = g * sigmoid(g) * v in FP32 (no intermediate rounding to the input
// dtype), in a form that never overflows.  With e = exp(-|g|) in (0, 1],
// sigmoid(g) = 1 / (1 + e) for g >= 0 and e / (1 + e) for g < 0, so
// h = (g >= 0 ? g : g * e) * (1 / (1 + e)) * v, and the divisor stays in
// [1, 2].  The direct g / (1 + exp(-g)) divides by an overflowing exp(-g)
// once g < -88.7, and a fast division returns 0 for divisors above 2^126
// (g < -87.3) even before that, where h is still a normal FP32 number.
// Below g = -87.3, e is subnormal and g * e stays normal down to g = -92.
template <int DT>
__device__ __forceinline__ void pairs_swiglu(const Raw<DT>& g, const Raw<DT>& v, float2 (&P)[16]) {
#pragma unroll
  for (int b = 0; b < 16; ++b) {
    const float2 gg = make_float2(raw_elem<DT>(g, b), raw_elem<DT>(g, 16 + b));
    const float2 vv = make_float2(raw_elem<DT>(v, b), raw_elem<DT>(v, 16 + b));
    const float2 e = make_float2(exp_neg_abs(gg.x), exp_neg_abs(gg.y));
    const float2 ge = mul2(gg, e);
    const float2 num = make_float2(gg.x >= 0.f ? gg.x : ge.x, gg.y >= 0.f ? gg.y : ge.y);
    const float2 d = add2(make_float2(1.0f, 1.0f), e);
    P[b] = mul2(mul2(num, make_float2(rcp_1to2(d.x), rcp_1to2(d.y))), vv);
  }
}

// ------------------------------------------------------------------ kernels
// Both kernels run one CTA per row.  Every load of the row is issued before
// any arithmetic.  Slot s (threads 8s .. 8s+7) rotates blocks s, s + S,
// s + 2S, ... (at most NBMAX) of the row.

// Raw input of one token row for this thread: the pass-1 chunks of its blocks.
template <int DT, bool SWIGLU, int NBMAX>
struct ActRaw {
  Raw<DT> g[NBMAX];
  Raw<DT> v[SWIGLU ? NBMAX : 1];
};

template <int DT, bool SWIGLU, int NBMAX, int VEC>
__device__ __forceinline__ void load_act_row(const char* xrow, int K, int blk0, int nloc, int S, int slot,
                                             int lane8, ActRaw<DT, SWIGLU, NBMAX>& r) {
  constexpr size_t esize = (DT == DT_FP32) ? 4 : 2;
#pragma unroll
  for (int i = 0; i < NBMAX; ++i) {
    const int li = slot + S * i;
    if (slot < S && li < nloc) {
      const int c0 = (blk0 + li) * kBlock + 32 * lane8;
      load_raw<DT, VEC>(xrow, c0, K, r.g[i]);
      if constexpr (SWIGLU) load_raw<DT, VEC>(xrow + static_cast<size_t>(K) * esize, c0, K, r.v[i]);
    }
  }
}

// Channel pre-scales p[c0 .. c0+31] applied to the pass-1 pairs
// P[b] = (elem b, elem 16 + b), four pairs at a time; nothing at or past K
// is read.
__device__ __forceinline__ void apply_pre_scale(const float* __restrict__ p, int c0, int K, float2 (&P)[16]) {
  if (c0 >= K) return;
  const bool full = c0 + 32 <= K;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float4 lo, hi;                       // elements 4j..4j+3 and 16+4j..16+4j+3
    if (full) {
      lo = __ldg(reinterpret_cast<const float4*>(p + c0 + 4 * j));
      hi = __ldg(reinterpret_cast<const float4*>(p + c0 + 16 + 4 * j));
    } else {
      auto at = [&](int e) { return (c0 + e < K) ? __ldg(p + c0 + e) : 0.f; };
      lo = make_float4(at(4 * j), at(4 * j + 1), at(4 * j + 2), at(4 * j + 3));
      hi = make_float4(at(16 + 4 * j), at(17 + 4 * j), at(18 + 4 * j), at(19 + 4 * j));
    }
    P[4 * j] = mul2(P[4 * j], make_float2(lo.x, hi.x));
    P[4 * j + 1] = mul2(P[4 * j + 1], make_float2(lo.y, hi.y));
    P[4 * j + 2] = mul2(P[4 * j + 2], make_float2(lo.z, hi.z));
    P[4 * j + 3] = mul2(P[4 * j + 3], make_float2(lo.w, hi.w));
  }
}

// One activation row from its raw input: (SwiGLU,) (channel pre-scale,)
// rotation, CTA absmax, scale and codes.  `red` is this row's reduction buffer.
template <int DT, bool SWIGLU, int NBMAX, bool PRESCALE, int SPLIT, bool NORM>
__device__ __forceinline__ void act_row(const ActRaw<DT, SWIGLU, NBMAX>& cur, int row, int K, int blk0,
                                        int nloc, int S, int slot, int lane8, char* my, float* red,
                                        float* xred, const float* pre_scale, void* q, int f16_codes,
                                        int64_t ld_q, float* scale, float* norm) {
  BlockCols c[NBMAX];
  float amax = 0.f, ss = 0.f;                    // ss: sum of squares, for the norm bound (NORM)
#pragma unroll
  for (int i = 0; i < NBMAX; ++i) {
    const int li = slot + S * i, blk = blk0 + li;
    const bool active = (slot < S) && (li < nloc);
    float2 P[16];
    if (active) {
      if constexpr (SWIGLU) pairs_swiglu<DT>(cur.g[i], cur.v[SWIGLU ? i : 0], P);
      else pairs_from_raw<DT>(cur.g[i], P);
      if constexpr (PRESCALE) apply_pre_scale(pre_scale, blk * kBlock + 32 * lane8, K, P);
    }
    rotate_block(P, c[i], my, lane8, active);
    if (active) {
      amax = absmax_cols(amax, c[i]);
      if constexpr (NORM) ss = sumsq_cols(ss, c[i]);
    }
  }
  // z = x H; the rotated row is z / 16 (exact), so its absmax is amax / 16
  const float hsk = 0.5001f * sqrtf(static_cast<float>(((K + kBlock - 1) / kBlock) * kBlock));
  const RowQuant rq = SPLIT == 1 ? cta_rowquant(amax, ss, NORM, red, 0.0625f, hsk)
                                 : cluster_rowquant(amax, ss, NORM, red, xred, 0.0625f, hsk);
  if (threadIdx.x == 0 && blk0 == 0) {
    scale[row] = rq.s;
    if constexpr (NORM) norm[row] = SPLIT == 1 ? red[18] : xred[4];
  }
  void* qrow = static_cast<char*>(q) + static_cast<size_t>(row) * ld_q * (f16_codes ? 2 : 1);
  const float mult = rq.r * 0.0625f;           // fp32(z * (r / 16)) == fp32((z / 16) * r)
#pragma unroll
  for (int i = 0; i < NBMAX; ++i) {
    const int li = slot + S * i;
    if (slot < S && li < nloc) {
      scale_cols(c[i], mult);
      store_codes<SWIGLU>(qrow, f16_codes, blk0 + li, lane8, c[i]);
    }
  }
}

// L2 prefetch of a later activation row.  Each CTA reads its row once, at its start,
// and then computes with nothing in flight; the loads of the CTAs resident
// on an SM alone do not keep HBM busy.  So every CTA also prefetches into
// L2 the row that a CTA about kPfBytes of input later will read (one
// prefetch.global.L2 per 128-byte line, spread over the threads), and that
// CTA then finds its row in L2.  The distance is kPfBytes / row bytes rows,
// between 32 and 512: long enough to cover the HBM latency, short enough
// that the prefetched rows stay far below the L2 size.  It is computed on
// the host: a 64-bit division in every thread would cost more than the
// prefetch itself.
constexpr size_t kPfBytes = size_t(8) << 20;

static int prefetch_distance(size_t row_bytes) {
  const size_t d = kPfBytes / (row_bytes > 0 ? row_bytes : 1);
  return static_cast<int>(d < 32 ? 32 : d > 512 ? 512 : d);
}

__device__ __forceinline__ void l2_prefetch(const char* p, size_t bytes) {
  for (size_t off = static_cast<size_t>(threadIdx.x) * 128; off < bytes; off += static_cast<size_t>(blockDim.x) * 128)
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p + off));
}

// Kernel 2: one CTA per activation row, or (SPLIT == 2) a cluster of two
// CTAs per row, each owning half of the row's blocks.
template <int DT, bool SWIGLU, int NBMAX, int VEC, bool PRESCALE, int SPLIT, bool NORM>
__device__ __forceinline__ void quant_act_row(const void* __restrict__ x, int64_t ld_x, int M, int K, int nblocks,
                                              int S, int pf_dist, const float* __restrict__ pre_scale,
                                              void* __restrict__ q, int f16_codes, int64_t ld_q,
                                              float* __restrict__ scale, float* __restrict__ norm) {
  extern __shared__ __align__(16) char smem[];
  float* red = reinterpret_cast<float*>(smem + S * kSlotBytes);   // row reduction slots
  float* xred = red + 16;                                         // cluster exchange slots
  const int slot = threadIdx.x >> 3, lane8 = threadIdx.x & 7;
  constexpr size_t esize = (DT == DT_FP32) ? 4 : 2;
  const int row = blockIdx.x / SPLIT, part = blockIdx.x % SPLIT;
  const int nbl = (nblocks + SPLIT - 1) / SPLIT;
  const int blk0 = part * nbl, nloc = min(nbl, nblocks - blk0);
  ActRaw<DT, SWIGLU, NBMAX> cur;
  load_act_row<DT, SWIGLU, NBMAX, VEC>(static_cast<const char*>(x) + static_cast<size_t>(row) * ld_x * esize,
                                       K, blk0, nloc, S, slot, lane8, cur);
  {
    // this CTA's share (its part of the row) of a later row
    const size_t rb = static_cast<size_t>(SWIGLU ? 2 * K : K) * esize;
    const int later = row + pf_dist;
    if (later < M) {
      const size_t share = (rb + SPLIT - 1) / SPLIT, b0 = part * share, b1 = min(rb, b0 + share);
      l2_prefetch(static_cast<const char*>(x) + static_cast<size_t>(later) * ld_x * esize + b0, b1 - b0);
    }
  }
  act_row<DT, SWIGLU, NBMAX, PRESCALE, SPLIT, NORM>(cur, row, K, blk0, nloc, S, slot, lane8, smem + slot * kSlotBytes,
                                              red, xred, pre_scale, q, f16_codes, ld_q, scale, norm);
  if constexpr (SPLIT == 2) cluster_exit_wait();
}

template <int DT, bool SWIGLU, int NBMAX, int VEC, bool PRESCALE, int SPLIT, bool NORM>
__global__ void __launch_bounds__(kMaxThreads)
quant_act_kernel(const void* __restrict__ x, int64_t ld_x, int M, int K, int nblocks, int S, int pf_dist,
                 const float* __restrict__ pre_scale, void* __restrict__ q, int f16_codes, int64_t ld_q,
                 float* __restrict__ scale, float* __restrict__ norm) {
  quant_act_row<DT, SWIGLU, NBMAX, VEC, PRESCALE, SPLIT, NORM>(x, ld_x, M, K, nblocks, S, pf_dist, pre_scale, q,
                                                               f16_codes, ld_q, scale, norm);
}

// The plain single-CTA form (no SwiGLU, one block per slot) held to 48
// registers measured faster: QKV activations 76.5 -> 74.4 us (same box,
// alternating order; 42 registers measured slower), and 86.7 -> 84.3 us with
// the norm bound's sum of squares.  ncu reports the same register limit (6
// CTAs of a 21-block row per SM) for the 48-register form, so the gain is in
// the schedule, not the occupancy.  The other forms keep the 512-thread
// launch bound alone: held to 48 registers, the SwiGLU form spills and ran
// 25% slower.
template <int DT, int VEC, bool PRESCALE, bool NORM>
__global__ void __maxnreg__(48)
quant_act_kernel_r48(const void* __restrict__ x, int64_t ld_x, int M, int K, int nblocks, int S, int pf_dist,
                     const float* __restrict__ pre_scale, void* __restrict__ q, int f16_codes, int64_t ld_q,
                     float* __restrict__ scale, float* __restrict__ norm) {
  quant_act_row<DT, false, 1, VEC, PRESCALE, 1, NORM>(x, ld_x, M, K, nblocks, S, pf_dist, pre_scale, q, f16_codes,
                                                      ld_q, scale, norm);
}

// Raw NVFP4 input of one weight row for this thread.
template <int NBMAX>
struct WRaw {
  uint2 w0[NBMAX], w1[NBMAX];
  uint16_t sc[NBMAX];
};

template <int NBMAX, bool W16>
__device__ __forceinline__ void load_weight_row(const uint8_t* w_fp4, const uint8_t* w_sf, int row, int K,
                                                int K_s, int blk0, int nloc, int S, int slot, int lane8,
                                                WRaw<NBMAX>& r) {
  const uint8_t* prow = w_fp4 + static_cast<size_t>(row) * (K_s >> 1);
  const uint8_t* srow = w_sf + static_cast<size_t>(row) * (K_s >> 4);
#pragma unroll
  for (int i = 0; i < NBMAX; ++i) {
    const int li = slot + S * i;
    if (slot < S && li < nloc)
      load_nvfp4_raw<W16>(prow, srow, (blk0 + li) * kBlock + 32 * lane8, K, K_s, r.w0[i], r.w1[i], r.sc[i]);
  }
}

// One weight row from its raw input: decode, rotation, tensor scale, CTA
// absmax, scale and codes.
template <int NBMAX, int SPLIT, bool NORM>
__device__ __forceinline__ void weight_row(const WRaw<NBMAX>& r, int row, int K, int blk0, int nloc, int S,
                                           int slot, int lane8, float t16, char* my, float* red, float* xred,
                                           void* q, int f16_codes, int64_t ld_q, float* scale, float* norm) {
  BlockCols c[NBMAX];
  float amax = 0.f, ss = 0.f;                    // ss: sum of squares, for the norm bound (NORM)
#pragma unroll
  for (int i = 0; i < NBMAX; ++i) {
    const int li = slot + S * i, blk = blk0 + li;
    const bool active = (slot < S) && (li < nloc);
    float2 P[16];
    if (active) decode_nvfp4_pairs(r.w0[i], r.w1[i], r.sc[i], blk * kBlock + 32 * lane8, K, P);
    rotate_block(P, c[i], my, lane8, active);
    if (active) {
      scale_cols(c[i], t16);                   // rotated weight = fp32(z * t / 16)
      amax = absmax_cols(amax, c[i]);
      if constexpr (NORM) ss = sumsq_cols(ss, c[i]);
    }
  }
  const float hsk = 0.5001f * sqrtf(static_cast<float>(((K + kBlock - 1) / kBlock) * kBlock));
  const RowQuant rq = SPLIT == 1 ? cta_rowquant(amax, ss, NORM, red, 1.0f, hsk)
                                 : cluster_rowquant(amax, ss, NORM, red, xred, 1.0f, hsk);
  if (threadIdx.x == 0 && blk0 == 0) {
    scale[row] = rq.s;
    if constexpr (NORM) norm[row] = SPLIT == 1 ? red[18] : xred[4];
  }
  void* qrow = static_cast<char*>(q) + static_cast<size_t>(row) * ld_q * (f16_codes ? 2 : 1);
#pragma unroll
  for (int i = 0; i < NBMAX; ++i) {
    const int li = slot + S * i;
    if (slot < S && li < nloc) {
      scale_cols(c[i], rq.r);
      store_codes<false>(qrow, f16_codes, blk0 + li, lane8, c[i]);
    }
  }
}

// Kernel 1: one CTA per weight row, or (SPLIT == 2) a cluster of two CTAs
// per row, each owning half of the row's blocks.
template <int NBMAX, bool W16, int SPLIT, bool NORM>
__device__ __forceinline__ void prepare_weight_row(const uint8_t* __restrict__ w_fp4, const uint8_t* __restrict__ w_sf,
                                                   const float* __restrict__ tscale, int N, int K, int K_s,
                                                   int nblocks, int S, void* __restrict__ q, int f16_codes,
                                                   int64_t ld_q, float* __restrict__ scale, float* __restrict__ norm) {
  extern __shared__ __align__(16) char smem[];
  float* red = reinterpret_cast<float*>(smem + S * kSlotBytes);
  float* xred = red + 16;
  const int slot = threadIdx.x >> 3, lane8 = threadIdx.x & 7;
  const float t16 = __ldg(tscale) * 0.0625f;  // t / 16 is exact
  const int row = blockIdx.x / SPLIT, part = blockIdx.x % SPLIT;
  const int nbl = (nblocks + SPLIT - 1) / SPLIT;
  const int blk0 = part * nbl, nloc = min(nbl, nblocks - blk0);
  WRaw<NBMAX> r0;
  load_weight_row<NBMAX, W16>(w_fp4, w_sf, row, K, K_s, blk0, nloc, S, slot, lane8, r0);
  weight_row<NBMAX, SPLIT, NORM>(r0, row, K, blk0, nloc, S, slot, lane8, t16, smem + slot * kSlotBytes, red, xred, q,
                                 f16_codes, ld_q, scale, norm);
  if constexpr (SPLIT == 2) cluster_exit_wait();
}

// With one block per slot the kernel is held to 40 registers (at least 3 CTAs
// of 512 threads per SM): 7 CTAs of a 21-block row then fit an SM instead of
// 6, for a 4-byte spill, which measured 2-6% faster.  Two blocks per slot need
// their registers.
template <int NBMAX, bool W16, int SPLIT, bool NORM>
__global__ void __launch_bounds__(kMaxThreads, NBMAX == 1 ? 3 : 1)
prepare_weight_kernel(const uint8_t* __restrict__ w_fp4, const uint8_t* __restrict__ w_sf,
                      const float* __restrict__ tscale, int N, int K, int K_s, int nblocks, int S,
                      void* __restrict__ q, int f16_codes, int64_t ld_q, float* __restrict__ scale,
                      float* __restrict__ norm) {
  prepare_weight_row<NBMAX, W16, SPLIT, NORM>(w_fp4, w_sf, tscale, N, K, K_s, nblocks, S, q, f16_codes, ld_q, scale,
                                              norm);
}

// Short rows (at most kShortRowBlocks blocks, one per slot) held to 48
// registers instead: no spill (ncu: 6 CTAs of a 21-block row per SM by
// registers).  Measured on one box (alternating order): 21-block rows 82.1 ->
// 76.4 us, and 91.9 -> 88.7 us with the norm bound's sum of squares (which
// spills at 40 registers); on 56-block rows the 48-register form was even
// (62.1 -> 62.8 us) and, with the sum of squares, 13% slower, so longer rows
// keep the 40-register kernel.
constexpr int kShortRowBlocks = 32;
template <bool W16, int SPLIT, bool NORM>
__global__ void __maxnreg__(48)
prepare_weight_kernel_r48(const uint8_t* __restrict__ w_fp4, const uint8_t* __restrict__ w_sf,
                          const float* __restrict__ tscale, int N, int K, int K_s, int nblocks, int S,
                          void* __restrict__ q, int f16_codes, int64_t ld_q, float* __restrict__ scale,
                          float* __restrict__ norm) {
  prepare_weight_row<1, W16, SPLIT, NORM>(w_fp4, w_sf, tscale, N, K, K_s, nblocks, S, q, f16_codes, ld_q, scale,
                                          norm);
}

// ------------------------------------------------------------------ launch geometry
struct RowGeometry {
  int nblocks;     // 256-blocks per row
  int split;       // CTAs per row (1, or 2 in a cluster)
  int nbmax;       // blocks per slot (1 or 2)
  int S;           // slots (8 threads each) per CTA
  int threads;
  size_t smem;
};

// Rows of more than `split_above` blocks go to two CTAs of a cluster, each
// with half of the blocks; otherwise one CTA holds the row.  A slot takes
// one block, or two when a CTA's share exceeds 64 blocks (K_p <= 65536).
// Splitting halves a row's latency but, at one block per slot, holds fewer
// rows per SM than two blocks per slot: the activation rows gain from it
// above 64 blocks, the shorter weight rows only where two blocks per slot
// no longer fit one CTA (above 128).
[[maybe_unused]] static bool row_geometry(int K_p, int split_above, RowGeometry* g) {
  g->nblocks = K_p / kBlock;
  g->split = g->nblocks > split_above ? 2 : 1;
  const int nbl = (g->nblocks + g->split - 1) / g->split;
  const int nb = (nbl + kMaxSlots - 1) / kMaxSlots;
  if (nb > 2) return false;
  g->nbmax = nb;
  g->S = (nbl + nb - 1) / nb;
  g->threads = ((kSlotThreads * g->S + 31) / 32) * 32;
  g->smem = static_cast<size_t>(g->S) * kSlotBytes + kRedFloats * sizeof(float);
  return true;
}

template <typename Kern>
static cudaError_t prep_smem(Kern k, size_t smem) {
  if (smem <= 48 * 1024) return cudaSuccess;
  return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
}

// Launches `k` over `rows` rows: one CTA per row, or clusters of two.
template <typename Kern, typename... Args>
static cudaError_t launch_rows(Kern k, const RowGeometry& g, int rows, cudaStream_t st, Args... args) {
  cudaError_t e = prep_smem(k, g.smem);
  if (e != cudaSuccess) return e;
  if (g.split == 1) {
    k<<<rows, g.threads, g.smem, st>>>(args...);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(rows) * 2u);
  cfg.blockDim = dim3(g.threads);
  cfg.dynamicSmemBytes = g.smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, args...);
}

template <int DT, bool SWIGLU, int VEC, int NB, int SPLIT, bool NORM>
static cudaError_t launch_act_cfg(const RowGeometry& g, int M, const void* x, int64_t ld_x, int K,
                                  const float* ps, void* q, int f16, int64_t ld_q, float* scale, float* norm,
                                  cudaStream_t st) {
  const int pf = prefetch_distance(static_cast<size_t>(SWIGLU ? 2 * K : K) * (DT == DT_FP32 ? 4 : 2));
  if constexpr (!SWIGLU && NB == 1 && SPLIT == 1) {
    auto k = ps ? quant_act_kernel_r48<DT, VEC, true, NORM> : quant_act_kernel_r48<DT, VEC, false, NORM>;
    return launch_rows(k, g, M, st, x, ld_x, M, K, g.nblocks, g.S, pf, ps, q, f16, ld_q, scale, norm);
  } else {
    auto k = ps ? quant_act_kernel<DT, SWIGLU, NB, VEC, true, SPLIT, NORM>
                : quant_act_kernel<DT, SWIGLU, NB, VEC, false, SPLIT, NORM>;
    return launch_rows(k, g, M, st, x, ld_x, M, K, g.nblocks, g.S, pf, ps, q, f16, ld_q, scale, norm);
  }
}

template <int DT, bool SWIGLU, int VEC, bool NORM>
static cudaError_t launch_act_dt(const RowGeometry& g, int M, const void* x, int64_t ld_x, int K,
                                 const float* ps, void* q, int f16, int64_t ld_q, float* scale, float* norm,
                                 cudaStream_t st) {
  if (g.split == 1)
    return launch_act_cfg<DT, SWIGLU, VEC, 1, 1, NORM>(g, M, x, ld_x, K, ps, q, f16, ld_q, scale, norm, st);
  if (g.nbmax == 1)
    return launch_act_cfg<DT, SWIGLU, VEC, 1, 2, NORM>(g, M, x, ld_x, K, ps, q, f16, ld_q, scale, norm, st);
  return launch_act_cfg<DT, SWIGLU, VEC, 2, 2, NORM>(g, M, x, ld_x, K, ps, q, f16, ld_q, scale, norm, st);
}

template <int DT, bool NORM>
static cudaError_t launch_act(const RowGeometry& g, int M, const void* x, int64_t ld_x, int K,
                              bool swiglu, int vec, const float* ps, void* q, int f16, int64_t ld_q,
                              float* scale, float* norm, cudaStream_t st) {
  if (swiglu) {
    switch (vec) {
      case 2: return launch_act_dt<DT, true, 2, NORM>(g, M, x, ld_x, K, ps, q, f16, ld_q, scale, norm, st);
      case 1: return launch_act_dt<DT, true, 1, NORM>(g, M, x, ld_x, K, ps, q, f16, ld_q, scale, norm, st);
      default: return launch_act_dt<DT, true, 0, NORM>(g, M, x, ld_x, K, ps, q, f16, ld_q, scale, norm, st);
    }
  }
  switch (vec) {
    case 2: return launch_act_dt<DT, false, 2, NORM>(g, M, x, ld_x, K, ps, q, f16, ld_q, scale, norm, st);
    case 1: return launch_act_dt<DT, false, 1, NORM>(g, M, x, ld_x, K, ps, q, f16, ld_q, scale, norm, st);
    default: return launch_act_dt<DT, false, 0, NORM>(g, M, x, ld_x, K, ps, q, f16, ld_q, scale, norm, st);
  }
}

template <bool W16, int NB, int SPLIT, bool NORM>
static cudaError_t launch_weight_cfg(const RowGeometry& g, int N, const uint8_t* w_fp4, const uint8_t* w_sf,
                                     const float* t, int K, int K_s, void* q, int f16, int64_t ld_q,
                                     float* scale, float* norm, cudaStream_t st) {
  if constexpr (NB == 1 && SPLIT == 1) {
    if (g.nblocks <= kShortRowBlocks)
      return launch_rows(prepare_weight_kernel_r48<W16, SPLIT, NORM>, g, N, st, w_fp4, w_sf, t, N, K, K_s, g.nblocks,
                         g.S, q, f16, ld_q, scale, norm);
  }
  return launch_rows(prepare_weight_kernel<NB, W16, SPLIT, NORM>, g, N, st, w_fp4, w_sf, t, N, K, K_s, g.nblocks,
                     g.S, q, f16, ld_q, scale, norm);
}

template <bool W16, bool NORM>
static cudaError_t launch_weight(const RowGeometry& g, int N, const uint8_t* w_fp4, const uint8_t* w_sf,
                                 const float* t, int K, int K_s, void* q, int f16, int64_t ld_q, float* scale,
                                 float* norm, cudaStream_t st) {
  if (g.split == 1)
    return g.nbmax == 1
               ? launch_weight_cfg<W16, 1, 1, NORM>(g, N, w_fp4, w_sf, t, K, K_s, q, f16, ld_q, scale, norm, st)
               : launch_weight_cfg<W16, 2, 1, NORM>(g, N, w_fp4, w_sf, t, K, K_s, q, f16, ld_q, scale, norm, st);
  if (g.nbmax == 1)
    return launch_weight_cfg<W16, 1, 2, NORM>(g, N, w_fp4, w_sf, t, K, K_s, q, f16, ld_q, scale, norm, st);
  return launch_weight_cfg<W16, 2, 2, NORM>(g, N, w_fp4, w_sf, t, K, K_s, q, f16, ld_q, scale, norm, st);
}

// The launchers of the two objects this file compiles to: *_plain writes no
// norm bounds, *_norm writes them to `norm`.
cudaError_t launch_act_plain(const RowGeometry& g, int dt, int M, const void* x, int64_t ld_x, int K, bool swiglu,
                             int vec, const float* ps, void* q, int f16, int64_t ld_q, float* scale, float* norm,
                             cudaStream_t st);
cudaError_t launch_act_norm(const RowGeometry& g, int dt, int M, const void* x, int64_t ld_x, int K, bool swiglu,
                            int vec, const float* ps, void* q, int f16, int64_t ld_q, float* scale, float* norm,
                            cudaStream_t st);
cudaError_t launch_weight_plain(const RowGeometry& g, bool w16, int N, const uint8_t* w_fp4, const uint8_t* w_sf,
                                const float* t, int K, int K_s, void* q, int f16, int64_t ld_q, float* scale,
                                float* norm, cudaStream_t st);
cudaError_t launch_weight_norm(const RowGeometry& g, bool w16, int N, const uint8_t* w_fp4, const uint8_t* w_sf,
                               const float* t, int K, int K_s, void* q, int f16, int64_t ld_q, float* scale,
                               float* norm, cudaStream_t st);

template <bool NORM>
static cudaError_t launch_act_any(const RowGeometry& g, int dt, int M, const void* x, int64_t ld_x, int K,
                                  bool swiglu, int vec, const float* ps, void* q, int f16, int64_t ld_q,
                                  float* scale, float* norm, cudaStream_t st) {
  switch (dt) {
    case DT_BF16: return launch_act<DT_BF16, NORM>(g, M, x, ld_x, K, swiglu, vec, ps, q, f16, ld_q, scale, norm, st);
    case DT_FP16: return launch_act<DT_FP16, NORM>(g, M, x, ld_x, K, swiglu, vec, ps, q, f16, ld_q, scale, norm, st);
    default: return launch_act<DT_FP32, NORM>(g, M, x, ld_x, K, swiglu, vec, ps, q, f16, ld_q, scale, norm, st);
  }
}

template <bool NORM>
static cudaError_t launch_weight_any(const RowGeometry& g, bool w16, int N, const uint8_t* w_fp4,
                                     const uint8_t* w_sf, const float* t, int K, int K_s, void* q, int f16,
                                     int64_t ld_q, float* scale, float* norm, cudaStream_t st) {
  return w16 ? launch_weight<true, NORM>(g, N, w_fp4, w_sf, t, K, K_s, q, f16, ld_q, scale, norm, st)
             : launch_weight<false, NORM>(g, N, w_fp4, w_sf, t, K, K_s, q, f16, ld_q, scale, norm, st);
}

#if CONVROT_QUANT_NORM
cudaError_t launch_act_norm(const RowGeometry& g, int dt, int M, const void* x, int64_t ld_x, int K, bool swiglu,
                            int vec, const float* ps, void* q, int f16, int64_t ld_q, float* scale, float* norm,
                            cudaStream_t st) {
  return launch_act_any<true>(g, dt, M, x, ld_x, K, swiglu, vec, ps, q, f16, ld_q, scale, norm, st);
}
cudaError_t launch_weight_norm(const RowGeometry& g, bool w16, int N, const uint8_t* w_fp4, const uint8_t* w_sf,
                               const float* t, int K, int K_s, void* q, int f16, int64_t ld_q, float* scale,
                               float* norm, cudaStream_t st) {
  return launch_weight_any<true>(g, w16, N, w_fp4, w_sf, t, K, K_s, q, f16, ld_q, scale, norm, st);
}
#else
cudaError_t launch_act_plain(const RowGeometry& g, int dt, int M, const void* x, int64_t ld_x, int K, bool swiglu,
                             int vec, const float* ps, void* q, int f16, int64_t ld_q, float* scale, float* norm,
                             cudaStream_t st) {
  return launch_act_any<false>(g, dt, M, x, ld_x, K, swiglu, vec, ps, q, f16, ld_q, scale, norm, st);
}
cudaError_t launch_weight_plain(const RowGeometry& g, bool w16, int N, const uint8_t* w_fp4, const uint8_t* w_sf,
                                const float* t, int K, int K_s, void* q, int f16, int64_t ld_q, float* scale,
                                float* norm, cudaStream_t st) {
  return launch_weight_any<false>(g, w16, N, w_fp4, w_sf, t, K, K_s, q, f16, ld_q, scale, norm, st);
}
#endif

}  // namespace convrot

#if !CONVROT_QUANT_NORM
using namespace convrot;

extern "C" int convrot_quant_act(const void* x, convrot_dtype x_dtype, int64_t ld_x, int M, int K,
                                 int swiglu, const float* pre_scale, void* a_q, convrot_codes fmt,
                                 int64_t ld_aq, float* a_scale, float* a_norm, cudaStream_t stream) {
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
  if (reinterpret_cast<uintptr_t>(a_q) % (fmt == CONVROT_CODES_F16 ? 4 : 2) || ld_aq % 2)
    return CONVROT_ERR_MISALIGNED;
  if (reinterpret_cast<uintptr_t>(a_scale) % 4 || reinterpret_cast<uintptr_t>(pre_scale) % 16 ||
      reinterpret_cast<uintptr_t>(a_norm) % 4)
    return CONVROT_ERR_MISALIGNED;
  // vector paths: every row start and the value half (SwiGLU) aligned to 32 or 16 bytes
  auto aligned = [&](int64_t a) {
    return (reinterpret_cast<uintptr_t>(x) % a == 0) && ((ld_x * static_cast<int64_t>(esize)) % a == 0) &&
           (!swiglu || (static_cast<int64_t>(K) * esize) % a == 0);
  };
  const int vec = aligned(32) ? 2 : aligned(16) ? 1 : 0;
  RowGeometry g;
  if (!row_geometry(K_p, kMaxSlots, &g)) return CONVROT_ERR_UNSUPPORTED;
  const int f16 = fmt == CONVROT_CODES_F16;
  const int dt = x_dtype == CONVROT_BF16 ? DT_BF16 : x_dtype == CONVROT_FP16 ? DT_FP16 : DT_FP32;
  const cudaError_t e =
      a_norm ? launch_act_norm(g, dt, M, x, ld_x, K, swiglu != 0, vec, pre_scale, a_q, f16, ld_aq, a_scale, a_norm,
                               stream)
             : launch_act_plain(g, dt, M, x, ld_x, K, swiglu != 0, vec, pre_scale, a_q, f16, ld_aq, a_scale, nullptr,
                                stream);
  return e == cudaSuccess ? CONVROT_OK : convrot::record_cuda_error("quant_act launch", e);
}

extern "C" int convrot_prepare_weight(const uint8_t* w_fp4, const uint8_t* w_sf,
                                      const float* w_tensor_scale, int N, int K, void* w_q,
                                      convrot_codes fmt, int64_t ld_wq, float* w_scale, float* w_norm,
                                      cudaStream_t stream) {
  if (N < 0 || K <= 0) return CONVROT_ERR_INVALID_ARG;
  if (fmt != CONVROT_CODES_S8 && fmt != CONVROT_CODES_F16) return CONVROT_ERR_UNSUPPORTED;
  const int K_p = convrot_padded_k(K);
  if (K_p > CONVROT_MAX_KP) return CONVROT_ERR_UNSUPPORTED;
  if (ld_wq < K_p) return CONVROT_ERR_INVALID_ARG;
  if (N == 0) return CONVROT_OK;
  if (!w_fp4 || !w_sf || !w_tensor_scale || !w_q || !w_scale) return CONVROT_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(w_fp4) % 8 || reinterpret_cast<uintptr_t>(w_tensor_scale) % 4 ||
      reinterpret_cast<uintptr_t>(w_scale) % 4 || reinterpret_cast<uintptr_t>(w_norm) % 4)
    return CONVROT_ERR_MISALIGNED;
  if (reinterpret_cast<uintptr_t>(w_q) % (fmt == CONVROT_CODES_F16 ? 4 : 2) || ld_wq % 2)
    return CONVROT_ERR_MISALIGNED;
  RowGeometry g;
  if (!row_geometry(K_p, 2 * kMaxSlots, &g)) return CONVROT_ERR_UNSUPPORTED;
  const int K_s = ((K + 15) / 16) * 16;
  const int f16 = fmt == CONVROT_CODES_F16;
  // one 16-byte load per thread when every packed row starts 16-byte aligned
  const bool w16 = (reinterpret_cast<uintptr_t>(w_fp4) % 16 == 0) && ((K_s / 2) % 16 == 0);
  const cudaError_t e =
      w_norm ? launch_weight_norm(g, w16, N, w_fp4, w_sf, w_tensor_scale, K, K_s, w_q, f16, ld_wq, w_scale, w_norm,
                                  stream)
             : launch_weight_plain(g, w16, N, w_fp4, w_sf, w_tensor_scale, K, K_s, w_q, f16, ld_wq, w_scale, nullptr,
                                   stream);
  return e == cudaSuccess ? CONVROT_OK : convrot::record_cuda_error("prepare_weight launch", e);
}

// ------------------------------------------------------------------ S8 -> FP16 code widening
// W8A8 with resident weights (the page's W8A8 comparison runs on these same
// rotated S8 weights derived from NVFP4): weights kept as 1-byte S8 codes are
// widened to the FP16-held codes the GEMM reads.  Each thread converts 16
// codes (one 16-byte load, two 16-byte stores); rows and pitches must keep
// those accesses aligned.
namespace convrot {
__global__ void __launch_bounds__(256)
widen_codes_kernel(const int8_t* __restrict__ src, int64_t ld_src, int rows, int cols,
                   __half* __restrict__ dst, int64_t ld_dst) {
  const int per_row = cols / 16;
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= static_cast<int64_t>(rows) * per_row) return;
  const int r = static_cast<int>(i / per_row), c = static_cast<int>(i % per_row) * 16;
  const uint4 v = __ldg(reinterpret_cast<const uint4*>(src + r * ld_src + c));
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t h[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t word = w[j >> 1] >> (16 * (j & 1));
    const int lo = static_cast<int8_t>(word & 0xffu), hi = static_cast<int8_t>((word >> 8) & 0xffu);
    const __half2 p = __halves2half2(__int2half_rn(lo), __int2half_rn(hi));
    h[j] = *reinterpret_cast<const uint32_t*>(&p);
  }
  uint4* d = reinterpret_cast<uint4*>(dst + r * ld_dst + c);
  d[0] = make_uint4(h[0], h[1], h[2], h[3]);
  d[1] = make_uint4(h[4], h[5], h[6], h[7]);
}
}  // namespace convrot

extern "C" int convrot_widen_codes(const int8_t* src, int64_t ld_src, int rows, int cols, void* dst,
                                   int64_t ld_dst, cudaStream_t stream) {
  if (rows < 0 || cols < 0 || cols % 16 || ld_src < cols || ld_dst < cols) return CONVROT_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return CONVROT_OK;
  if (!src || !dst) return CONVROT_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(src) % 16 || reinterpret_cast<uintptr_t>(dst) % 16 || ld_src % 16 ||
      ld_dst % 8)
    return CONVROT_ERR_MISALIGNED;
  const int64_t n = static_cast<int64_t>(rows) * (cols / 16);
  const int64_t blocks = (n + 255) / 256;
  if (blocks > 0x7fffffff) return CONVROT_ERR_UNSUPPORTED;
  widen_codes_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(src, ld_src, rows, cols,
                                                                        static_cast<__half*>(dst), ld_dst);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? CONVROT_OK : convrot::record_cuda_error("widen_codes launch", e);
}
#endif  // !CONVROT_QUANT_NORM
