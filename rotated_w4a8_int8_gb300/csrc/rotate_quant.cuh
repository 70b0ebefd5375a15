// Shared device code of the two ConvRot256 rotation + row-scaled S8 kernels.
//
// One CTA owns one row.  The padded row is split into 256-element blocks;
// a group of 8 threads ("slot") rotates one block at a time.  The Sylvester
// Walsh-Hadamard matrix factorises as H_256 = H_16 (x) H_16 over the index
// j = 16 a + b (a: block "row", b: block "column"), so the rotation is two
// 16-point passes with one transpose through shared memory:
//
//   pass 1: thread p holds rows 2p and 2p+1 as 16 FP32 pairs
//           P[b] = (x[2p][b], x[2p+1][b]) and transforms over b -- every
//           butterfly is one packed FP32x2 add or sub;
//   transpose: P[b] goes to shared memory as 8-byte units, rows padded to 18
//           units so that both sides use base + immediate addresses and the
//           16-byte reads are free of bank conflicts;
//   pass 2: thread q reads columns 2q and 2q+1 as pairs U[p] = (x[2p][2q],
//           x[2p+1][2q]) and V[p] = (x[2p][2q+1], x[2p+1][2q+1]) and
//           transforms over a = 2p + s: one scalar stage over s, three packed
//           stages over p.
//
// The result is the unnormalised transform z = x H; the rotation x R with
// R = H/16 is z * (1/16), an exact power-of-two scaling that is folded into
// the multiplier applied afterwards.  After all blocks of the row are
// transformed (they stay in registers), the CTA reduces the row absmax and
// writes the S8 codes; thread q of a slot owns the code pairs at columns
// (2q, 2q+1) of every block row.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>

namespace convrot {

constexpr int kBlock = 256;
constexpr int kSlotThreads = 8;                 // threads rotating one block
constexpr int kMaxThreads = 512;
constexpr int kMaxSlots = kMaxThreads / kSlotThreads;
constexpr int kRowUnits = 18;                   // 16 units of 8 bytes + 2 pad
constexpr int kSlotBytes = 8 * kRowUnits * 8;   // 1152 bytes per slot

// ------------------------------------------------------------------ packed FP32x2
__device__ __forceinline__ unsigned long long u64_of(float2 v) {
  return *reinterpret_cast<unsigned long long*>(&v);
}
__device__ __forceinline__ float2 f2_of(unsigned long long v) {
  return *reinterpret_cast<float2*>(&v);
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(u64_of(a)), "l"(u64_of(b)));
  return f2_of(d);
}
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
  unsigned long long d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(u64_of(a)), "l"(u64_of(b)));
  return f2_of(d);
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(u64_of(a)), "l"(u64_of(b)), "l"(u64_of(c)));
  return f2_of(d);
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(u64_of(a)), "l"(u64_of(b)));
  return f2_of(d);
}

// 16-point unnormalised Walsh-Hadamard transform over the array index,
// applied to both lanes of every pair at once.
__device__ __forceinline__ void fwht16x2(float2 (&P)[16]) {
#pragma unroll
  for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if ((i & h) == 0) {
        const float2 s = add2(P[i], P[i + h]);
        const float2 d = sub2(P[i], P[i + h]);
        P[i] = s;
        P[i + h] = d;
      }
    }
  }
}

// 8-point transform over the array index of pairs.
__device__ __forceinline__ void fwht8x2(float2 (&P)[8]) {
#pragma unroll
  for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if ((i & h) == 0) {
        const float2 s = add2(P[i], P[i + h]);
        const float2 d = sub2(P[i], P[i + h]);
        P[i] = s;
        P[i + h] = d;
      }
    }
  }
}

// Block state after pass 2: U[p] = (z[2p][2q], z[2p+1][2q]),
// V[p] = (z[2p][2q+1], z[2p+1][2q+1]).
struct BlockCols {
  float2 U[8], V[8];
};

// Pass 1 (on P, in place), transpose through `slot_smem`, pass 2 into `out`.
// Must be reached by every lane of the warp (`active` masks the work only).
__device__ __forceinline__ void rotate_block(float2 (&P)[16], BlockCols& out, char* slot_smem,
                                             int lane8, bool active) {
  if (active) {
    fwht16x2(P);
    // unit (p, b) at p * 18 + b; thread p writes its 16 units as 8 x 16 bytes
    float4* wrow = reinterpret_cast<float4*>(slot_smem + lane8 * kRowUnits * 8);
#pragma unroll
    for (int b = 0; b < 16; b += 2) wrow[b / 2] = make_float4(P[b].x, P[b].y, P[b + 1].x, P[b + 1].y);
  }
  __syncwarp();
  if (active) {
    const char* rbase = slot_smem + 2 * lane8 * 8;
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      const float4 w = *reinterpret_cast<const float4*>(rbase + p * kRowUnits * 8);
      // scalar stage over s (a = 2p + s)
      out.U[p] = make_float2(w.x + w.y, w.x - w.y);
      out.V[p] = make_float2(w.z + w.w, w.z - w.w);
    }
    fwht8x2(out.U);
    fwht8x2(out.V);
  }
  __syncwarp();
}

__device__ __forceinline__ float absmax_cols(float m, const BlockCols& c) {
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    m = fmaxf(m, fmaxf(fabsf(c.U[p].x), fabsf(c.U[p].y)));
    m = fmaxf(m, fmaxf(fabsf(c.V[p].x), fabsf(c.V[p].y)));
  }
  return m;
}

// Sum of squares of a block's 32 values held by this thread.
__device__ __forceinline__ float sumsq_cols(float ss, const BlockCols& c) {
  float2 a = make_float2(0.f, 0.f);
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    a = fma2(c.U[p], c.U[p], a);
    a = fma2(c.V[p], c.V[p], a);
  }
  return ss + (a.x + a.y);
}

__device__ __forceinline__ void scale_cols(BlockCols& c, float f) {
  const float2 ff = make_float2(f, f);
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    c.U[p] = mul2(c.U[p], ff);
    c.V[p] = mul2(c.V[p], ff);
  }
}

// Completes cluster_rowquant: the peer may read this CTA's slot until here.
__device__ __forceinline__ void cluster_exit_wait() {
  __syncwarp();
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// FP32 quantiser shared by both operands, for a row of rotated values v:
// s = fp32(amax / 127), r = fp32(1 / s), code = rint(fp32(v * r)) (half to
// even).  |v| <= amax bounds |v * r| by 127 * (1 + 3 * 2^-24), so the code
// never leaves [-127, 127].  Degenerate rows (s == 0 or r overflowing) get
// s = 0 and all-zero codes.
struct RowQuant {
  float s, r;
  __device__ __forceinline__ explicit RowQuant(float amax) {
    s = __fdiv_rn(amax, 127.0f);
    r = __frcp_rn(s);
    if ((s == 0.0f) || isinf(r)) {    // degenerate row
      s = 0.0f;
      r = 0.0f;
    }
  }
  __device__ __forceinline__ RowQuant(float s_, float r_) : s(s_), r(r_) {}
};

// Upper bound on the Euclidean norm of a row's codes, for the GEMM's choice
// of exact FP32 chunk length.  The codes are q = clamp(rint(fp32(v * r)));
// rounding moves each by at most 1/2 (plus the product's FP32 rounding,
// below 127 * 2^-24) and the clamp only shrinks them, so
// ||q|| <= r ||v|| + 0.5001 sqrt(K_p).  ||v|| = pre * sqrt(ss), ss being the
// FP32 sum of squares of the values the quantiser saw before its `pre`
// scaling; the factor 1 + 2^-10 covers that sum's rounding.  0 for a
// degenerate row (all codes zero).
__device__ __forceinline__ float code_norm_bound(const RowQuant& q, float ss, float pre, float half_sqrt_kp) {
  if (q.s == 0.0f) return 0.0f;
  return __fmaf_ru(sqrtf(ss) * (pre * q.r), 1.0f + 0.0009765625f, half_sqrt_kp);
}

// Sum over the warp (butterfly, every lane gets the total).
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Maximum over the warp of a non-negative float: non-negative floats order
// like their bit patterns, so the integer warp reduction (one instruction)
// applies.  It measured 2.5-6% faster than five shuffle-and-max steps in the
// weight and plain activation kernels and 0.6-0.7% faster in the SwiGLU one.
__device__ __forceinline__ float warp_max_nonneg(float v) {
  return __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(v)));
}

// Row absmax and quantiser of a row held by one CTA, set up once: warp 0
// reduces the per-warp maxima and computes s and r from amax * pre; every
// thread reads them after a second barrier.  Cheaper than every warp
// reducing the maxima and computing the division and the reciprocal itself.
// With with_ss, the row's sum of squares rides along and thread 0 leaves the
// code-norm bound in red[18] (uniform across the CTA: the caller asked for
// norms or not).  Warp 0 finishes the bound after the second barrier, where
// no other warp waits for it: QKV activations 84.6 -> 80.5 us, weights
// 89.2 -> 86.7 us, SwiGLU 344.8 -> 328.5 us (same box, alternating order).
// `red` layout (floats): [0, 16) per-warp maxima, [16] s, [17] r, [18] norm
// bound, [24, 40) per-warp sums of squares.
constexpr int kRedFloats = 48;
__device__ __forceinline__ RowQuant cta_rowquant(float local, float ss, bool with_ss, float* red, float pre,
                                                 float half_sqrt_kp) {
  local = warp_max_nonneg(local);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  if (with_ss) ss = warp_sum(ss);
  if (lane == 0) {
    red[warp] = local;
    if (with_ss) red[24 + warp] = ss;
  }
  __syncthreads();
  if (warp == 0) {
    const float m = warp_max_nonneg(lane < nwarps ? red[lane] : 0.f);
    const RowQuant q(m * pre);
    if (lane == 0) {
      red[16] = q.s;
      red[17] = q.r;
    }
  }
  __syncthreads();
  const RowQuant out(red[16], red[17]);
  if (with_ss && warp == 0) {
    const float t = warp_sum(lane < nwarps ? red[24 + lane] : 0.f);
    if (lane == 0) red[18] = code_norm_bound(out, t, pre, half_sqrt_kp);
  }
  return out;
}

// The same for a row split over the two CTAs of a cluster: warp 0 reduces
// this CTA's per-warp maxima and sums of squares and publishes them in
// xred[0], xred[1]; after a cluster barrier it reads the peer's, computes s
// and r and leaves them in xred[2], xred[3] for the CTA; thread 0 leaves the
// norm bound in xred[4] after the last barrier.  Every thread of both CTAs
// must call it and then call cluster_exit_wait() once before the CTA exits
// (the peer may read xred until then).  xred = red + 16; the per-warp sums
// use red[24, 40).
__device__ __forceinline__ RowQuant cluster_rowquant(float local, float ss, bool with_ss, float* red, float* xred,
                                                     float pre, float half_sqrt_kp) {
  local = warp_max_nonneg(local);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  if (with_ss) ss = warp_sum(ss);
  if (lane == 0) {
    red[warp] = local;
    if (with_ss) red[24 + warp] = ss;
  }
  __syncthreads();
  float m = 0.f, t = 0.f;
  if (warp == 0) {
    m = warp_max_nonneg(lane < nwarps ? red[lane] : 0.f);
    if (with_ss) t = warp_sum(lane < nwarps ? red[24 + lane] : 0.f);
    if (lane == 0) {
      xred[0] = m;
      xred[1] = t;
    }
  }
  __syncwarp();
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
  if (warp == 0) {
    uint32_t rank, remote;
    const uint32_t local_addr = static_cast<uint32_t>(__cvta_generic_to_shared(xred));
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank ^ 1u));
    float peer, peer_ss;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(peer) : "r"(remote) : "memory");
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(peer_ss) : "r"(remote + 4) : "memory");
    const RowQuant q(fmaxf(m, peer) * pre);
    t += peer_ss;
    if (lane == 0) {
      xred[2] = q.s;
      xred[3] = q.r;
    }
  }
  __syncwarp();
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");   // done reading the peer
  __syncthreads();
  const RowQuant out(xred[2], xred[3]);
  if (with_ss && threadIdx.x == 0) xred[4] = code_norm_bound(out, t, pre, half_sqrt_kp);
  return out;
}

// Round half to even of the FP32 product, two equivalent ways (bit-identical
// codes; the kernel picks the one whose pipe has room):
//  - cvt.rni.f32.f32: one instruction, on a conversion pipe that does 16
//    results per clock per SM (measured), an eighth of the FP32 add rate;
//  - adding 1.5 * 2^23 (|v| < 2^22): v lands where the FP32 spacing is 1, so
//    the nearest-even add itself rounds v to an integer, and subtracting the
//    constant back is exact; the bit pattern of the sum is 0x4B400000 + code,
//    so its low byte is the two's-complement S8 code.  __fadd_rn / __fsub_rn
//    are never contracted into a multiply-add with the product before them
//    (that would round the exact product instead of the FP32 one).
// The weight and plain activation kernels are bound by instruction issue and
// take cvt.rni (fewer instructions); the SwiGLU kernel's exponentials and
// reciprocals already load the conversion pipe, so it takes the adds.
constexpr float kRoundMagic = 12582912.0f;

template <bool MAGIC>
__device__ __forceinline__ float rint_f(float v) {
  if constexpr (MAGIC) {
    return __fsub_rn(__fadd_rn(v, kRoundMagic), kRoundMagic);
  } else {
    float d;
    asm("cvt.rni.f32.f32 %0, %1;" : "=f"(d) : "f"(v));
    return d;
  }
}

template <bool MAGIC>
__device__ __forceinline__ uint32_t code_byte(float v) {
  if constexpr (MAGIC) return __float_as_uint(__fadd_rn(v, kRoundMagic)) & 0xffu;
  else return static_cast<uint32_t>(__float2int_rn(v)) & 0xffu;
}

// FP16 codes of two values (already multiplied by r) without the conversion
// pipe.  kF16Magic = 1.5 * 2^23 + 0x6600 is an even integer in [2^23, 2^24),
// where the FP32 spacing is 1, so fp32(v + kF16Magic) = kF16Magic + rint(v)
// (half to even, as kF16Magic is even) for |v| < 2^21; its bit pattern is
// 0x4B406600 + code, whose low 16 bits 0x6600 + code (code in [-127, 127])
// are the FP16 encoding of 1536 + code.  One byte permute gathers the two
// low halves, and an exact FP16 subtraction of 1536 leaves the two codes.
constexpr float kF16Magic = 12609024.0f;

__device__ __forceinline__ __half2 f16_code_pair(float v0, float v1) {
  const uint32_t b0 = __float_as_uint(__fadd_rn(v0, kF16Magic));
  const uint32_t b1 = __float_as_uint(__fadd_rn(v1, kF16Magic));
  const uint32_t w = __byte_perm(b0, b1, 0x5410);
  return __hsub2(*reinterpret_cast<const __half2*>(&w), __float2half2_rn(1536.0f));
}

// Writes the codes of one block: values (already multiplied by r, so only
// the rounding is left) for rows 2p, 2p+1 and columns 2q, 2q+1.
template <bool MAGIC>
__device__ __forceinline__ void store_codes(void* q_row, bool f16_codes, int blk, int lane8,
                                            const BlockCols& c) {
  const int col = blk * kBlock + 2 * lane8;
  if (f16_codes) {
    __half2* q = reinterpret_cast<__half2*>(static_cast<__half*>(q_row) + col);
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      if constexpr (MAGIC) {
        q[(32 * p) / 2] = f16_code_pair(c.U[p].x, c.V[p].x);                                       // row 2p
        q[(32 * p + 16) / 2] = f16_code_pair(c.U[p].y, c.V[p].y);                                  // row 2p+1
      } else {
        q[(32 * p) / 2] = __floats2half2_rn(rint_f<false>(c.U[p].x), rint_f<false>(c.V[p].x));     // row 2p
        q[(32 * p + 16) / 2] = __floats2half2_rn(rint_f<false>(c.U[p].y), rint_f<false>(c.V[p].y));
      }
    }
  } else {
    uint16_t* q = reinterpret_cast<uint16_t*>(static_cast<int8_t*>(q_row) + col);
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      q[(32 * p) / 2] = static_cast<uint16_t>(code_byte<MAGIC>(c.U[p].x) | (code_byte<MAGIC>(c.V[p].x) << 8));
      q[(32 * p + 16) / 2] = static_cast<uint16_t>(code_byte<MAGIC>(c.U[p].y) | (code_byte<MAGIC>(c.V[p].y) << 8));
    }
  }
}

}  // namespace convrot
