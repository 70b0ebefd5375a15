// Kernel 3 of the ConvRot W4A8 layer: the row-scaled integer GEMM with its
// dequantising epilogue, and the C-ABI entry points convrot_gemm,
// convrot_gemm_i32 and convrot_device_error.
//
// What it computes (ComfyUI Turing Utils page on comfy.icu, node list, the
// entry on the ConvRot loaders reading native NVFP4 layers: an INT8
// tensor-core GEMM over row-scaled
// operands, FP16 / BF16 / FP32 outputs, logical N tails; MiniMax-H3
// explainer on modelpad.app: the rescale lives inside the matmul so the
// int32 intermediate never touches memory):
//     acc[m, n] = sum_k q_a[m, k] * q_w[n, k]            (exact int32)
//     y[m, n]   = fp32(acc) * s_a[m] * s_w[n]  -> out dtype
//
// GB300 design.  sm_103a has no 8-bit integer tcgen05 MMA, so the S8 codes
// arrive stored as FP16 integers and the product runs on tcgen05.mma
// kind::f16 with FP32 accumulation in tensor memory.  Products are at most
// 127^2 and a 1024-deep partial sum at most 127^2 * 1024 = 16,516,096 < 2^24,
// so every FP32 partial sum is an exact integer (tests drive running sums
// that are odd and above 2^23).  The K loop is therefore cut into equal
// chunks of at most 1024, each accumulated afresh in one of two TMEM buffers;
// epilogue warps convert each finished chunk to int32 (exact) and add it to
// per-thread int32 registers while the tensor core fills the other buffer.
// Given bounds on the rows' code norms, a work item whose bounds keep every
// partial sum below 2^24 (Cauchy-Schwarz) runs its whole K loop as one chunk,
// and the epilogue keeps the accumulator's FP32 bits (the exact integer).
//
// Mainloop: the MMA runs on CTA pairs (tcgen05.mma.cta_group::2, M = 256,
// N = 256, K = 16).  Each CTA of a pair holds its own 128 rows of A and one
// half (128 columns) of the pair's B tile, so every SM's tensor core reads
// 32 KiB of shared memory per 64-deep K step instead of the 48 KiB of a
// one-CTA 128 x 256 tile, and a stage costs 32 KiB: the ring is 6 stages
// deep.  The even CTA of a pair issues the MMAs; every load of the pair
// completes the even CTA's stage barrier.  A cluster is one pair (NPAIRS = 1):
// 76 clusters fill the 152 SMs.  With two pairs per cluster (NPAIRS = 2) the
// pairs share A by multicast, which saves a quarter of the L2 reads, but only
// 36 four-CTA clusters fit at once, 144 SMs, and it measured 3-8% slower.
// With two pairs, an odd number of 256-column N tiles leaves a last column
// that the pairs take separately ("solo" work items).  An odd number of
// 128-row M tiles leaves the last pair half empty (its rows past M load as
// zeros and are not stored).  Clusters are persistent over a grouped tile
// order.
// Warp 0: TMA producer.  Warp 1: TMEM owner and (even CTA) MMA issuer.
// Warps 2..9: epilogue, which applies y = fp32(acc) * s_a * s_w (+ bias),
// stages 32-row x 64-byte boxes in swizzled shared memory and writes them
// with TMA tensor stores (per-element stores for unaligned outputs).
// Warp 10 (even CTA, with norm bounds): evaluates the chunk count of the
// coming work items ahead of the MMA issuer.  Every
// mbarrier wait is bounded: after about two seconds the waiting role records
// an error code, the CTA drains what it has in flight and returns.
#include <cstdint>
#include <cstring>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "../../include/convrot.h"
#include "errors.h"

namespace crgemm {

constexpr int BM = 128, BN = 256, BK = 64;       // per-CTA output tile 128 x 256; pair tile 256 x 256
constexpr int STAGES = 6;
constexpr int KCHUNK_STEPS = 16;                 // 16 * 64 = 1024 K per exact FP32 chunk
constexpr int A_BYTES = BM * BK * 2;             // 16 KiB: this CTA's 128 rows of A
constexpr int A_HALF_BYTES = A_BYTES / 2;        // 64 rows, the part one CTA loads and multicasts
constexpr int B_BYTES = (BN / 2) * BK * 2;       // 16 KiB: this CTA's half (128 columns) of the pair's B
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;   // 32 KiB per CTA
constexpr int PAIR_STAGE_BYTES = 2 * STAGE_BYTES;// bytes landing in both CTAs of a pair per stage
constexpr int NUM_EPI_WARPS = 8;
constexpr int NORM_WARP = 2 + NUM_EPI_WARPS;     // warp 10: chunking of the coming work items
constexpr int THREADS = 64 + NUM_EPI_WARPS * 32 + 32;   // 352
// Eleven warps put at most three on one SM sub-partition (16K registers):
// the launch bound is declared for 384 threads so that the compiler keeps a
// thread at 168 registers (3 x 32 x 168 <= 16384).
constexpr int THREADS_BOUND = 384;
constexpr int NRING = 4;                         // chunk counts evaluated ahead of the MMA issuer
constexpr int TMEM_COLS = 512;                   // two 256-column FP32 buffers
constexpr int NPAIRS = 1;                        // CTA pairs per cluster (2: they share A by multicast)
constexpr int CLUSTER = 2 * NPAIRS;              // rank = 2 * pair + half
constexpr int A_BOX_ROWS = NPAIRS == 2 ? BM / 2 : BM;   // rows of A per TMA load (halves when multicast)
constexpr int GROUP_M2 = 16;                     // tile raster: 16 pair rows (4096 rows) share each B tile
// Output staging: each epilogue warp writes its 32 rows x 128 columns as
// boxes of 32 rows x 64 bytes (64-byte swizzle), OUT_BUFS buffers per warp,
// and hands every box to a TMA tensor store.
constexpr int OUT_BOX_BYTES = 64;
constexpr int OUT_BOX = 32 * OUT_BOX_BYTES;                  // 2 KiB
constexpr int OUT_BUFS = 2;
constexpr int OUT_STAGING = NUM_EPI_WARPS * OUT_BUFS * OUT_BOX;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + OUT_STAGING + 1024 /*align*/ + 256 /*barriers*/;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;
static_assert((2 * STAGES + 7 + 2 * NRING) * 8 + NRING * 4 <= 256, "barrier area");

// Codes recorded in g_error: which wait ran out first.
enum ErrCode : int { ERR_NONE = 0, ERR_WAIT_FULL = 1, ERR_WAIT_EMPTY = 2, ERR_WAIT_ACC_FULL = 3,
                     ERR_WAIT_ACC_EMPTY = 4, ERR_WAIT_CHUNKS = 5 };

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

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// try_wait with a suspend-time hint: a waiting thread sleeps until the phase
// completes (or kSuspendNs pass) instead of polling.  Polling waits (the
// epilogue warps for a finished accumulator, the producer for a free stage,
// the issuer for a full one) cost the QKV GEMM 5% (2.282 -> 2.166 ms, same
// box, alternating order); a 1 us hint measured the same as 20 us.
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

// TMA load of one box into this CTA's shared memory at `dst`; its bytes
// complete the mbarrier at shared::cluster address `bar`, which may lie in
// the pair's even CTA (.cta_group::2).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%3, %4}], [%2];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

// The same box delivered to the same shared-memory offset in every CTA of
// `mask`; in each destination the bytes complete the mbarrier at the offset
// of `bar` in that destination's even (MMA-issuing) CTA, `bar` being an
// address in an even CTA.
__device__ __forceinline__ void tma_load_2d_mc(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y,
                                               uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster"
      ".cta_group::2 [%0], [%1, {%3, %4}], [%2], %5;"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "h"(mask)
      : "memory");
}

// Shared::cluster address of this CTA's shared-memory word `local` in CTA `rank`.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}

// Arrive on a barrier of this CTA (release at CTA scope: writes before it are
// seen by a thread whose wait completes the phase).
__device__ __forceinline__ void mbar_arrive_local(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Arrive on an mbarrier given by its shared::cluster address (this CTA's or
// another's), with the default CTA-scope release: the epilogue uses it to
// hand a drained TMEM buffer back to the pair's MMA issuer, and the tensor
// memory reads it orders are fenced by tcgen05.fence::before_thread_sync (a
// cluster-scope release here made every arrive a cluster-wide memory fence).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}

// TMA tensor store of one box from shared memory; completion is tracked
// per thread with bulk groups.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];"
               ::"l"(reinterpret_cast<uint64_t>(map)), "r"(src), "r"(x), "r"(y) : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most N of this thread's bulk store groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Every thread of both CTAs; the barrier instructions are warp-aligned.
__device__ __forceinline__ void cluster_sync() {
  __syncwarp();
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrive on the mbarrier at this offset in every CTA of `mask` once all
// previously issued tcgen05 operations of this thread (pair MMAs) have
// completed.
__device__ __forceinline__ void tc_commit_mc(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
      ::"r"(bar), "h"(mask) : "memory");
}

// Pair MMA: D[tmem] (+)= A * B^T over both CTAs of the pair (M = 256: each
// CTA's 128 rows of A; N = 256: each CTA's 128 columns of B, at the same
// shared-memory offsets in both), FP16 inputs, FP32 accumulate; D lands in
// each CTA's tensor memory for its own 128 rows.
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns (thread i: row lane base + i).
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
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
// N = 256, M = 256 (the pair).
constexpr uint32_t kIdesc = (1u << 4)                         // D format: F32
                            | (0u << 7) | (0u << 10)          // A, B: F16
                            | (0u << 15) | (0u << 16)         // K-major A and B
                            | (static_cast<uint32_t>(BN >> 3) << 17)
                            | (static_cast<uint32_t>((2 * BM) >> 4) << 24);

struct Params {
  int M, N, K_p;
  int num_m, num_n, k_steps;
  int num_m2;          // pair rows: 256-row strips (the last one half empty when num_m is odd)
  int num_shared;      // work items whose two pairs share A: num_m2 * (num_n / 2)
  int num_items;       // num_shared, then ceil(num_m2 / 2) solo items for the last N tile when num_n is odd
  const float* a_scale;
  const float* w_scale;
  const float* bias;   // optional, [N]
  const float* a_norm; // optional, [M]: bounds on the Euclidean norms of A's rows of codes
  const float* w_norm; // optional, [N]: the same for B's rows
  void* out;
  int64_t ld_out;
  int out_vec;      // 16-byte vector stores allowed (base and pitch aligned)
  int out_tma;      // output written by TMA tensor stores (base and pitch 16-byte aligned)
  int test_stall;   // failure-detection self-test: the producer issues no loads
};

// Work item -> this CTA's pair row (256-row strip) and N tile.  Shared items
// run in a grouped order (GROUP_M2 pair rows in a row reuse each B tile from
// L2); pair `pair` takes N tile 2 * nb + pair, and both pairs own the same
// rows, so A is multicast between them.  Solo items cover the last N tile
// when num_n is odd: the two pairs take pair rows 2 j and 2 j + 1 of it (the
// second may lie past the last row strip: it then computes zeros and stores
// nothing).  Returns true for a shared item.
__device__ __forceinline__ bool work_coords(const Params& p, int item, int pair, int& m2, int& nt) {
  if (NPAIRS == 1) {              // one pair per cluster: items are (pair row, N tile)
    const int per_group = GROUP_M2 * p.num_n;
    const int g = item / per_group;
    const int first = g * GROUP_M2;
    const int gsize = min(GROUP_M2, p.num_m2 - first);
    const int r = item - g * per_group;
    m2 = first + r % gsize;
    nt = r / gsize;
    return false;
  }
  if (item < p.num_shared) {
    const int n2 = p.num_n >> 1;
    const int per_group = GROUP_M2 * n2;
    const int g = item / per_group;
    const int first = g * GROUP_M2;
    const int gsize = min(GROUP_M2, p.num_m2 - first);
    const int r = item - g * per_group;
    m2 = first + r % gsize;
    nt = 2 * (r / gsize) + pair;
    return true;
  }
  m2 = 2 * (item - p.num_shared) + pair;
  nt = p.num_n - 1;
  return false;
}

// ------------------------------------------------------------------ chunking of a work item
// Every partial sum of a dot product q_a[m, :] . q_w[n, :], in any order, is
// at most ||q_a[m, :]|| ||q_w[n, :]|| (Cauchy-Schwarz).  When the largest
// bound among the work item's 256 A rows times the largest among its 256 B
// rows is below 2^24, every FP32 partial sum of the tile is an exact integer,
// so the whole K loop runs as one chunk; otherwise it is cut into exact
// chunks of at most KCHUNK_STEPS.  A warp evaluates it (lane l reads rows
// l, l + 32, ...): the chunking warp for the MMA issuer, each epilogue warp
// for itself; all reach the same answer for an item.
__device__ __forceinline__ int tile_chunks(const Params& p, int m2, int nt, int lane, int default_chunks) {
  // maxima over the bit patterns: non-negative floats (and NaN, which then
  // fails the test) order like their bits; four rows of each operand in flight
  uint32_t ma = 0u, mw = 0u;
#pragma unroll 2
  for (int j = 0; j < 8; j += 4) {
    float a[4], w[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int ra = m2 * (2 * BM) + lane + 32 * (j + u), rw = nt * BN + lane + 32 * (j + u);
      a[u] = ra < p.M ? __ldg(p.a_norm + ra) : 0.f;
      w[u] = rw < p.N ? __ldg(p.w_norm + rw) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      ma = max(ma, __float_as_uint(a[u]) & 0x7fffffffu);
      mw = max(mw, __float_as_uint(w[u]) & 0x7fffffffu);
    }
  }
  ma = __reduce_max_sync(0xffffffffu, ma);
  mw = __reduce_max_sync(0xffffffffu, mw);
  const float prod = __fmul_ru(__uint_as_float(ma), __uint_as_float(mw));   // rounded up
  return prod < 16777216.0f ? 1 : default_chunks;
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

// Two outputs rounded (nearest even, each on its own) into one 32-bit word,
// the first in the low half: one packed conversion instead of two.
template <int OUT>
__device__ __forceinline__ uint32_t to_out2(float y0, float y1);
template <> __device__ __forceinline__ uint32_t to_out2<CONVROT_BF16>(float y0, float y1) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(y0, y1);
  return *reinterpret_cast<const uint32_t*>(&h);
}
template <> __device__ __forceinline__ uint32_t to_out2<CONVROT_FP16>(float y0, float y1) {
  const __half2 h = __floats2half2_rn(y0, y1);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// OUT = CONVROT_BF16 / FP16 / FP32, or -1 for raw int32 accumulators.
// BIAS: p.bias is non-null and added in the epilogue.
// TMA_OUT: staged output boxes go out by TMA tensor stores (output base and
// pitch 16-byte aligned); otherwise the warp writes them with element stores.
template <int OUT, bool BIAS, bool TMA_OUT>
__global__ void __launch_bounds__(THREADS_BOUND, 1)
gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
            const __grid_constant__ CUtensorMap tmap_out, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* staging = smem + STAGES * STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(staging + OUT_STAGING);
  // barrier slots: full[STAGES], empty[STAGES], acc_full[2], acc_empty[2], drain, then the
  // TMEM address, the abort flag, the chunk-count ring's full[NRING] and empty[NRING] and
  // the ring itself
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + STAGES);
  const uint32_t accf0 = smem_u32(bars + 2 * STAGES), acce0 = smem_u32(bars + 2 * STAGES + 2);
  const uint32_t drain = smem_u32(bars + 2 * STAGES + 4);
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(bars + 2 * STAGES + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * STAGES + 6);
  const uint32_t nfull0 = smem_u32(bars + 2 * STAGES + 7), nempty0 = smem_u32(bars + 2 * STAGES + 7 + NRING);
  volatile int* ring = reinterpret_cast<volatile int*>(bars + 2 * STAGES + 7 + 2 * NRING);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const uint32_t half = rank & 1u, pair = rank >> 1;     // half: which 128 rows of the pair's 256
  const uint32_t leader = rank & ~1u;                     // the pair's even CTA: issues the MMAs
  const bool is_leader = half == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);               // the even CTA's producer + PAIR_STAGE_BYTES of loads
      mbar_init(empty0 + 8 * s, NPAIRS);         // released by the MMAs of every pair
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf0 + 8 * b, 1);
      mbar_init(acce0 + 8 * b, 2 * NUM_EPI_WARPS);   // epilogue warps of both CTAs of the pair
    }
    mbar_init(drain, 1);
    for (int r = 0; r < NRING; ++r) {
      mbar_init(nfull0 + 8 * r, 1);              // the chunking warp wrote ring[r]
      mbar_init(nempty0 + 8 * r, 1);             // the MMA issuer has read it
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_a)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_b)) : "memory");
  }
  if (warp == 1) {
    // one warp of each CTA of the pair allocates the same columns in both
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_u32(const_cast<uint32_t*>(tmem_slot))), "r"(TMEM_COLS) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  // other CTAs' loads, multicasts and commits target our barriers: every CTA
  // of the cluster must have initialised its barriers before any is issued
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int cluster_id = blockIdx.x / CLUSTER, num_clusters = gridDim.x / CLUSTER;
  constexpr uint16_t kAll = (1u << CLUSTER) - 1u;
  const uint16_t pair_mask = static_cast<uint16_t>(3u << (2 * pair));
  const uint16_t a_mask = static_cast<uint16_t>(NPAIRS == 2 ? (1u << half) | (1u << (half + 2)) : 0u);

  const int k_steps = p.k_steps;
  // Without norm bounds (or when they do not allow a single chunk) the K
  // steps are split into equal chunks of at most KCHUNK_STEPS: a short last
  // chunk would leave the epilogue less time to drain the buffer it follows
  // (K = 5376: six chunks of 896 instead of five of 1024 and one of 256).
  const int chunks_per_tile = (k_steps + KCHUNK_STEPS - 1) / KCHUNK_STEPS;
  const bool eval_chunks = p.a_norm != nullptr && p.w_norm != nullptr && chunks_per_tile > 1;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      uint32_t issued_mask = 0, issued_phase = 0;   // even CTA: last outstanding stage phase
      const uint32_t lfull0 = map_to_rank(full0, leader);
      for (int tile = cluster_id; tile < p.num_items && ok && !p.test_stall; tile += num_clusters) {
        int m2, nt;
        const bool shared_a = work_coords(p, tile, static_cast<int>(pair), m2, nt);
        const int m_row = (2 * m2 + static_cast<int>(half)) * BM;
        for (int ks = 0; ks < k_steps; ++ks) {
          // the stage is free once the MMAs of BOTH pairs have consumed it
          if (!mbar_wait(empty0 + 8 * stage, phase ^ 1u, ERR_WAIT_EMPTY, abort_flag)) { ok = false; break; }
          const uint32_t fb = lfull0 + 8 * stage;
          if (is_leader) mbar_arrive_expect_tx(full0 + 8 * stage, PAIR_STAGE_BYTES);
          const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
          if (shared_a) {
            // our half of the 128 rows, into this CTA and the same-rows CTA of the other pair
            tma_load_2d_mc(sa + pair * A_HALF_BYTES, &tmap_a, fb, ks * BK, m_row + static_cast<int>(pair) * (BM / 2),
                           a_mask);
          } else {
#pragma unroll
            for (int h = 0; h < BM / A_BOX_ROWS; ++h)
              tma_load_2d(sa + h * (A_BOX_ROWS * BK * 2), &tmap_a, fb, ks * BK, m_row + h * A_BOX_ROWS);
          }
          tma_load_2d(sa + A_BYTES, &tmap_b, fb, ks * BK, nt * BN + static_cast<int>(half) * (BN / 2));
          issued_mask |= 1u << stage;
          issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      if (ok) {
        // the other CTAs' MMA commits arrive on our empty barriers: wait until
        // both pairs have released the last use of every stage before leaving
        for (int i = 0; i < STAGES; ++i) {
          if (!mbar_wait(empty0 + 8 * stage, phase ^ 1u, ERR_WAIT_EMPTY, abort_flag)) break;
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      } else if (is_leader) {
        // let every load still in flight into the pair land before the CTAs
        // can exit (the even CTA's barriers count the whole pair's bytes)
        for (int s = 0; s < STAGES; ++s)
          if (issued_mask & (1u << s)) {
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(full0 + 8 * s, (issued_phase >> s) & 1u) &&
                   globaltimer() - t0 < kWaitLimitNs) {}
          }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer (even CTA)
    // Lane 0 issues.  With norm bounds, each work item's chunk count comes
    // from the chunking warp through the ring; evaluating it here put about
    // 0.8 us between two items' MMAs (3% at K = 5376).
    if (is_leader && lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t chunk = 0;          // running chunk counter -> TMEM buffer and its phase
      bool ok = true;
      bool any = false;
      int item = 0;                // this cluster's work items so far -> ring slot and its phase
      for (int tile = cluster_id; tile < p.num_items && ok; tile += num_clusters, ++item) {
        int nchunks = chunks_per_tile;
        if (eval_chunks) {
          const int r = item % NRING;
          const uint32_t use = static_cast<uint32_t>(item / NRING);
          if (!mbar_wait(nfull0 + 8 * r, use & 1u, ERR_WAIT_CHUNKS, abort_flag)) { ok = false; break; }
          nchunks = ring[r];
          mbar_arrive_local(nempty0 + 8 * r);
        }
        const int csteps = (k_steps + nchunks - 1) / nchunks;
        for (int c = 0; c < nchunks && ok; ++c, ++chunk) {
          const uint32_t buf = chunk & 1u, use = chunk >> 1;
          if (!mbar_wait(acce0 + 8 * buf, (use & 1u) ^ 1u, ERR_WAIT_ACC_EMPTY, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + buf * BN;
          const int ks0 = c * csteps, ks1 = min(k_steps, ks0 + csteps);
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
            tc_commit_mc(empty0 + 8 * stage, kAll);
            if (++stage == STAGES) { stage = 0; phase ^= 1u; }
          }
          if (ok) tc_commit_mc(accf0 + 8 * buf, pair_mask);
        }
      }
      if (!ok && any) {
        // wait for the tensor cores to finish everything issued before TMEM is freed
        tc_commit_mc(drain, static_cast<uint16_t>(1u << rank));
        const uint64_t t0 = globaltimer();
        while (!mbar_try_wait(drain, 0) && globaltimer() - t0 < kWaitLimitNs) {}
      }
    }
  } else if (warp == NORM_WARP) {
    // ---------------------------------------------------------------- chunking (even CTA)
    // Evaluates the chunk count of this cluster's work items up to NRING
    // ahead of the MMA issuer and hands them over through ring[].
    if (is_leader && eval_chunks) {
      int item = 0;
      for (int tile = cluster_id; tile < p.num_items; tile += num_clusters, ++item) {
        const int r = item % NRING;
        const uint32_t use = static_cast<uint32_t>(item / NRING);
        int got = 1;
        if (lane == 0) got = mbar_wait(nempty0 + 8 * r, (use & 1u) ^ 1u, ERR_WAIT_CHUNKS, abort_flag) ? 1 : 0;
        if (!__shfl_sync(0xffffffffu, got, 0)) break;
        int m2, nt;
        work_coords(p, tile, static_cast<int>(pair), m2, nt);
        const int n = tile_chunks(p, m2, nt, lane, chunks_per_tile);
        if (lane == 0) {
          ring[r] = n;
          mbar_arrive_local(nfull0 + 8 * r);
        }
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int ew = warp - 2;                  // 0..7
    const int quarter = warp & 3;             // TMEM lanes this warp may access
    const int col_half = ew >> 2;             // columns [0,128) or [128,256) of the tile
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    uint32_t chunk = 0;
    uint32_t boxes = 0;                       // output boxes staged by this warp so far
    bool ok = true;
    const uint32_t lacce0 = map_to_rank(acce0, leader);   // the even CTA's acc_empty barriers
    for (int tile = cluster_id; tile < p.num_items && ok; tile += num_clusters) {
      int m2, nt;
      work_coords(p, tile, static_cast<int>(pair), m2, nt);
      const int mb = 2 * m2 + static_cast<int>(half), nb = nt;
      int nchunks = chunks_per_tile;
      if (eval_chunks) {
        // the chunking warp's evaluation, repeated: its loads wait in the
        // shadow of this item's first accumulator (measured free)
        nchunks = tile_chunks(p, m2, nt, lane, chunks_per_tile);
      }
      // One chunk (dequantised outputs): the FP32 accumulator already is the
      // exact integer sum (below 2^24), so acc keeps its bits, with no
      // conversion.  Several chunks (or int32 output): each chunk is converted
      // to int32 (exact) and added; for dequantised outputs the total is
      // turned into FP32 bits once at the end.  The FP32 value either way is
      // fp32(sum), rounded to nearest.
      const bool keep_bits = OUT >= 0 && nchunks == 1;
      int32_t acc[128];
#pragma unroll
      for (int j = 0; j < 128; ++j) acc[j] = 0;
      for (int c = 0; c < nchunks; ++c, ++chunk) {
        const uint32_t buf = chunk & 1u, use = chunk >> 1;
        // one lane polls, the warp follows: tcgen05.ld below needs a converged warp
        int got = 1;
        if (lane == 0) got = mbar_wait(accf0 + 8 * buf, use & 1u, ERR_WAIT_ACC_FULL, abort_flag) ? 1 : 0;
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) { ok = false; break; }
        tc_fence_after();
        const uint32_t t_base = tmem_base + lane_addr + buf * BN + col_half * 128;
        // 16 columns per load: with 32, the 128 accumulators and the load's
        // registers exceed the 168-register budget and spill
        if (keep_bits) {
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            uint32_t r[16];
            tmem_ld_32x32b_x16(t_base + g * 16, r);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j) acc[g * 16 + j] = static_cast<int32_t>(r[j]);
          }
        } else {
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            uint32_t r[16];
            tmem_ld_32x32b_x16(t_base + g * 16, r);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              // the FP32 value is an exact integer below 2^24: conversion is exact
              acc[g * 16 + j] += __float2int_rn(__uint_as_float(r[j]));
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(lacce0 + 8 * buf);
      }
      if (!ok) break;
      if (OUT >= 0 && !keep_bits) {
#pragma unroll
        for (int j = 0; j < 128; ++j) acc[j] = __float_as_int(static_cast<float>(acc[j]));
      }
      // ---- output: this thread owns row m, columns n0 .. n0+127
      const int m_base = mb * BM + quarter * 32;
      const int m = m_base + lane;
      const int n0 = nb * BN + col_half * 128;
      if constexpr (OUT < 0) {
        if (m < p.M) {
          int32_t* orow = static_cast<int32_t*>(p.out) + static_cast<int64_t>(m) * p.ld_out;
#pragma unroll
          for (int j = 0; j < 128; ++j)
            if (n0 + j < p.N) orow[n0 + j] = acc[j];
        }
      } else {
        using T = typename OutT<OUT>::T;
        constexpr int VEC = 16 / sizeof(T);           // outputs per 16-byte chunk
        const float sa = (m < p.M) ? __ldg(p.a_scale + m) : 0.f;
        {
          // staged 32-row boxes, written by a TMA tensor store, or (output
          // base or pitch not 16-byte aligned) by the warp with element
          // stores that walk each row: consecutive lanes, consecutive columns
          constexpr int CPB = OUT_BOX_BYTES / sizeof(T);   // columns per box
          uint8_t* wstage = staging + ew * OUT_BUFS * OUT_BOX;
#pragma unroll
          for (int b = 0; b < 128 / CPB; ++b) {
            const int buf = static_cast<int>(boxes % OUT_BUFS);
            if (boxes >= OUT_BUFS) {
              // the store issued from this buffer OUT_BUFS boxes ago must have read it
              if (lane == 0) bulk_wait_read<OUT_BUFS - 1>();
              __syncwarp();
            }
            ++boxes;
            uint8_t* rowp = wstage + buf * OUT_BOX + lane * OUT_BOX_BYTES;
#pragma unroll
            for (int c = 0; c < OUT_BOX_BYTES / 16; ++c) {
              const int j0 = b * CPB + c * VEC;            // first column of this chunk
              const int n = n0 + j0;
              float sw[VEC], bs[VEC];
              if (n + VEC <= p.N) {
#pragma unroll
                for (int q = 0; q < VEC; q += 4) {
                  const float4 f = __ldg(reinterpret_cast<const float4*>(p.w_scale + n + q));
                  sw[q] = f.x; sw[q + 1] = f.y; sw[q + 2] = f.z; sw[q + 3] = f.w;
                  if constexpr (BIAS) {
                    const float4 g = __ldg(reinterpret_cast<const float4*>(p.bias + n + q));
                    bs[q] = g.x; bs[q + 1] = g.y; bs[q + 2] = g.z; bs[q + 3] = g.w;
                  } else {
                    bs[q] = bs[q + 1] = bs[q + 2] = bs[q + 3] = 0.f;
                  }
                }
              } else {
#pragma unroll
                for (int q = 0; q < VEC; ++q) {
                  sw[q] = (n + q < p.N) ? __ldg(p.w_scale + n + q) : 0.f;
                  bs[q] = (BIAS && n + q < p.N) ? __ldg(p.bias + n + q) : 0.f;
                }
              }
              union { T v[VEC]; uint32_t w[4]; uint4 u; } pk;
              float yv[VEC];
#pragma unroll
              for (int q = 0; q < VEC; ++q) {
                const float y = __fmul_rn(__fmul_rn(__int_as_float(acc[j0 + q]), sa), sw[q]);
                yv[q] = BIAS ? __fadd_rn(y, bs[q]) : y;
              }
              if constexpr (sizeof(T) == 2) {
#pragma unroll
                for (int q = 0; q < VEC; q += 2) pk.w[q / 2] = to_out2<OUT>(yv[q], yv[q + 1]);
              } else {
#pragma unroll
                for (int q = 0; q < VEC; ++q) pk.v[q] = to_out<OUT>(yv[q]);
              }
              // 64-byte swizzle: 16-byte chunk c of row r sits at chunk c ^ ((r >> 1) & 3)
              *reinterpret_cast<uint4*>(rowp + ((c ^ ((lane >> 1) & 3)) << 4)) = pk.u;
            }
            if constexpr (TMA_OUT) {
              fence_proxy_async_smem();
              __syncwarp();
              // boxes wholly outside the matrix (M or N tail) are not stored
              if (lane == 0 && m_base < p.M && n0 + b * CPB < p.N) {
                tma_store_2d(&tmap_out, smem_u32(wstage + buf * OUT_BOX), n0 + b * CPB, m_base);
                bulk_commit();
              }
            } else {
              __syncwarp();
              const uint8_t* box = wstage + buf * OUT_BOX;
#pragma unroll 4
              for (int it = 0; it < CPB; ++it) {
                const int idx = it * 32 + lane;              // element of the 32 x CPB box, row-major
                const int r = idx / CPB, col = idx % CPB;
                const int bo = col * static_cast<int>(sizeof(T));
                const int mr = m_base + r, n = n0 + b * CPB + col;
                if (mr < p.M && n < p.N) {
                  const T v = *reinterpret_cast<const T*>(box + r * OUT_BOX_BYTES +
                                                          ((((bo >> 4) ^ ((r >> 1) & 3))) << 4) + (bo & 15));
                  static_cast<T*>(p.out)[static_cast<int64_t>(mr) * p.ld_out + n] = v;
                }
              }
              __syncwarp();                                  // box read before its buffer is refilled
            }
          }
        }
      }
    }
    // every TMA store of this warp must be complete before the CTA exits
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();            // no CTA leaves while another may still write into it
  tc_fence_after();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
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

// Store map over the output [M][N] (pitch ld_out elements): boxes of 32 rows x
// 64 bytes with 64-byte swizzle; TMA clips the parts outside the matrix.
static bool make_out_map(CUtensorMap* map, void* base, int out_kind, int M, int N, int64_t ld) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const size_t es = out_kind == CONVROT_FP32 ? 4 : 2;
  const CUtensorMapDataType dt = out_kind == CONVROT_FP32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : out_kind == CONVROT_FP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                            : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * es};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(OUT_BOX_BYTES / es), 32};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, dt, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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

// Persistent grid: as many clusters as can be resident at once (one CTA per
// SM), never more than there are work items.
template <int OUT, bool BIAS, bool TMA_OUT>
static cudaError_t launch(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mo,
                          const Params& p, cudaStream_t st) {
  static int max_clusters_by_dev[64] = {0};   // resident clusters, per device and instantiation
  int dev = 0;
  {
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
  }
  int dummy = 0;
  int& max_clusters = (dev >= 0 && dev < 64) ? max_clusters_by_dev[dev] : dummy;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CLUSTER;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (max_clusters == 0) {
    cudaError_t e = cudaFuncSetAttribute(gemm_kernel<OUT, BIAS, TMA_OUT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SMEM_BYTES);
    if (e != cudaSuccess) return e;
    int sms = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    cfg.gridDim = dim3(sms / CLUSTER * CLUSTER);
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, gemm_kernel<OUT, BIAS, TMA_OUT>, &cfg);
    if (e != cudaSuccess || n <= 0) {
      (void)cudaGetLastError();
      n = sms / CLUSTER;
    }
    max_clusters = n;
  }
  const int clusters = p.num_items < max_clusters ? p.num_items : max_clusters;
  cfg.gridDim = dim3(clusters * CLUSTER);
  return cudaLaunchKernelEx(&cfg, gemm_kernel<OUT, BIAS, TMA_OUT>, ma, mb, mo, p);
}

template <int OUT>
static cudaError_t launch_out(bool bias, bool tma, const CUtensorMap& ma, const CUtensorMap& mb,
                              const CUtensorMap& mo, const Params& p, cudaStream_t st) {
  if (bias) return tma ? launch<OUT, true, true>(ma, mb, mo, p, st) : launch<OUT, true, false>(ma, mb, mo, p, st);
  return tma ? launch<OUT, false, true>(ma, mb, mo, p, st) : launch<OUT, false, false>(ma, mb, mo, p, st);
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

static int run(int out_kind, const void* a_q, int64_t ld_aq, const float* a_scale, const float* a_norm,
               const void* w_q, int64_t ld_wq, const float* w_scale, const float* w_norm, const float* bias,
               int M, int N, int K_p, void* out, int64_t ld_out, size_t out_esize, cudaStream_t stream,
               int test_stall = 0) {
  Params p;
  p.test_stall = test_stall;
  p.bias = bias;
  p.a_norm = a_norm;
  p.w_norm = w_norm;
  p.M = M;
  p.N = N;
  p.K_p = K_p;
  p.num_m = (M + BM - 1) / BM;
  p.num_n = (N + BN - 1) / BN;
  p.num_m2 = (p.num_m + 1) / 2;
  if (NPAIRS == 2) {
    p.num_shared = p.num_m2 * (p.num_n / 2);
    p.num_items = p.num_shared + (p.num_n % 2 ? (p.num_m2 + 1) / 2 : 0);
  } else {
    p.num_shared = 0;
    p.num_items = p.num_m2 * p.num_n;
  }
  p.k_steps = K_p / BK;
  p.a_scale = a_scale;
  p.w_scale = w_scale;
  p.out = out;
  p.ld_out = ld_out;
  p.out_vec = (reinterpret_cast<uintptr_t>(out) % 16 == 0) && ((ld_out * static_cast<int64_t>(out_esize)) % 16 == 0);
  CUtensorMap ma, mb;
  if (!make_map(&ma, a_q, M, K_p, ld_aq, A_BOX_ROWS) || !make_map(&mb, w_q, N, K_p, ld_wq, BN / 2))
    return convrot::record_error("cuTensorMapEncodeTiled failed for an operand map");
  CUtensorMap mo;
  memset(&mo, 0, sizeof(mo));
  p.out_tma = 0;
  if (out_kind >= 0 && p.out_vec) p.out_tma = make_out_map(&mo, out, out_kind, M, N, ld_out) ? 1 : 0;
  cudaError_t e;
  const bool b = bias != nullptr;
  switch (out_kind) {
    case CONVROT_BF16: e = launch_out<CONVROT_BF16>(b, p.out_tma != 0, ma, mb, mo, p, stream); break;
    case CONVROT_FP16: e = launch_out<CONVROT_FP16>(b, p.out_tma != 0, ma, mb, mo, p, stream); break;
    case CONVROT_FP32: e = launch_out<CONVROT_FP32>(b, p.out_tma != 0, ma, mb, mo, p, stream); break;
    default: e = launch<-1, false, false>(ma, mb, mo, p, stream); break;
  }
  return e == cudaSuccess ? CONVROT_OK : convrot::record_cuda_error("GEMM launch", e);
}

}  // namespace crgemm

using namespace crgemm;

// Norm bounds: both or neither are used; 4-byte aligned.
static int check_norms(const float* a_norm, const float* w_norm) {
  if (reinterpret_cast<uintptr_t>(a_norm) % 4 || reinterpret_cast<uintptr_t>(w_norm) % 4)
    return CONVROT_ERR_MISALIGNED;
  return CONVROT_OK;
}

extern "C" int convrot_gemm(const void* a_q, int64_t ld_aq, const float* a_scale, const float* a_norm,
                            const void* w_q, int64_t ld_wq, const float* w_scale, const float* w_norm,
                            const float* bias, int M, int N, int K_p, void* out, convrot_dtype out_dtype,
                            int64_t ld_out, cudaStream_t stream) {
  if (out_dtype != CONVROT_BF16 && out_dtype != CONVROT_FP16 && out_dtype != CONVROT_FP32)
    return CONVROT_ERR_UNSUPPORTED;
  int st = validate_operands(a_q, ld_aq, w_q, ld_wq, M, N, K_p);
  if (st != CONVROT_OK) return st;
  if (ld_out < N) return CONVROT_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return CONVROT_OK;
  if (!a_scale || !w_scale || !out) return CONVROT_ERR_INVALID_ARG;
  const size_t es = out_dtype == CONVROT_FP32 ? 4 : 2;
  // w_scale and bias are read four at a time: 16-byte aligned
  if (reinterpret_cast<uintptr_t>(out) % es || reinterpret_cast<uintptr_t>(a_scale) % 4 ||
      reinterpret_cast<uintptr_t>(w_scale) % 16 || reinterpret_cast<uintptr_t>(bias) % 16)
    return CONVROT_ERR_MISALIGNED;
  if ((st = check_norms(a_norm, w_norm)) != CONVROT_OK) return st;
  return run(out_dtype, a_q, ld_aq, a_scale, a_norm, w_q, ld_wq, w_scale, w_norm, bias, M, N, K_p, out, ld_out, es,
             stream);
}

extern "C" int convrot_gemm_i32(const void* a_q, int64_t ld_aq, const float* a_norm, const void* w_q,
                                int64_t ld_wq, const float* w_norm, int M, int N, int K_p, int32_t* acc,
                                int64_t ld_acc, cudaStream_t stream) {
  int st = validate_operands(a_q, ld_aq, w_q, ld_wq, M, N, K_p);
  if (st != CONVROT_OK) return st;
  if (ld_acc < N) return CONVROT_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return CONVROT_OK;
  if (!acc) return CONVROT_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(acc) % 4) return CONVROT_ERR_MISALIGNED;
  if ((st = check_norms(a_norm, w_norm)) != CONVROT_OK) return st;
  return run(-1, a_q, ld_aq, nullptr, a_norm, w_q, ld_wq, nullptr, w_norm, nullptr, M, N, K_p, acc, ld_acc, 4,
             stream);
}

extern "C" int convrot_gemm_timeout_selftest(const void* a_q, int64_t ld_aq, const float* a_norm, const void* w_q,
                                             int64_t ld_wq, const float* w_norm, int M, int N, int K_p,
                                             int32_t* acc, int64_t ld_acc, cudaStream_t stream) {
  int st = validate_operands(a_q, ld_aq, w_q, ld_wq, M, N, K_p);
  if (st != CONVROT_OK) return st;
  if (M == 0 || N == 0 || !acc || ld_acc < N) return CONVROT_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(acc) % 4) return CONVROT_ERR_MISALIGNED;
  if ((st = check_norms(a_norm, w_norm)) != CONVROT_OK) return st;
  return run(-1, a_q, ld_aq, nullptr, a_norm, w_q, ld_wq, nullptr, w_norm, nullptr, M, N, K_p, acc, ld_acc, 4,
             stream, 1);
}

extern "C" int convrot_device_error(cudaStream_t stream, int* code) {
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return convrot::record_cuda_error("cudaStreamSynchronize", e);
  int v = 0;
  e = cudaMemcpyFromSymbol(&v, g_error, sizeof(int));
  if (e != cudaSuccess) return convrot::record_cuda_error("reading the device error word", e);
  if (v != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_error, &zero, sizeof(int));
    if (e != cudaSuccess) return convrot::record_cuda_error("clearing the device error word", e);
  }
  if (code) *code = v;
  return v ? CONVROT_ERR_DEVICE_TIMEOUT : CONVROT_OK;
}
