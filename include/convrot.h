/*
 * convrot.h -- C ABI of the ConvRot W4A8 linear layer for GB300 (sm_103a).
 *
 * The layer (ComfyUI Turing Utils page on comfy.icu, node list, the entry on
 * the ConvRot DiT / CLIP loaders reading native NVFP4 layers; cited below as
 * "the NVFP4 loader entry") keeps its weights in NVFP4, applies the same 256-point block rotation
 * (paired ConvRot256) to the activations and to the decoded weights,
 * quantises both to row-scaled S8 and multiplies them with an integer GEMM
 * whose epilogue dequantises to BF16 / FP16 / FP32:
 *
 *     y[m, n] = s_a[m] * s_w[n] * sum_k q_a[m, k] * q_w[n, k]
 *
 * Three calls make one layer: convrot_prepare_weight (NVFP4 decode + FP32
 * rotation + S8 quantisation of the weight rows), convrot_quant_act
 * ((SwiGLU +) FP32 rotation + S8 quantisation of the token rows) and
 * convrot_gemm (integer GEMM + dequant epilogue).
 *
 * Conventions shared by every call:
 *   - Every pointer is a DEVICE pointer owned by the caller; nothing is
 *     allocated, freed or retained by the library.
 *   - Work is enqueued on `stream` (0 = legacy default stream) and the call
 *     returns without synchronising.  Outputs are valid once the stream has
 *     reached the work.  Since the three layer calls only enqueue kernels,
 *     a caller may capture them into a CUDA graph (after one eager call on
 *     the device, which sets up per-device launch attributes) and replay it
 *     on new contents of the same buffers.
 *   - Matrices are row-major.  Leading dimensions (ld_*) count ELEMENTS of
 *     the matrix's own storage type.
 *   - K is the logical reduction width; K_p = convrot_padded_k(K) is K
 *     rounded up to a multiple of 256 (both operands are zero-padded before
 *     the rotation).  K_p <= CONVROT_MAX_KP.
 *   - M == 0 or N == 0 is a valid empty call (nothing is launched).
 *   - Return value: CONVROT_OK or one of the error codes below.  A failing
 *     call launches nothing and leaves the outputs untouched.  No call
 *     aborts or throws.
 *
 * S8 code storage.  The rotated operands are quantised to integer codes in
 * [-127, 127].  They can be written either as int8 (CONVROT_CODES_S8, one
 * byte per code) or as FP16 values holding the same integers exactly
 * (CONVROT_CODES_F16, two bytes per code).  convrot_gemm reads the FP16
 * form: sm_103a tensor cores have no 8-bit integer MMA, so the GEMM runs the
 * FP16 tensor-core path, whose FP32 accumulation of these integer products
 * is exact while partial sums stay below 2^24: it converts to int32 every
 * 1024 K, or once per output tile when the rows' code-norm bounds show that
 * no partial sum can reach 2^24.  The int32 accumulator is therefore
 * bit-exact either way.
 */
#ifndef CONVROT_H
#define CONVROT_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CONVROT_BLOCK 256          /* rotation block (ConvRot256)           */
#define CONVROT_MAX_KP 65536       /* largest padded K accepted             */

typedef enum {
    CONVROT_OK = 0,
    CONVROT_ERR_INVALID_ARG = 1,   /* null pointer, negative size, ld too small, ... */
    CONVROT_ERR_MISALIGNED = 2,    /* a pointer / pitch breaks an alignment rule     */
    CONVROT_ERR_UNSUPPORTED = 3,   /* dtype / code format / K_p beyond the limit     */
    CONVROT_ERR_CUDA = 4,          /* a CUDA launch or runtime call failed           */
    CONVROT_ERR_DEVICE_TIMEOUT = 5 /* a kernel gave up waiting (see convrot_device_error) */
} convrot_status;

typedef enum { CONVROT_BF16 = 0, CONVROT_FP16 = 1, CONVROT_FP32 = 2 } convrot_dtype;

typedef enum { CONVROT_CODES_S8 = 0, CONVROT_CODES_F16 = 1 } convrot_codes;

/* K rounded up to a multiple of CONVROT_BLOCK; 0 for K <= 0. */
int convrot_padded_k(int K);

/* Human-readable name of a status code (static string, never NULL). */
const char* convrot_status_string(int status);

/*
 * Weight preparation: NVFP4 decode + ConvRot256 rotation in FP32 + row-scaled
 * S8 quantisation in one fused step.  Source: the NVFP4 loader entry's weight
 * path -- the NVFP4 tensor is decoded, rotated in FP32 by the same ConvRot256
 * as the activations and quantised per row with a rounded FP32 reciprocal of
 * the row scale, and the serialised padding past K is skipped.  The stored
 * NVFP4 bytes are only read.
 *
 * Row ranges: the call has no row-offset argument.  To prepare rows
 * [n0, n0 + n) of a weight, pass w_fp4 + n0 * (K_s/2), w_sf + n0 * (K_s/16),
 * w_q + n0 * ld_wq (in code elements), w_scale + n0 and (if used)
 * w_norm + n0 with N = n; rows are
 * independent, so the result equals that of the whole-weight call (the
 * alignment rules below apply to the offset pointers).
 *
 *   w_fp4   [N][K_s/2] uint8, K_s = ceil(K/16)*16, rows contiguous.  Byte j of
 *           a row holds element 2j in its low nibble, 2j+1 in its high nibble;
 *           each nibble is an E2M1 code (sign bit 3).  Elements K..K_s-1 are
 *           serialised padding and are ignored whatever they hold.
 *   w_sf    [N][K_s/16] uint8 E4M3 ("FN") block scales, row-major.
 *   w_tensor_scale  one FP32 (device memory): the NVFP4 tensor scale t.
 *   w_q     [N][ld_wq] codes in `fmt`, columns 0..K_p-1 written (the zero
 *           padding included); ld_wq >= K_p.
 *   w_scale [N] FP32 row scales s_w (0 for a degenerate row).
 *   w_norm  NULL, or [N] FP32 (4-byte aligned): an upper bound on the
 *           Euclidean norm of each row's codes, for convrot_gemm (see there;
 *           the cost and the codes as for convrot_quant_act's a_norm).
 *
 * Decoded weight w = E2M1 * E4M3 * t.  Per row: r = rotate(w padded to K_p);
 * s_w = fp32(max|r| / 127); q = clamp(rint(r * fp32(1/s_w)), -127, 127), the
 * product and rounding done in FP32 (half to even).  A row whose s_w is 0 or
 * whose reciprocal overflows is written as all-zero codes with s_w = 0.
 * A row holding an Inf or NaN value gets unspecified codes and scale.
 * Alignment: w_fp4 8-byte aligned; w_q 4-byte (F16 codes) or 2-byte (S8
 * codes) aligned with ld_wq even (codes are written in pairs).
 */
int convrot_prepare_weight(const uint8_t* w_fp4, const uint8_t* w_sf,
                           const float* w_tensor_scale, int N, int K,
                           void* w_q, convrot_codes fmt, int64_t ld_wq,
                           float* w_scale, float* w_norm, cudaStream_t stream);

/*
 * Activation quantisation: optional SwiGLU prologue, optional channel
 * pre-scales, then ConvRot256 rotation in FP32 and row-scaled S8 quantisation.
 * Source: the NVFP4 loader entry's activation path -- ConvRot256 on the
 * activations, one INT8 scale per token row, FP16 inputs rotated and
 * quantised in FP32; the channel pre-scales and SwiGLU are applied before the
 * rotation, SwiGLU fused into it with no BF16 rounding of its result.  The
 * SwiGLU itself (gate = first half, value = second half, swish(gate) * value)
 * is the MLP section of the MiniMax-H3 explainer on modelpad.app.
 *
 *   x       [M][ld_x] in x_dtype (BF16 / FP16 / FP32).  swiglu == 0: columns
 *           0..K-1 are the input.  swiglu != 0: columns 0..K-1 are the gate
 *           g and K..2K-1 the value v, and the layer input is
 *           h = g * sigmoid(g) * v computed in FP32 with no intermediate
 *           rounding.  ld_x >= K (or 2K).
 *   pre_scale  NULL, or [K] FP32 channel multipliers (16-byte aligned): the
 *           layer input becomes h[m, k] * pre_scale[k] (after SwiGLU, before
 *           the rotation, in FP32).
 *   a_q     [M][ld_aq] codes in `fmt`, columns 0..K_p-1 written; ld_aq >= K_p.
 *   a_scale [M] FP32 token scales s_a (0 for a degenerate row).
 *   a_norm  NULL, or [M] FP32 (4-byte aligned): an upper bound on the
 *           Euclidean norm of each row's codes, for convrot_gemm.  Asking
 *           for it adds a sum of squares to the kernel (a few percent of its
 *           time); the bounds let the GEMM run a tile as one chunk, which
 *           for ordinary rotated data holds up to K_p of about 8192 (at
 *           K_p = 5376 the drains it skips cost about as much, 1% of the
 *           GEMM).
 *           The codes and scales are the same either way.
 *
 * Quantiser as for the weights (FP32 scale, FP32 reciprocal, FP32 product,
 * round half to even, clamp to +-127).  A row holding an Inf or NaN value
 * gets unspecified codes and scale.  FP16 inputs are widened to FP32
 * before anything else.  x needs only element alignment; rows aligned to 32
 * or 16 bytes take the vectorised load paths.  a_q is 4-byte (F16 codes) or
 * 2-byte (S8 codes) aligned with ld_aq even (codes are written in pairs).
 */
int convrot_quant_act(const void* x, convrot_dtype x_dtype, int64_t ld_x,
                      int M, int K, int swiglu, const float* pre_scale,
                      void* a_q, convrot_codes fmt, int64_t ld_aq,
                      float* a_scale, float* a_norm, cudaStream_t stream);

/*
 * Integer GEMM with the dequantising epilogue.  Source: the NVFP4 loader
 * entry's GEMM -- an INT8 tensor-core product of the row-scaled operands with
 * logical N tails and FP16, BF16 or FP32 outputs; the rescale sits inside the
 * matmul (the MiniMax-H3 explainer's table on moving the rescaling into the
 * matmul), so no int32 matrix is ever written.
 *
 *   a_q     [M][ld_aq] FP16-stored S8 codes of the rotated activations.
 *   w_q     [N][ld_wq] FP16-stored S8 codes of the rotated weights.
 *   a_scale [M], w_scale [N] FP32 row scales (w_scale 16-byte aligned).
 *   a_norm, w_norm  NULL, or the [M] and [N] code-norm bounds written by
 *           convrot_quant_act and convrot_prepare_weight (4-byte aligned;
 *           both are needed, one alone is ignored).
 *           The tensor cores accumulate in FP32, so the int32 result is exact
 *           only while every partial sum stays below 2^24.  Without the
 *           bounds the K loop is cut into exact chunks of at most 1024
 *           (127^2 * 1024 < 2^24), each drained to int32.  With them, a
 *           256 x 256 output tile whose largest a_norm times largest w_norm
 *           is below 2^24 runs as one chunk: by Cauchy-Schwarz every partial
 *           sum of q_a[m, :] . q_w[n, :], in any order, is at most
 *           ||q_a[m, :]|| ||q_w[n, :]||.  The result is the same int32 sum;
 *           only the number of drains changes.  Bounds smaller than the true
 *           norms void that guarantee.
 *   bias    NULL, or [N] FP32 per-output-channel bias (16-byte aligned).
 *   K_p     padded reduction width, a multiple of 256, <= CONVROT_MAX_KP.
 *   out     [M][ld_out] in out_dtype; ld_out >= N.  Only columns 0..N-1 of
 *           rows 0..M-1 are written.
 *
 * y[m, n] = fp32(acc) * s_a[m] * s_w[n] (+ bias[n]) in FP32, rounded to
 * out_dtype (nearest even).  acc is the exact int32 sum over K_p.
 * Alignment: a_q and w_q 16-byte aligned with ld_aq, ld_wq multiples of 8
 * (TMA rule); out needs only element alignment (a 16-byte aligned out with a
 * 16-byte multiple pitch is written by TMA tensor stores, any other by
 * per-element stores).
 */
int convrot_gemm(const void* a_q, int64_t ld_aq, const float* a_scale,
                 const float* a_norm, const void* w_q, int64_t ld_wq,
                 const float* w_scale, const float* w_norm,
                 const float* bias, int M, int N, int K_p,
                 void* out, convrot_dtype out_dtype, int64_t ld_out,
                 cudaStream_t stream);

/*
 * W8A8 with resident weights: widens S8 codes (CONVROT_CODES_S8, e.g. weight
 * codes prepared once and kept at one byte each) into the FP16-held codes
 * that convrot_gemm reads.  Source: the NVFP4 loader entry's W8A8 comparison,
 * which runs on these same rotated S8 weights derived from the NVFP4
 * checkpoint.
 *
 *   src  [rows][ld_src] int8, 16-byte aligned, ld_src a multiple of 16.
 *   dst  [rows][ld_dst] FP16, 16-byte aligned, ld_dst a multiple of 8.
 *   cols a multiple of 16; columns 0..cols-1 are converted exactly.
 */
int convrot_widen_codes(const int8_t* src, int64_t ld_src, int rows, int cols,
                        void* dst, int64_t ld_dst, cudaStream_t stream);

/*
 * Test hook: the same GEMM, writing the raw int32 accumulators
 * acc[m, n] = sum_k q_a[m, k] * q_w[n, k] into acc [M][ld_acc] instead of
 * dequantising.  Arguments and rules as convrot_gemm (a_norm and w_norm
 * choose the chunking the same way).
 */
int convrot_gemm_i32(const void* a_q, int64_t ld_aq, const float* a_norm,
                     const void* w_q, int64_t ld_wq, const float* w_norm,
                     int M, int N, int K_p,
                     int32_t* acc, int64_t ld_acc, cudaStream_t stream);

/*
 * Failure-detection self-test: launches the GEMM of convrot_gemm_i32 on the
 * given operands with its TMA producer switched off, so the first wait for
 * operand tiles runs out (after about two seconds).  The kernel then records
 * the failure, drains and returns; acc is left incomplete.  Afterwards
 * convrot_device_error reports CONVROT_ERR_DEVICE_TIMEOUT with a nonzero
 * code, and the CUDA context stays usable.  With norm bounds (as for
 * convrot_gemm_i32) and K_p > 1024, the warp that hands chunk counts to the
 * MMA issuer runs as well and must leave its waits on the abort too.  Returns
 * the launch status.
 */
int convrot_gemm_timeout_selftest(const void* a_q, int64_t ld_aq, const float* a_norm,
                                  const void* w_q, int64_t ld_wq, const float* w_norm,
                                  int M, int N, int K_p,
                                  int32_t* acc, int64_t ld_acc, cudaStream_t stream);

/*
 * Measurement aid, not part of the layer (the pages have no counterpart): runs
 * the warp-level INT8 tensor instruction (mma.sync m16n8k32, s8 x s8 -> s32)
 * from registers, `blocks` CTAs of 4 warps, each warp issuing 8 independent
 * MMAs per iteration for `iters` iterations (2 * 16 * 8 * 32 = 8192 integer
 * operations per MMA).  Every operand byte is 1, so each warp writes
 * 8 * 32 * iters to out[warp] (out: blocks * 4 int32, device).  Timing the
 * call gives this GPU's INT8 rate on that path, the denominator of "% of
 * INT8 roofline".  iters in [1, 2^22].
 */
int convrot_int8_mma_probe(int blocks, int iters, int32_t* out, cudaStream_t stream);

/*
 * Measurement aid, not part of the layer: the producer side of a GEMM that
 * would decode, rotate and quantise the NVFP4 weight inside the GEMM.  The
 * pages run the weight work beside the GEMM instead (ComfyUI Turing Utils
 * page, node list, the ConvRot loaders' NVFP4 entry); this measures the
 * fused form.  One CTA per SM runs the m_strips * ceil(N/128) work units of a
 * GEMM over m_strips strips of 256 tokens.  For unit u, producer_warps (8 or
 * 16) warps build the FP16 codes of weight rows 128 * (u % ceil(N/128)) +
 * [0, 128) over the padded K, one 256-column rotation block at a time, in the
 * tensor core's swizzled shared-memory layout (two 64 KiB stages), and one
 * consumer warp releases each stage as soon as it is full.  A fused GEMM is
 * no faster than this producer.
 *   w_fp4, w_sf, w_tensor_scale, N, K   as for convrot_prepare_weight.
 *   w_scale  [N] FP32 row scales that convrot_prepare_weight wrote for this
 *            weight (a fused layer needs a scales-only pass first).
 *   dump     optional (NULL: none), device FP16 [128][ld_dump], ld_dump >=
 *            K_p and even, 4-byte aligned: receives the codes of unit
 *            dump_unit (rows past N as zeros).  They equal rows
 *            128 * (dump_unit % ceil(N/128)) + [0, 128) of
 *            convrot_prepare_weight's FP16 codes.
 *   status   device int32, set to 0 by the call; the kernel writes a nonzero
 *            code there if a wait runs out (about two seconds).
 * Returns the launch status.
 */
int convrot_decode_gemm_probe(const uint8_t* w_fp4, const uint8_t* w_sf, const float* w_tensor_scale,
                              const float* w_scale, int N, int K, int m_strips, int producer_warps,
                              void* dump, int64_t ld_dump, int dump_unit, int32_t* status,
                              cudaStream_t stream);

/*
 * Text of the last CUDA error that made a call of this library return
 * CONVROT_ERR_CUDA in the calling thread, naming the failing CUDA call
 * ("" if none).  The string is owned by the library and stays valid until
 * the thread's next failing call.
 */
const char* convrot_last_error(void);

/*
 * Device-side failure report.  Kernels that wait on asynchronous copies or
 * tensor-core work give up after about two seconds, record a nonzero code in
 * a device word and return early (their outputs are then incomplete).  This
 * call synchronises `stream`, copies the word to *code (0 = no failure),
 * clears it and returns CONVROT_ERR_DEVICE_TIMEOUT if it was set,
 * CONVROT_OK otherwise.  `code` may be NULL.
 */
int convrot_device_error(cudaStream_t stream, int* code);

#ifdef __cplusplus
}
#endif

#endif /* CONVROT_H */
