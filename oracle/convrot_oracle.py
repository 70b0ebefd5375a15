"""Plain, slow CPU oracle of the ConvRot W4A8 linear layer.

TEST INFRASTRUCTURE ONLY: used by tests, the smoke check and the benchmark's
CPU baseline; never by the product path.  Shares no code with the CUDA side.

What the layer computes (ComfyUI Turing Utils page on comfy.icu, node list,
the entry on the ConvRot DiT / CLIP loaders reading native NVFP4 layers):

  1. decode the NVFP4 weight W[n, k] = E2M1(nibble) * E4M3(block scale) *
     FP32 tensor scale for k < K (serialised padding ignored);
  2. zero-pad both operands to K_p = ceil(K / 256) * 256;
  3. apply the same ConvRot256 block rotation to activations and weights, so
     that (x R)(W R)^T = x W^T;
  4. quantise both to row-scaled symmetric S8 (one FP32 scale per token row
     and per weight row) -- the weight side multiplies by a rounded FP32
     reciprocal of its scale;
  5. integer GEMM of the S8 codes with exact int32 accumulation;
  6. dequantise y = acc * s_a[m] * s_w[n] into BF16 / FP16 / FP32.

An optional SwiGLU prologue (MiniMax-H3 explainer on modelpad.app, MLP
section: gate, value = fc1(x).chunk(2); hidden = swish(gate) * value) runs
on the activations before the rotation, without intermediate rounding.

Precision: FP64 throughout, except where the method fixes FP32: the rotated
operands are held in FP32 (the page rotates the weights in FP32, and rotates
and quantises FP16 inputs in FP32), and the S8 code of every element is
decided in FP32 (FP32 scale, FP32 reciprocal, FP32 product, round half to
even).

Readings where the pages are silent (each listed with its reason in the
design notes):
  * ConvRot256's matrix is never printed.  The modelpad glossary names a
    Hadamard rotation, i.e. an orthogonal matrix with entries of +-1 before
    normalisation; we take the normalised 256-point Sylvester Walsh-Hadamard
    matrix R = H_256 / 16.
  * E2M1 / E4M3 follow the OCP Microscaling and OFP8 definitions (E4M3 "FN":
    bias 7, no infinities, S.1111.111 is NaN).
  * Nibble order: byte j of a row holds element 2j in its low nibble.
  * Scale layout: plain row-major [N, K_s / 16].
  * S8 range is symmetric [-127, 127]; rounding is half to even.
  * A row whose FP32 scale is zero, or whose FP32 reciprocal overflows, is a
    degenerate row: its scale is stored as 0 and all of its codes are 0.
  * The activation side uses the same quantiser as the weight side.
  * Channel pre-scales (which the page places before the rotation, like
    SwiGLU) multiply the layer's input channel-wise after SwiGLU and before
    the rotation; the optional bias is added in FP32 before the output
    rounding.

Pins: every step is checked against something other than this file in the
oracle pin tests (the OCP tables, closed forms of the rotation, invariance
of the rotated product, brute-force integer GEMMs, single-rounding output
cases, the pages' printed 1.31% / 1.39% added error).  Exact reproduction of
the pages' own codes is parity unpinned: the pages print no vectors.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "BLOCK", "padded_k", "e2m1_value", "e4m3_value", "decode_nvfp4",
    "hadamard_sylvester", "rotation_matrix", "rotate_blocks", "swiglu",
    "quantize_rows", "int_gemm", "round_to_dtype", "dequantize",
    "prepare_weight", "quant_act", "convrot_linear", "storage_to_f64",
]

BLOCK = 256


def padded_k(K: int) -> int:
    """ConvRot256 needs K padded with zeros to a whole number of 256-blocks."""
    return -(-K // BLOCK) * BLOCK


# ----------------------------------------------------------------------------
# step 1: NVFP4 decode
# ----------------------------------------------------------------------------
def e2m1_value(code: int) -> float:
    """Value of a 4-bit E2M1 code: 1 sign, 2 exponent (bias 1), 1 mantissa bit."""
    sign = -1.0 if (code >> 3) & 1 else 1.0
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:                                   # subnormal: 0 or 0.5
        mag = m * 0.5
    else:
        mag = (1.0 + 0.5 * m) * 2.0 ** (e - 1)
    return sign * mag


def e4m3_value(code: int) -> float:
    """Value of an 8-bit E4M3 ("FN") code: bias 7, subnormals, no inf, NaN=S.1111.111."""
    sign = -1.0 if (code >> 7) & 1 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        mag = (m / 8.0) * 2.0 ** -6
    else:
        mag = (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return sign * mag


_E2M1 = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)
_E4M3 = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)


def decode_nvfp4(packed: np.ndarray, scales: np.ndarray, tensor_scale, K: int) -> np.ndarray:
    """W[n, k] = E2M1(nib) * E4M3(scale[n, k // 16]) * t for k < K, in FP64.

    ``packed`` is [N, K_s/2] uint8 (element 2j in the low nibble of byte j),
    ``scales`` is [N, K_s/16] uint8.  Elements K..K_s-1 are serialised padding
    and are ignored.  Every product here is exact in FP64.
    """
    packed = np.asarray(packed, dtype=np.uint8)
    N, half = packed.shape
    nib = np.empty((N, 2 * half), dtype=np.uint8)
    nib[:, 0::2] = packed & 0x0F
    nib[:, 1::2] = packed >> 4
    vals = _E2M1[nib[:, :K]]
    blk_scale = _E4M3[np.asarray(scales, dtype=np.uint8)]          # [N, K_s/16]
    per_elem = np.repeat(blk_scale, 16, axis=1)[:, :K]
    return vals * per_elem * float(np.float32(tensor_scale))


# ----------------------------------------------------------------------------
# steps 2-3: zero padding and ConvRot256 rotation
# ----------------------------------------------------------------------------
def hadamard_sylvester(n: int = BLOCK) -> np.ndarray:
    """Unnormalised Sylvester Hadamard matrix: H_1 = [1], H_2m = [[H, H], [H, -H]]."""
    H = np.ones((1, 1), dtype=np.float64)
    while H.shape[0] < n:
        H = np.block([[H, H], [H, -H]])
    if H.shape[0] != n:
        raise ValueError("n must be a power of two")
    return H


def rotation_matrix() -> np.ndarray:
    """R = H_256 / 16: orthogonal, so R R^T = I and x W^T = (x R)(W R)^T."""
    return hadamard_sylvester(BLOCK) / math.sqrt(BLOCK)


def rotate_blocks(x: np.ndarray, R: np.ndarray | None = None) -> np.ndarray:
    """Zero-pad rows of x [rows, K] to K_p and right-multiply each 256-block by R."""
    if R is None:
        R = rotation_matrix()
    x = np.asarray(x, dtype=np.float64)
    rows, K = x.shape
    Kp = padded_k(K)
    xp = np.zeros((rows, Kp), dtype=np.float64)
    xp[:, :K] = x
    nb = Kp // BLOCK
    return (xp.reshape(rows, nb, BLOCK) @ R).reshape(rows, Kp)


# ----------------------------------------------------------------------------
# optional prologue: SwiGLU
# ----------------------------------------------------------------------------
def swiglu(x2: np.ndarray, K: int) -> np.ndarray:
    """hidden = swish(gate) * value with gate = x2[:, :K], value = x2[:, K:2K] (FP64)."""
    x2 = np.asarray(x2, dtype=np.float64)
    gate = x2[:, :K]
    value = x2[:, K:2 * K]
    return gate / (1.0 + np.exp(-gate)) * value


# ----------------------------------------------------------------------------
# step 4: row-scaled S8 quantisation, decided in FP32
# ----------------------------------------------------------------------------
def quantize_rows(xhat: np.ndarray):
    """Row-scaled symmetric S8 codes of the rotated rows.

    In FP32: v = fp32(xhat); s = fp32(max|v| / 127); r = fp32(1 / s);
    q = clamp(rint(fp32(v * r)), -127, 127) with rint = half to even.
    Degenerate rows (s == 0 or r not finite) get s = 0 and q = 0.
    Returns (q int8 [rows, K_p], s float32 [rows]).
    """
    v = np.asarray(xhat, dtype=np.float64).astype(np.float32)
    amax = np.max(np.abs(v), axis=1)
    s = (amax / np.float32(127.0)).astype(np.float32)
    with np.errstate(divide="ignore", over="ignore", invalid="ignore"):
        r = (np.float32(1.0) / s).astype(np.float32)
        prod = (v * r[:, None]).astype(np.float32)
    degenerate = (s == 0) | ~np.isfinite(r)
    prod[degenerate] = 0.0
    q = np.clip(np.rint(prod), -127, 127).astype(np.int8)
    s = np.where(degenerate, np.float32(0.0), s).astype(np.float32)
    return q, s


# ----------------------------------------------------------------------------
# step 5: exact integer GEMM
# ----------------------------------------------------------------------------
def int_gemm(qa: np.ndarray, qw: np.ndarray) -> np.ndarray:
    """acc[m, n] = sum_k qa[m, k] * qw[n, k], exact, returned as int64.

    The float64 matrix product is exact here: every product is an integer of
    magnitude <= 127^2 and every partial sum stays far below 2^53.
    """
    qa = np.asarray(qa)
    qw = np.asarray(qw)
    if qa.shape[1] != qw.shape[1]:
        raise ValueError("K mismatch")
    bound = 127 * 127 * qa.shape[1]
    if bound >= 2 ** 53:
        raise ValueError("K too large for an exact float64 product")
    acc = qa.astype(np.float64) @ qw.astype(np.float64).T
    out = acc.astype(np.int64)
    if np.any(np.abs(out) >= 2 ** 31):
        raise OverflowError("int32 accumulator overflow")
    return out


# ----------------------------------------------------------------------------
# step 6: dequantisation and output rounding
# ----------------------------------------------------------------------------
def _round_significand(y: np.ndarray, man_bits: int, emin: int, emax_val: float) -> np.ndarray:
    """Round FP64 values once to a binary format with man_bits stored mantissa bits."""
    y = np.asarray(y, dtype=np.float64)
    out = np.zeros_like(y)
    nz = y != 0
    a = np.abs(y[nz])
    e = np.floor(np.log2(a)).astype(np.int64)
    # log2 may be off by one near powers of two; fix with exact comparisons
    e = np.where(np.ldexp(1.0, e) > a, e - 1, e)
    e = np.where(np.ldexp(1.0, e + 1) <= a, e + 1, e)
    e = np.maximum(e, emin)                       # subnormal range: fixed quantum
    quantum_exp = e - man_bits
    r = np.ldexp(np.rint(np.ldexp(a, -quantum_exp)), quantum_exp)   # rint = ties to even
    r = np.where(r > emax_val, np.inf, r)
    out[nz] = np.sign(y[nz]) * r
    return out


_BF16_MAX = float.fromhex("0x1.fep127")
_FP16_MAX = 65504.0


def round_to_dtype(y: np.ndarray, dtype: str) -> np.ndarray:
    """Round FP64 once (nearest, ties to even) to bf16/fp16/fp32; returned as FP64."""
    if dtype == "fp32":
        return np.asarray(y, dtype=np.float64).astype(np.float32).astype(np.float64)
    if dtype == "bf16":
        # values beyond max+half-ulp overflow to inf
        return _round_significand(y, 7, -126, _BF16_MAX)
    if dtype == "fp16":
        return _round_significand(y, 10, -14, _FP16_MAX)
    raise ValueError(dtype)


def dequantize(acc: np.ndarray, sa: np.ndarray, sw: np.ndarray, out_dtype: str,
               bias: np.ndarray | None = None) -> np.ndarray:
    """y[m, n] = acc[m, n] * s_a[m] * s_w[n] (+ bias[n]) in FP64, then one rounding.

    The bias is the linear layer's y = x W^T + b (MiniMax-H3 explainer on
    modelpad.app, "Foundations"); the ConvRot entry names none, so it is
    optional.
    """
    y = (np.asarray(acc, dtype=np.float64)
         * np.asarray(sa, dtype=np.float64)[:, None]
         * np.asarray(sw, dtype=np.float64)[None, :])
    if bias is not None:
        y = y + np.asarray(bias, dtype=np.float32).astype(np.float64)[None, :]
    return round_to_dtype(y, out_dtype)


# ----------------------------------------------------------------------------
# the three calls of the layer, composed
# ----------------------------------------------------------------------------
def storage_to_f64(x: np.ndarray, dtype: str) -> np.ndarray:
    """Interpret raw activation storage (uint16 bits for bf16/fp16) as FP64."""
    x = np.asarray(x)
    if dtype == "bf16":
        return (x.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    if dtype == "fp16":
        return x.view(np.float16).astype(np.float64)
    if dtype == "fp32":
        return x.astype(np.float64)
    raise ValueError(dtype)


def prepare_weight(packed, scales, tensor_scale, K: int):
    """Decode NVFP4 -> pad -> rotate -> row-scaled S8.  Returns (q_w, s_w)."""
    w = decode_nvfp4(packed, scales, tensor_scale, K)
    return quantize_rows(rotate_blocks(w))


def quant_act(x_storage, x_dtype: str, K: int, swiglu_flag: bool = False, pre_scale=None):
    """(SwiGLU ->) (channel pre-scale ->) pad -> rotate -> row-scaled S8.

    Channel pre-scales multiply the layer's input h[:, k] by p[k] before the
    rotation.  The page places pre-scales and SwiGLU before the rotation and
    keeps the order of the unfused computation; read here as: the scale
    belongs to this layer's input, so it follows the SwiGLU that produces
    that input.
    Returns (q_a, s_a).
    """
    x = storage_to_f64(x_storage, x_dtype)
    h = swiglu(x, K) if swiglu_flag else x[:, :K]
    if pre_scale is not None:
        h = h * np.asarray(pre_scale, dtype=np.float32).astype(np.float64)[None, :K]
    return quantize_rows(rotate_blocks(h))


def convrot_linear(x_storage, x_dtype, packed, scales, tensor_scale, K, out_dtype,
                   swiglu_flag=False, pre_scale=None, bias=None):
    """The whole layer; returns (y as FP64 holding out_dtype values, intermediates)."""
    qw, sw = prepare_weight(packed, scales, tensor_scale, K)
    qa, sa = quant_act(x_storage, x_dtype, K, swiglu_flag, pre_scale)
    acc = int_gemm(qa, qw)
    y = dequantize(acc, sa, sw, out_dtype, bias)
    return y, dict(qa=qa, sa=sa, qw=qw, sw=sw, acc=acc)
