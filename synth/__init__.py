"""Seeded synthetic inputs for the ConvRot W4A8 linear layer.

This module only *makes inputs*: random activations rounded to their storage
dtype, and random weights stored in NVFP4 (packed E2M1 nibbles, one E4M3 scale
per 16 K-elements, one FP32 tensor scale).  It holds none of the layer's own
arithmetic (no decode, no rotation, no S8 quantisation, no GEMM); both the CPU
oracle and the CUDA path consume the same bytes produced here.

Workload shapes follow the MiniMax-H3 video DiT (hidden 5376, packed qkv
[21504, 5376], SwiGLU fc1 [28672, 5376], fc2 [5376, 14336]) and the token count
M = 19989 at which the ConvRot W4A8 layer is benchmarked.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

__all__ = [
    "Workload", "WORKLOADS", "make_activations", "make_nvfp4_weight",
    "bf16_bits_from_f32", "f32_from_bf16_bits", "stored_k",
]


@dataclass(frozen=True)
class Workload:
    name: str
    M: int              # tokens
    K: int              # logical reduction width (after SwiGLU when swiglu=True)
    N: int              # output channels
    x_dtype: str        # "bf16" | "fp16" | "fp32"
    out_dtype: str      # "bf16" | "fp16" | "fp32"
    swiglu: bool        # activation input is [M, 2K] = gate | value
    outlier_frac: float # fraction of input channels scaled by outlier_mult
    outlier_mult: float
    seed: int

    @property
    def k_in(self) -> int:
        return 2 * self.K if self.swiglu else self.K


WORKLOADS = {
    "tiny": Workload("tiny", 256, 512, 512, "bf16", "bf16", False, 0.02, 20.0, 0),
    "qkv": Workload("qkv", 19989, 5376, 21504, "bf16", "bf16", False, 0.01, 20.0, 1),
    "ffn_down": Workload("ffn_down", 19989, 14336, 5376, "bf16", "bf16", True, 0.0, 1.0, 2),
    "ffn_up": Workload("ffn_up", 19989, 5376, 28672, "fp16", "fp32", False, 0.01, 20.0, 3),
    "ragged": Workload("ragged", 4097, 5000, 21500, "fp16", "fp32", False, 0.01, 20.0, 3),
    "wide_k": Workload("wide_k", 8192, 20480, 5376, "bf16", "bf16", False, 0.01, 50.0, 4),
}


def stored_k(K: int) -> int:
    """NVFP4 rows are serialised in whole 16-element scale blocks."""
    return -(-K // 16) * 16


# ----------------------------------------------------------------------------
# storage-dtype rounding of activations
# ----------------------------------------------------------------------------
def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    return ((b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def f32_from_bf16_bits(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _round_storage(x32: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return bf16_bits_from_f32(x32)
    if dtype == "fp16":
        return x32.astype(np.float16).view(np.uint16)
    if dtype == "fp32":
        return np.ascontiguousarray(x32, dtype=np.float32)
    raise ValueError(dtype)


def make_activations(wl: Workload, rows: int | None = None,
                     row_chunk: int = 4096) -> np.ndarray:
    """Activations [M, k_in] ~ N(0, 1) with a seeded set of outlier channels.

    The outlier channels (floor(outlier_frac * k_in) of them, the same for
    every token) are multiplied by ``outlier_mult``.  Returned as raw storage:
    uint16 bits for bf16/fp16, float32 for fp32.  ``rows`` truncates M (the
    first ``rows`` tokens of the same stream).
    """
    M = wl.M if rows is None else rows
    rng = np.random.default_rng(wl.seed)
    n_out = int(np.floor(wl.outlier_frac * wl.k_in))
    chans = np.sort(rng.choice(wl.k_in, size=n_out, replace=False)) if n_out else None
    out_dt = np.float32 if wl.x_dtype == "fp32" else np.uint16
    out = np.empty((M, wl.k_in), dtype=out_dt)
    xr = np.random.default_rng([wl.seed, 1])
    for r0 in range(0, M, row_chunk):
        r1 = min(M, r0 + row_chunk)
        blk = xr.standard_normal((r1 - r0, wl.k_in), dtype=np.float32)
        if chans is not None:
            blk[:, chans] *= np.float32(wl.outlier_mult)
        out[r0:r1] = _round_storage(blk, wl.x_dtype)
    return out


# ----------------------------------------------------------------------------
# NVFP4 weight storage (input encoder; the layer itself only decodes)
# ----------------------------------------------------------------------------
def _fp_grid(exp_bits: int, man_bits: int, bias: int, n_codes: int) -> np.ndarray:
    """Magnitudes of the non-negative codes 0..n_codes-1 of a small float format."""
    vals = []
    for c in range(n_codes):
        e = c >> man_bits
        m = c & ((1 << man_bits) - 1)
        if e == 0:
            vals.append(m / (1 << man_bits) * 2.0 ** (1 - bias))
        else:
            vals.append((1 + m / (1 << man_bits)) * 2.0 ** (e - bias))
    return np.array(vals, dtype=np.float64)


_E2M1_GRID = _fp_grid(2, 1, 1, 8)          # 0 .. 6
_E4M3_GRID = _fp_grid(4, 3, 7, 127)        # 0 .. 448 (code 127 is NaN, unused)


def _nearest_code(v: np.ndarray, grid: np.ndarray) -> np.ndarray:
    """Index of the nearest grid value to v >= 0; ties go to the even code."""
    v = np.minimum(v, grid[-1])
    hi = np.clip(np.searchsorted(grid, v, side="left"), 1, len(grid) - 1)
    lo = hi - 1
    d_lo = v - grid[lo]
    d_hi = grid[hi] - v
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    return np.where(pick_hi, hi, lo).astype(np.uint8)


def _nearest_e2m1(v: np.ndarray) -> np.ndarray:
    """Nearest E2M1 magnitude code of v >= 0 (same rule as _nearest_code, ties to
    the even code), by counting the midpoints of the grid that v lies above."""
    mids = 0.5 * (_E2M1_GRID[1:] + _E2M1_GRID[:-1])
    code = np.zeros(v.shape, dtype=np.uint8)
    for i, m in enumerate(mids):
        m = np.float32(m)
        # a tie goes up when the upper neighbour (code i+1) is even
        code += (v >= m) if (i + 1) % 2 == 0 else (v > m)
    return code


def make_nvfp4_weight(wl: Workload, rows: int | None = None, std: float = 0.02,
                      row_chunk: int = 2048):
    """Weights W [N, K] ~ N(0, std) stored as NVFP4.

    Returns (packed uint8 [N, K_s/2], scales uint8 [N, K_s/16], tensor_scale
    float32).  Deterministic round-to-nearest quantiser: tensor scale
    t = max|W| / (6 * 448); block scale = nearest E4M3 of max|block| / (6 t);
    element = nearest E2M1 of w / (scale * t).  Byte j of a row holds element
    2j in its low nibble and 2j+1 in its high nibble.  Elements K..K_s-1 of a
    row (serialised padding) are stored as zero nibbles.
    """
    N = wl.N if rows is None else rows
    K, Ks = wl.K, stored_k(wl.K)
    rng = np.random.default_rng([wl.seed, 2])
    W = (rng.standard_normal((wl.N, K), dtype=np.float32) * np.float32(std))[:N]
    t = np.float32(np.max(np.abs(W)) / np.float32(6.0 * 448.0))
    packed = np.empty((N, Ks // 2), dtype=np.uint8)
    scales = np.empty((N, Ks // 16), dtype=np.uint8)
    for r0 in range(0, N, row_chunk):
        r1 = min(N, r0 + row_chunk)
        w = np.zeros((r1 - r0, Ks), dtype=np.float64)
        w[:, :K] = W[r0:r1]
        blk = w.reshape(r1 - r0, Ks // 16, 16)
        amax = np.max(np.abs(blk), axis=2)
        sc = _nearest_code(amax / 6.0 / float(t), _E4M3_GRID)
        sval = _E4M3_GRID[sc] * float(t)
        with np.errstate(divide="ignore", invalid="ignore"):
            v = np.where(sval[..., None] > 0, blk / sval[..., None], 0.0)
        mag = _nearest_e2m1(np.abs(v).astype(np.float32))
        nib = np.where((v < 0) & (mag > 0), mag | 8, mag).astype(np.uint8)
        nib = nib.reshape(r1 - r0, Ks)
        packed[r0:r1] = nib[:, 0::2] | (nib[:, 1::2] << 4)
        scales[r0:r1] = sc
    return packed, scales, t
