"""GPU parity on the method's edge cases, against the CPU oracle.

NVFP4 weights that come from another quantiser can hold any byte: every E2M1
nibble (including -0, code 8) in any mix within a block, and any non-NaN E4M3
block scale -- zero, the subnormals 0x01..0x07, the largest value 448 (0x7E),
scales with the sign bit set -- with a tensor scale far from 1.  The Load
ConvRot DiT entry of the ComfyUI Turing Utils page (comfy.icu, node list)
has the layer read ComfyUI-native NVFP4 checkpoints, so the decode must hold
on the whole code space, not only on the synthetic encoder's scale band.

SwiGLU (MiniMax-H3 explainer on modelpad.app, MLP section), fused in FP32
before the rotation, must hold for gates far into both tails, where exp(-g)
overflows or underflows in FP32, with no intermediate rounding of the
hidden value.

Bars as everywhere: codes >= 99.99% equal with |diff| <= 1, scales within
1e-6 relative (zero where the oracle's is zero).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import (assert_codes_match, assert_scales_match, codes_to_np, ensure_built,
                      gpu_prepare_weight, gpu_quant_act)

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

E4M3_NAN = (0x7F, 0xFF)


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    import rotated_w4a8_int8_gb300 as cr
    yield
    assert cr.device_error() == 0


def random_nvfp4(N, K, seed):
    """Uniformly random packed nibbles and uniformly random non-NaN E4M3 scale
    bytes; the first rows hold the named special scales in every block."""
    rng = np.random.default_rng(seed)
    Ks = synth.stored_k(K)
    packed = rng.integers(0, 256, (N, Ks // 2), dtype=np.uint8)
    scales = rng.integers(0, 256, (N, Ks // 16), dtype=np.uint8)
    nan = np.isin(scales, E4M3_NAN)
    scales[nan] = rng.integers(0, 0x7F, int(nan.sum()), dtype=np.uint8)
    special = [
        np.arange(1, 8, dtype=np.uint8),                     # positive subnormals
        np.arange(0x81, 0x88, dtype=np.uint8),               # negative subnormals
        np.array([0x00, 0x80], dtype=np.uint8),              # +0, -0 scales (zero blocks)
        np.array([0x7E, 0xFE], dtype=np.uint8),              # +-448
        np.array([0x01, 0x7E], dtype=np.uint8),              # smallest next to largest
    ]
    for i, vals in enumerate(special):
        if i < N:
            scales[i] = np.resize(vals, scales.shape[1])
    if N > len(special):
        packed[len(special)] = 0x88                          # every element -0
    return packed, scales


RANDOM_W_CASES = [
    # (K, N, tensor scale): ragged K (K_s = 5008, odd scale count, no 16-byte
    # loads), K_p = 16384 (64 blocks, one CTA), K_p > 32768 (rows split over a
    # CTA pair), small K
    (5000, 24, 0.37),
    (16384, 12, 1.0),
    (40000, 7, 2.0 ** -100),
    (40, 9, 2.0 ** 90),
    (512, 40, 3.5e-3),
]


@pytest.mark.parametrize("K,N,t", RANDOM_W_CASES, ids=[f"K{c[0]}" for c in RANDOM_W_CASES])
def test_prepare_weight_on_random_nvfp4_bytes(K, N, t):
    packed, scales = random_nvfp4(N, K, seed=K + N)
    t = np.float32(t)
    Kp = oracle.padded_k(K)
    rq, rs = oracle.prepare_weight(packed, scales, t, K)
    for fmt in ("f16", "s8"):
        q, s = gpu_prepare_weight(packed, scales, t, K, fmt=fmt)
        assert_codes_match(codes_to_np(q, Kp), rq)
        assert_scales_match(s.cpu().numpy(), rs)
    # rows 2 (zero scales in every block) and 5 (every element -0) are degenerate
    assert rs[2] == 0 and np.all(rq[2] == 0)
    if N > 5:
        assert rs[5] == 0 and np.all(rq[5] == 0)


def test_prepare_weight_exhaustive_nibble_scale_pairs():
    # every (E4M3 scale byte, E2M1 code) pair appears: row r uses the r-th
    # non-NaN scale byte for all its blocks and walks the 16 nibbles in every
    # block.  A single scale per row keeps the FP32 rotation exact, so the
    # codes must equal the oracle's bit for bit.
    scale_bytes = np.array([b for b in range(256) if b not in E4M3_NAN], dtype=np.uint8)
    N, K = len(scale_bytes), 256
    nib = np.tile(np.arange(16, dtype=np.uint8), K // 16)[None, :].repeat(N, axis=0)
    packed = nib[:, 0::2] | (nib[:, 1::2] << 4)
    scales = np.repeat(scale_bytes[:, None], K // 16, axis=1)
    t = np.float32(1.0)
    rq, rs = oracle.prepare_weight(packed, scales, t, K)
    q, s = gpu_prepare_weight(packed, scales, t, K)
    assert np.array_equal(codes_to_np(q, K), rq)
    assert_scales_match(s.cpu().numpy(), rs)


GATES = {
    "tail_-87.5": -87.5,     # 1 + exp(-g) lies between 2^126 and 2^128
    "tail_-80": -80.0,
    "tail_-90": -90.0,       # exp(-g) overflows FP32
    "tail_-200": -200.0,
    "head_+90": 90.0,        # exp(-g) underflows
    "pm_1e4": None,          # +-1e4, random signs
}


def swiglu_rows(dtype, seed):
    """Rows of [gate | value] that drive the gates into both tails.

    Row kinds: every gate at one extreme value; gates +-1e4; a mix of all the
    extremes with N(0, 1) gates; gates N(0, 1) * 40 (spanning +-120); values
    scaled by 1e30 or 1e-30 under ordinary gates.  Every hidden value stays
    finite (|h| < 1e36).
    """
    rng = np.random.default_rng(seed)
    K = 1000
    rows = []
    for name, g in GATES.items():
        gate = (np.full(K, g, np.float32) if g is not None
                else np.where(rng.random(K) < 0.5, -1e4, 1e4).astype(np.float32))
        rows.append((gate, rng.standard_normal(K).astype(np.float32)))
    mix = rng.standard_normal(K).astype(np.float32)
    pick = rng.random(K)
    ext = np.array([-87.5, -80, -90, -200, 90, 1e4, -1e4], np.float32)
    mix[pick < 0.5] = ext[rng.integers(0, len(ext), int((pick < 0.5).sum()))]
    rows.append((mix, rng.standard_normal(K).astype(np.float32)))
    rows.append(((rng.standard_normal(K) * 40).astype(np.float32), rng.standard_normal(K).astype(np.float32)))
    rows.append((rng.standard_normal(K).astype(np.float32), (rng.standard_normal(K) * 1e30).astype(np.float32)))
    rows.append((rng.standard_normal(K).astype(np.float32), (rng.standard_normal(K) * 1e-30).astype(np.float32)))
    x = np.stack([np.concatenate([g, v]) for g, v in rows]).astype(np.float32)
    if dtype == "fp32":
        return x, K
    if dtype == "bf16":
        return synth.bf16_bits_from_f32(x), K
    raise ValueError(dtype)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_swiglu_extreme_gates_match_oracle(dtype):
    x, K = swiglu_rows(dtype, seed=61)
    Kp = oracle.padded_k(K)
    with np.errstate(over="ignore"):
        rq, rs = oracle.quant_act(x, dtype, K, True)
    # the -87.5 and -80 rows are tiny but not degenerate: their codes carry the row
    assert rs[0] > 0 and rs[1] > 0 and np.abs(rq[0]).max() == 127
    for fmt in ("f16", "s8"):
        q, s = gpu_quant_act(x, dtype, K, swiglu=True, fmt=fmt)
        assert_codes_match(codes_to_np(q, Kp), rq)
        assert_scales_match(s.cpu().numpy(), rs)
