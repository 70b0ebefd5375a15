"""Pins of the CPU oracle against facts fixed outside the oracle itself.

Each test targets one step of the layer so that a plausible slip in the
oracle (a dropped term, a wrong sign or index, a transposed operand, a wrong
rounding mode) fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from conftest import read_golden

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ---------------------------------------------------------------- NVFP4 decode
def test_e2m1_all_codes_match_ocp_table():
    rows = read_golden("e2m1_ocp_mx.txt")
    assert len(rows) == 16
    for code, val in rows:
        got = oracle.e2m1_value(int(code))
        assert got == float(val)
        assert math.copysign(1.0, got) == math.copysign(1.0, float(val))


def test_e4m3_golden_values():
    for code, val in read_golden("e4m3_ocp_ofp8.txt"):
        got = oracle.e4m3_value(int(code, 16))
        if val == "nan":
            assert math.isnan(got)
        else:
            assert got == float(val)


def test_e4m3_all_codes_match_torch_cast():
    codes = torch.arange(256, dtype=torch.uint8)
    lib = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = np.array([oracle.e4m3_value(c) for c in range(256)])
    nan = np.isnan(lib)
    assert np.array_equal(nan, np.isnan(ours))
    assert np.array_equal(lib[~nan], ours[~nan])


def test_decode_nibble_order_and_block_scale_indexing():
    # one row, K = 32 (two scale blocks).  byte 0 = 0x21 -> element 0 is code 1
    # (0.5) and element 1 is code 2 (1.0); byte 8 = 0xF7 -> element 16 is code 7
    # (6.0), element 17 is code 15 (-6.0).  Block 0 scale 0x38 = 1.0, block 1
    # scale 0x40 = 2.0, tensor scale 0.25.
    packed = np.zeros((1, 16), np.uint8)
    packed[0, 0] = 0x21
    packed[0, 8] = 0xF7
    scales = np.array([[0x38, 0x40]], np.uint8)
    w = oracle.decode_nvfp4(packed, scales, np.float32(0.25), 32)
    expect = np.zeros((1, 32))
    expect[0, 0] = 0.5 * 1.0 * 0.25
    expect[0, 1] = 1.0 * 1.0 * 0.25
    expect[0, 16] = 6.0 * 2.0 * 0.25
    expect[0, 17] = -6.0 * 2.0 * 0.25
    assert np.array_equal(w, expect)


def test_decode_ignores_serialised_padding():
    wl = synth.Workload("pad", 8, 40, 24, "bf16", "bf16", False, 0.0, 1.0, 7)
    packed, scales, t = synth.make_nvfp4_weight(wl)
    assert packed.shape == (24, 24)          # K_s = 48
    dirty = packed.copy()
    # elements 40..47 live in bytes 20..23: fill both nibbles with code 7 (6.0)
    dirty[:, 20:24] = 0x77
    a = oracle.decode_nvfp4(packed, scales, t, 40)
    b = oracle.decode_nvfp4(dirty, scales, t, 40)
    assert a.shape == (24, 40) and np.array_equal(a, b)
    qa, sa = oracle.prepare_weight(packed, scales, t, 40)
    qb, sb = oracle.prepare_weight(dirty, scales, t, 40)
    assert np.array_equal(qa, qb) and np.array_equal(sa, sb)


# ---------------------------------------------------------------- rotation
def test_rotation_is_orthogonal_with_pm_one_over_16_entries():
    R = oracle.rotation_matrix()
    assert R.shape == (256, 256)
    assert np.max(np.abs(R @ R.T - np.eye(256))) < 1e-15
    assert np.all(np.abs(np.abs(R) - 1.0 / 16) == 0)


def test_rotation_closed_form_sylvester_entries():
    # Sylvester ordering: H[i, j] = (-1) ** popcount(i & j)
    R = oracle.rotation_matrix()
    i = np.arange(256)[:, None]
    j = np.arange(256)[None, :]
    pop = np.vectorize(lambda v: bin(int(v)).count("1"))(i & j)
    assert np.array_equal(R * 16, np.where(pop % 2 == 0, 1.0, -1.0))


def test_rotation_unit_vector_gives_row_and_spike_spreads():
    R = oracle.rotation_matrix()
    for i in (0, 1, 37, 255):
        e = np.zeros((1, 256))
        e[0, i] = 1.0
        assert np.array_equal(oracle.rotate_blocks(e), R[i:i + 1])
    # an outlier of size v in one channel becomes |v|/16 on every channel
    x = np.zeros((1, 512))
    x[0, 300] = -32.0
    y = oracle.rotate_blocks(x)
    assert np.all(y[0, :256] == 0) and np.all(np.abs(y[0, 256:]) == 2.0)


def test_rotation_preserves_norm_and_blocks_are_independent():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((3, 768))
    y = oracle.rotate_blocks(x)
    assert np.allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-14)
    x2 = x.copy()
    x2[:, 256:512] = 0
    y2 = oracle.rotate_blocks(x2)
    assert np.array_equal(y2[:, :256], y[:, :256])
    assert np.array_equal(y2[:, 512:], y[:, 512:])
    assert np.all(y2[:, 256:512] == 0)


@pytest.mark.parametrize("K", [256, 512, 5000, 5376])
def test_paired_rotation_invariance(K):
    rng = np.random.default_rng(K)
    x = rng.standard_normal((5, K))
    w = rng.standard_normal((7, K))
    xr = oracle.rotate_blocks(x)
    wr = oracle.rotate_blocks(w)
    assert xr.shape[1] == oracle.padded_k(K) and xr.shape[1] % 256 == 0
    ref = x @ w.T
    assert np.max(np.abs(xr @ wr.T - ref)) <= 1e-12 * np.max(np.abs(ref)) * math.sqrt(K)


def test_padded_k():
    assert oracle.padded_k(5376) == 5376
    assert oracle.padded_k(5000) == 5120
    assert oracle.padded_k(1) == 256
    assert oracle.padded_k(20480) == 20480


# ---------------------------------------------------------------- SwiGLU
def test_swiglu_closed_forms_and_half_order():
    K = 4
    g = np.array([0.0, math.log(3.0), 40.0, -40.0])
    v = np.array([5.0, 2.0, 1.0, 1.0])
    h = oracle.swiglu(np.concatenate([g, v])[None, :], K)[0]
    assert h[0] == 0.0
    assert abs(h[1] - 0.75 * math.log(3.0) * 2.0) < 1e-15      # sigmoid(ln 3) = 3/4
    assert abs(h[2] - 40.0) < 1e-12                             # swish(g) -> g
    assert abs(h[3]) < 1e-15                                    # swish(g) -> 0
    swapped = oracle.swiglu(np.concatenate([v, g])[None, :], K)[0]
    assert not np.allclose(swapped, h)


# ---------------------------------------------------------------- quantiser
def test_quant_zero_row_and_single_spike():
    x = np.zeros((2, 256))
    x[1, 10] = -3.5
    q, s = oracle.quantize_rows(x)
    assert s[0] == 0 and np.all(q[0] == 0)
    assert q[1, 10] == -127 and np.count_nonzero(q[1]) == 1
    assert s[1] == np.float32(3.5) / np.float32(127)


def test_quant_ties_go_to_even_and_use_reciprocal():
    # max 254 -> s = 2, r = 0.5 exactly: 1 -> 0.5 -> 0, 3 -> 1.5 -> 2, 5 -> 2.5 -> 2
    x = np.zeros((1, 256))
    x[0, :5] = [254.0, 1.0, 3.0, 5.0, -7.0]
    q, s = oracle.quantize_rows(x)
    assert s[0] == 2.0
    assert list(q[0, :5]) == [127, 0, 2, 2, -4]


def test_quant_constant_row_and_negative_max():
    q, s = oracle.quantize_rows(np.full((1, 256), -0.3))
    assert np.all(q == -127) and s[0] == np.float32(np.float32(0.3) / np.float32(127))


def test_quant_degenerate_tiny_row():
    x = np.zeros((1, 256))
    x[0, 0] = 1e-44          # FP32 subnormal: its reciprocal scale overflows
    q, s = oracle.quantize_rows(x)
    assert s[0] == 0 and np.all(q == 0)


def test_quant_codes_bound_the_rounding_error():
    rng = np.random.default_rng(11)
    x = rng.standard_normal((20, 512)) * rng.uniform(0.01, 100, (20, 1))
    q, s = oracle.quantize_rows(x)
    assert q.dtype == np.int8 and np.max(np.abs(q)) == 127
    err = np.abs(q * s[:, None].astype(np.float64) - x.astype(np.float32))
    assert np.all(err <= 0.5 * s[:, None] * (1 + 1e-5))


# ---------------------------------------------------------------- integer GEMM
def _brute(qa, qw):
    M, K = qa.shape
    N = qw.shape[0]
    out = [[0] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            acc = 0
            for k in range(K):
                acc += int(qa[m, k]) * int(qw[n, k])
            out[m][n] = acc
    return np.array(out, dtype=np.int64)


@pytest.mark.parametrize("M,N,K", [(3, 5, 256), (7, 4, 512), (1, 33, 256)])
def test_int_gemm_matches_brute_force(M, N, K):
    rng = np.random.default_rng(M * 100 + N)
    qa = rng.integers(-127, 128, (M, K)).astype(np.int8)
    qw = rng.integers(-127, 128, (N, K)).astype(np.int8)
    qa[0, :] = 127
    qw[0, :] = -127
    assert np.array_equal(oracle.int_gemm(qa, qw), _brute(qa, qw))


def test_int_gemm_extremes_and_orientation():
    K = 512
    qa = np.full((2, K), -127, np.int8)
    qw = np.full((3, K), 127, np.int8)
    acc = oracle.int_gemm(qa, qw)
    assert acc.shape == (2, 3) and np.all(acc == -127 * 127 * K)
    # non-square operands catch a transposed product
    qa = np.zeros((2, 256), np.int8)
    qw = np.zeros((5, 256), np.int8)
    qa[1, 3] = 2
    qw[4, 3] = -3
    acc = oracle.int_gemm(qa, qw)
    assert acc[1, 4] == -6 and np.count_nonzero(acc) == 1


# ---------------------------------------------------------------- output rounding
def test_bf16_rounding_single_step_ties_to_even():
    one = 1.0
    vals = np.array([one + 2 ** -8, one + 3 * 2 ** -8, one + 2 ** -8 + 2 ** -40,
                     -(one + 2 ** -8 + 2 ** -40), 2.0 ** -133, 3 * 2.0 ** -134, 1e39])
    got = oracle.round_to_dtype(vals, "bf16")
    assert got[0] == 1.0                       # tie -> even
    assert got[1] == one + 2 ** -6             # tie -> even (upwards)
    assert got[2] == one + 2 ** -7             # just above the tie: no double rounding
    assert got[3] == -(one + 2 ** -7)
    assert got[4] == 2.0 ** -133               # smallest subnormal
    assert got[5] == 2.0 ** -132               # subnormal tie -> even
    assert np.isinf(got[6])


def test_bf16_rounding_matches_torch_on_fp32_values():
    rng = np.random.default_rng(3)
    v = (rng.standard_normal(20000) * np.exp(rng.uniform(-30, 30, 20000))).astype(np.float32)
    lib = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(oracle.round_to_dtype(v.astype(np.float64), "bf16"), lib)


def test_fp16_rounding_matches_numpy_cast():
    rng = np.random.default_rng(4)
    v = rng.standard_normal(20000) * np.exp(rng.uniform(-20, 12, 20000))
    lib = v.astype(np.float16).astype(np.float64)
    assert np.array_equal(oracle.round_to_dtype(v, "fp16"), lib)


# ---------------------------------------------------------------- whole layer
def _rel_l2(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def _layer_error(wl, rows, cols):
    x = synth.make_activations(wl, rows=rows)
    packed, scales, t = synth.make_nvfp4_weight(wl, rows=cols)
    y, _ = oracle.convrot_linear(x, wl.x_dtype, packed, scales, t, wl.K, "fp32", wl.swiglu)
    xf = oracle.storage_to_f64(x, wl.x_dtype)
    h = oracle.swiglu(xf, wl.K) if wl.swiglu else xf
    ref = h @ oracle.decode_nvfp4(packed, scales, t, wl.K).T
    return y, ref, x, (packed, scales, t)


@pytest.mark.parametrize("name,page_key", [("qkv", "rel_l2_qkv"), ("ffn_down", "rel_l2_ffn_down")])
def test_added_error_matches_the_pages(name, page_key):
    page = dict((k, float(v)) for k, v in read_golden("pages_numbers.txt"))[page_key]
    wl = synth.WORKLOADS[name]
    y, ref, _, _ = _layer_error(wl, rows=48, cols=96)
    err = _rel_l2(y, ref)
    # the pages measured real weights on an A40; accept the same order of magnitude
    assert 0.5 * page <= err <= 1.6 * page, err


def test_rotation_lowers_the_error_and_must_be_paired():
    wl = synth.WORKLOADS["qkv"]
    x = synth.make_activations(wl, rows=48)
    packed, scales, t = synth.make_nvfp4_weight(wl, rows=96)
    xf = oracle.storage_to_f64(x, wl.x_dtype)
    w = oracle.decode_nvfp4(packed, scales, t, wl.K)
    ref = xf @ w.T
    I = np.eye(256)

    def run(Ra, Rw):
        qa, sa = oracle.quantize_rows(oracle.rotate_blocks(xf, Ra))
        qw, sw = oracle.quantize_rows(oracle.rotate_blocks(w, Rw))
        return oracle.dequantize(oracle.int_gemm(qa, qw), sa, sw, "fp32")

    rotated = _rel_l2(run(None, None), ref)
    plain = _rel_l2(run(I, I), ref)
    one_sided = _rel_l2(run(None, I), ref)
    assert rotated < 0.6 * plain
    assert one_sided > 0.5


def test_dequant_scales_are_per_row_and_per_column():
    acc = np.array([[10, -20, 30]], dtype=np.int64)
    y = oracle.dequantize(np.vstack([acc, 2 * acc]), np.array([0.5, 0.25], np.float32),
                          np.array([1.0, 2.0, 4.0], np.float32), "fp32")
    assert np.array_equal(y, np.array([[5.0, -20.0, 60.0], [5.0, -20.0, 60.0]]))


def test_synth_shapes_follow_the_pages():
    g = dict((k, float(v)) for k, v in read_golden("pages_numbers.txt"))
    W = synth.WORKLOADS
    assert W["qkv"].K == g["hidden"] and W["qkv"].N == g["qkv_out"]
    assert W["ffn_down"].K == g["ffn_hidden"] and W["ffn_down"].k_in == g["fc1_out"]
    assert W["ffn_up"].N == g["fc1_out"]


# ---------------------------------------------------------------- pre-scales and bias
def test_pre_scale_folds_into_the_weights():
    # (x * p) W'^T with W' = W / p equals x W^T: the pre-scale acts on the
    # layer input before the rotation, and the rotation stays paired
    rng = np.random.default_rng(41)
    K = 512
    x = rng.standard_normal((6, K))
    w = rng.standard_normal((5, K))
    p = np.exp(rng.uniform(-2, 2, K))
    xs = x * p
    ws = w / p
    lhs = oracle.rotate_blocks(xs) @ oracle.rotate_blocks(ws).T
    assert np.allclose(lhs, x @ w.T, rtol=1e-10, atol=1e-10)


def test_pre_scale_applies_after_swiglu_and_before_rotation():
    K = 256
    x2 = np.zeros((1, 2 * K), np.float32)
    x2[0, 3] = 1.0            # gate 1 at channel 3
    x2[0, K + 3] = 2.0        # value 2 at channel 3
    p = np.ones(K, np.float32)
    p[3] = 4.0
    bits = synth.bf16_bits_from_f32(x2)
    q, s = oracle.quant_act(bits, "bf16", K, True, p)
    h3 = 1.0 / (1.0 + math.exp(-1.0)) * 2.0 * 4.0     # swish(1) * 2, then * 4
    # a single nonzero channel rotates to +-h3/16 everywhere: codes +-127
    assert np.all(np.abs(q) == 127)
    assert abs(float(s[0]) - np.float32(np.float32(h3 / 16) / np.float32(127))) <= 2e-7 * h3


def test_bias_adds_per_output_channel():
    acc = np.zeros((2, 3), np.int64)
    b = np.array([0.5, -1.0, 2.0], np.float32)
    y = oracle.dequantize(acc, np.ones(2, np.float32), np.ones(3, np.float32), "fp32", b)
    assert np.array_equal(y, np.array([[0.5, -1.0, 2.0], [0.5, -1.0, 2.0]]))
