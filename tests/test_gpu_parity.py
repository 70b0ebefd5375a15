"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Bars: identical S8 operands give bit-exact int32 accumulators; S8 codes agree
on >= 99.99% of entries with |diff| <= 1 (FP32 rotation order vs the oracle's
FP64 rotation rounded to FP32); scales agree to 1e-6 relative; outputs are
within relative L2 1e-3 of the oracle and within 2 BF16 ulp of the row max
per element.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import (DEV, assert_codes_match, assert_output_match, assert_scales_match,
                      codes_to_np, ensure_built, f16_codes_from_np, gpu_gemm, gpu_prepare_weight,
                      gpu_quant_act, storage_to_dev)

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    import rotated_w4a8_int8_gb300 as cr
    yield
    assert cr.device_error() == 0


def small(name, M, N):
    wl = synth.WORKLOADS[name]
    return synth.Workload(f"{name}_small", M, wl.K, N, wl.x_dtype, wl.out_dtype, wl.swiglu,
                          wl.outlier_frac, wl.outlier_mult, wl.seed)


# ---------------------------------------------------------------- kernel 2
ACT_CASES = [
    ("tiny", synth.WORKLOADS["tiny"]),
    ("qkv_rows", small("qkv", 200, 8)),
    ("ffn_down_rows", small("ffn_down", 64, 8)),
    ("ffn_up_rows", small("ffn_up", 96, 8)),
    ("ragged_rows", small("ragged", 77, 8)),
    ("wide_rows", small("wide_k", 40, 8)),
    ("fp32_in", synth.Workload("fp32_in", 33, 1000, 8, "fp32", "fp32", False, 0.01, 20.0, 9)),
    ("swiglu_fp16", synth.Workload("sw16", 50, 768, 8, "fp16", "bf16", True, 0.0, 1.0, 10)),
    ("swiglu_fp32_ragged", synth.Workload("sw32", 21, 300, 8, "fp32", "bf16", True, 0.0, 1.0, 11)),
    ("k16", synth.Workload("k16", 17, 16, 8, "bf16", "bf16", False, 0.0, 1.0, 12)),
    ("k1", synth.Workload("k1", 5, 1, 8, "bf16", "bf16", False, 0.0, 1.0, 13)),
    ("max_kp", synth.Workload("maxkp", 3, 65536, 8, "bf16", "bf16", False, 0.01, 20.0, 17)),
    ("max_kp_swiglu", synth.Workload("maxkps", 2, 65536, 8, "bf16", "bf16", True, 0.0, 1.0, 18)),
    # rows split over a CTA pair with one block per slot (16384 < K_p <= 32768), SwiGLU and FP16 inputs
    ("split_swiglu", synth.Workload("spsw", 6, 20480, 8, "bf16", "bf16", True, 0.0, 1.0, 26)),
    ("split_fp16_ragged", synth.Workload("spf16", 5, 17000, 8, "fp16", "fp32", False, 0.01, 20.0, 27)),
]


@pytest.mark.parametrize("case,wl", ACT_CASES, ids=[c[0] for c in ACT_CASES])
def test_quant_act_matches_oracle(case, wl):
    x = synth.make_activations(wl)
    Kp = oracle.padded_k(wl.K)
    q, s = gpu_quant_act(x, wl.x_dtype, wl.K, wl.swiglu, fmt="f16")
    q8, s8 = gpu_quant_act(x, wl.x_dtype, wl.K, wl.swiglu, fmt="s8")
    rq, rs = oracle.quant_act(x, wl.x_dtype, wl.K, wl.swiglu)
    got = codes_to_np(q, Kp)
    assert np.array_equal(got, codes_to_np(q8, Kp))
    assert torch.equal(s, s8)
    assert_codes_match(got, rq)
    assert_scales_match(s.cpu().numpy(), rs)


def test_quant_act_unaligned_pitch_and_wide_ld():
    # bf16 pitch of K+1 elements: rows are not 16-byte aligned -> scalar path
    wl = synth.Workload("pitch", 40, 700, 8, "bf16", "bf16", False, 0.02, 20.0, 14)
    x = synth.make_activations(wl)
    wide = np.zeros((wl.M, wl.K + 1), np.uint16)
    wide[:, :wl.K] = x
    wide[:, wl.K] = 0x7F80          # +inf in the column past K: must be ignored
    xd = storage_to_dev(wide, "bf16")
    Kp = oracle.padded_k(wl.K)
    q, s = gpu_quant_act(None, "bf16", wl.K, xdev=xd, ld=Kp + 64)
    rq, rs = oracle.quant_act(x, "bf16", wl.K)
    assert_codes_match(codes_to_np(q, Kp), rq)
    assert_scales_match(s.cpu().numpy(), rs)


def test_quant_act_degenerate_rows():
    wl = synth.Workload("deg", 6, 512, 8, "bf16", "bf16", False, 0.0, 1.0, 15)
    x = synth.make_activations(wl)
    x[1] = 0                        # all-zero row
    x[3] = 0
    x[3, 7] = 0x0001                # one bf16 subnormal: reciprocal scale overflows
    q, s = gpu_quant_act(x, "bf16", wl.K)
    rq, rs = oracle.quant_act(x, "bf16", wl.K)
    got = codes_to_np(q, 512)
    assert np.all(got[1] == 0) and np.all(got[3] == 0)
    sc = s.cpu().numpy()
    assert sc[1] == 0 and sc[3] == 0
    assert_codes_match(got, rq)
    assert_scales_match(sc, rs)


def _fp32_tie_rows(rows, nblocks, seed):
    """FP32 rows whose quantiser products land exactly on k + 1/2.

    Block 0 of each row holds one value 16 A, so its rotated entries are all A
    (the row maximum).  Every other block holds one value 16 v at a random
    position; rotated, it becomes +-v on all 256 entries.  v is chosen so that
    the FP32 product v * r (r the FP32 reciprocal of the FP32 scale) rounds to
    exactly k + 1/2 while the exact product lies on the side of the odd
    neighbour: rounding the FP32 product half to even gives the even code, and
    rounding the exact product (a fused multiply-add style shortcut) gives the
    odd one.  Returns the rows and the (row, block) list of the ties.
    """
    rng = np.random.default_rng(seed)
    x = np.zeros((rows, nblocks * 256), np.float32)
    ties = []
    for m in range(rows):
        A = np.float32(rng.uniform(1.0, 100.0))
        x[m, 0] = np.float32(16) * A
        s = np.float32(A / np.float32(127))
        r = np.float32(np.float32(1) / s)
        for b in range(1, nblocks):
            for _ in range(64):
                k = int(rng.integers(0, 126))
                t = k + 0.5
                v = np.float32(t / float(r))
                for _ in range(64):
                    exact = float(v) * float(r)          # exact in float64
                    if np.float32(v * r) == np.float32(t) and (exact > t) == (k % 2 == 0) and exact != t:
                        break
                    v = np.nextafter(v, np.float32(np.inf) if exact < t else np.float32(0))
                else:
                    continue
                break
            else:
                raise AssertionError("no tie found")
            x[m, b * 256 + int(rng.integers(0, 256))] = np.float32(16) * v
            ties.append((m, b))
    return x, ties


def test_quant_codes_round_the_fp32_product_half_to_even():
    x, ties = _fp32_tie_rows(48, 12, seed=21)
    K = x.shape[1]
    rq, rs = oracle.quant_act(x, "fp32", K)
    # the construction bites: every tie block holds even codes that the exact
    # product would have rounded the other way
    for m, b in ties[:50]:
        blk = rq[m, b * 256:(b + 1) * 256].astype(np.int64)
        assert np.all(blk % 2 == 0) and np.all(np.abs(blk) == abs(blk[0]))
    for fmt in ("f16", "s8"):
        q, s = gpu_quant_act(x, "fp32", K, fmt=fmt)
        assert np.array_equal(codes_to_np(q, K), rq), fmt
        assert np.array_equal(s.cpu().numpy(), rs), fmt


def test_swiglu_quant_codes_round_the_fp32_product_half_to_even():
    # the SwiGLU kernel rounds through FP32 adds, the others through cvt.rni:
    # the same tie rows, fed through the SwiGLU prologue.  A gate of 128 makes
    # exp(-g) underflow to 0 in FP32 and FP64 alike, so h = 128 v exactly and
    # the value half carries the tie rows divided by 128 (a power of two).
    ties, _ = _fp32_tie_rows(32, 12, seed=24)
    K = ties.shape[1]
    x = np.concatenate([np.full_like(ties, 128.0), ties / np.float32(128.0)], axis=1).astype(np.float32)
    rq, rs = oracle.quant_act(x, "fp32", K, True)
    rq0, rs0 = oracle.quant_act(ties, "fp32", K)
    assert np.array_equal(rq, rq0) and np.array_equal(rs, rs0)
    for fmt in ("f16", "s8"):
        q, s = gpu_quant_act(x, "fp32", K, swiglu=True, fmt=fmt)
        assert np.array_equal(codes_to_np(q, K), rq), fmt
        assert np.array_equal(s.cpu().numpy(), rs), fmt


# ---------------------------------------------------------------- kernel 1
W_CASES = [
    ("tiny", synth.WORKLOADS["tiny"]),
    ("qkv_rows", small("qkv", 8, 300)),
    ("ffn_down_rows", small("ffn_down", 8, 130)),
    ("ragged_rows", small("ragged", 8, 257)),
    ("wide_rows", small("wide_k", 8, 64)),
    ("k40", synth.Workload("k40", 8, 40, 24, "bf16", "bf16", False, 0.0, 1.0, 16)),
    ("max_kp", synth.Workload("maxkpw", 8, 65536, 5, "bf16", "bf16", False, 0.0, 1.0, 19)),
]


@pytest.mark.parametrize("case,wl", W_CASES, ids=[c[0] for c in W_CASES])
def test_prepare_weight_matches_oracle(case, wl):
    packed, scales, t = synth.make_nvfp4_weight(wl)
    Kp = oracle.padded_k(wl.K)
    q, s = gpu_prepare_weight(packed, scales, t, wl.K, fmt="f16")
    q8, s8 = gpu_prepare_weight(packed, scales, t, wl.K, fmt="s8")
    rq, rs = oracle.prepare_weight(packed, scales, t, wl.K)
    got = codes_to_np(q, Kp)
    assert np.array_equal(got, codes_to_np(q8, Kp))
    assert_codes_match(got, rq)
    assert_scales_match(s.cpu().numpy(), rs)


def test_prepare_weight_ignores_serialised_padding():
    wl = small("ragged", 8, 100)          # K = 5000, K_s = 5008
    packed, scales, t = synth.make_nvfp4_weight(wl)
    dirty = packed.copy()
    dirty[:, 2500:] = 0x77                # elements 5000..5007 -> code 7 (6.0)
    qa, sa = gpu_prepare_weight(packed, scales, t, wl.K)
    qb, sb = gpu_prepare_weight(dirty, scales, t, wl.K)
    assert torch.equal(qa, qb) and torch.equal(sa, sb)


GUARD_CASES = [("qkv_rows", small("qkv", 40, 24)), ("wide_rows", small("wide_k", 12, 8)),
               ("ragged_rows", small("ragged", 21, 9)),
               ("max_kp", synth.Workload("maxkpg", 3, 65536, 3, "bf16", "bf16", False, 0.01, 20.0, 23))]


@pytest.mark.parametrize("case,wl", GUARD_CASES, ids=[c[0] for c in GUARD_CASES])
@pytest.mark.parametrize("fmt", ["f16", "s8"])
def test_quant_kernels_write_nothing_outside_their_outputs(case, wl, fmt):
    # codes and scales sit inside poisoned buffers: extra columns past K_p (a
    # wider pitch), a row after the last and a scale after the last must keep
    # the poison; inside, the results equal those of the plain layout
    import rotated_w4a8_int8_gb300 as cr
    Kp = oracle.padded_k(wl.K)
    dt = torch.float16 if fmt == "f16" else torch.int8
    poison = 77
    x = synth.make_activations(wl)
    packed, scales, t = synth.make_nvfp4_weight(wl)
    for rows, run, ref in (
            (wl.M, lambda q, s: cr.quant_act(storage_to_dev(x, wl.x_dtype), wl.K, q, s),
             lambda: gpu_quant_act(x, wl.x_dtype, wl.K, fmt=fmt)),
            (wl.N, lambda q, s: cr.prepare_weight(torch.from_numpy(packed).to(DEV), torch.from_numpy(scales).to(DEV),
                                                  torch.tensor([float(t)], dtype=torch.float32, device=DEV),
                                                  wl.K, q, s),
             lambda: gpu_prepare_weight(packed, scales, t, wl.K, fmt=fmt))):
        big = torch.full((rows + 1, Kp + 64), poison, dtype=dt, device=DEV)
        sbig = torch.full((rows + 1,), float(poison), dtype=torch.float32, device=DEV)
        run(big[:rows], sbig[:rows])
        torch.cuda.synchronize()
        b = big.to(torch.int32).cpu().numpy()
        assert np.all(b[:, Kp:] == poison) and np.all(b[rows] == poison)
        assert float(sbig[rows]) == float(poison)
        q, s = ref()
        assert np.array_equal(b[:rows, :Kp], codes_to_np(q, Kp))
        assert torch.equal(sbig[:rows], s)


# ---------------------------------------------------------------- kernel 3
GEMM_SHAPES = [(128, 256, 256), (300, 520, 1280), (1, 1, 256), (129, 257, 768), (513, 300, 5376),
               (64, 1000, 512), (130, 260, 65536), (2100, 1300, 512)]


@pytest.mark.parametrize("M,N,Kp", GEMM_SHAPES)
def test_gemm_int32_bit_exact(M, N, Kp):
    import rotated_w4a8_int8_gb300 as cr
    rng = np.random.default_rng(M * 7 + N)
    qa = rng.integers(-127, 128, (M, Kp)).astype(np.int8)
    qw = rng.integers(-127, 128, (N, Kp)).astype(np.int8)
    acc = torch.full((M, N), 12345, dtype=torch.int32, device=DEV)
    cr.gemm_i32(f16_codes_from_np(qa), f16_codes_from_np(qw), acc)
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), oracle.int_gemm(qa, qw))


@pytest.mark.parametrize("pattern", ["all_max", "alternating", "max_minus", "odd_groups"])
def test_gemm_int32_exact_at_extremes(pattern):
    # partial sums reach 127^2 * 1024 inside a chunk and 127^2 * 20480 in total;
    # "odd_groups" makes every 16-term group sum odd (15 * 127^2 + 127 * 126),
    # so the running sums inside a chunk are odd and pass 2^23: an FP32
    # accumulation that dropped a low bit above 2^23 would show
    import rotated_w4a8_int8_gb300 as cr
    M, N, Kp = 130, 260, 20480
    qa = np.full((M, Kp), 127, np.int8)
    qw = np.full((N, Kp), 127, np.int8)
    if pattern == "alternating":
        qw[:, 1::2] = -127
        qa[::2, :] = -127
    elif pattern == "max_minus":
        qw[:] = -127
        qa[:, -1] = 126
    elif pattern == "odd_groups":
        qw[:, 15::16] = 126
        qa[1::2, :] = -127
    acc = torch.zeros((M, N), dtype=torch.int32, device=DEV)
    cr.gemm_i32(f16_codes_from_np(qa), f16_codes_from_np(qw), acc)
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), oracle.int_gemm(qa, qw))


@pytest.mark.parametrize("out_dtype", ["bf16", "fp16", "fp32"])
def test_gemm_dequant_given_identical_operands(out_dtype):
    rng = np.random.default_rng(21)
    M, N, Kp = 257, 384, 1024
    qa = rng.integers(-127, 128, (M, Kp)).astype(np.int8)
    qw = rng.integers(-127, 128, (N, Kp)).astype(np.int8)
    sa = (rng.uniform(0.5, 2.0, M) * 1e-3).astype(np.float32)
    sw = (rng.uniform(0.5, 2.0, N) * 1e-4).astype(np.float32)
    sa[5] = 0
    y = gpu_gemm(f16_codes_from_np(qa), torch.from_numpy(sa).to(DEV), f16_codes_from_np(qw),
                 torch.from_numpy(sw).to(DEV), out_dtype, Kp)
    ref = oracle.dequantize(oracle.int_gemm(qa, qw), sa, sw, out_dtype)
    got = y.float().cpu().numpy().astype(np.float64)
    assert np.all(got[5] == 0)
    assert_output_match(got, ref)
    # one rounding of an FP32 product chain: at most one unit in the last place
    ulp = {"bf16": 2.0 ** -7, "fp16": 2.0 ** -10, "fp32": 2.0 ** -23}[out_dtype]
    mag = np.maximum(np.abs(ref), 1e-30)
    assert np.all(np.abs(got - ref) <= ulp * 2.0 ** np.floor(np.log2(mag)) * 1.0001)


@pytest.mark.parametrize("out_dtype", ["bf16", "fp16", "fp32"])
def test_gemm_output_pitch_guard_and_unaligned_base(out_dtype):
    # an output view whose base and pitch are not 16-byte aligned takes the
    # per-element store path of the epilogue; nothing around it may change
    rng = np.random.default_rng(22)
    M, N, Kp = 140, 270, 512
    qa = rng.integers(-127, 128, (M, Kp)).astype(np.int8)
    qw = rng.integers(-127, 128, (N, Kp)).astype(np.int8)
    sa = np.full(M, 1e-3, np.float32)
    sw = np.full(N, 1e-3, np.float32)
    import rotated_w4a8_int8_gb300 as cr
    tdt = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}[out_dtype]
    big = torch.full((M + 1, N + 9), -7.0, dtype=tdt, device=DEV)
    view = big[:M, 1:N + 1]               # base one element past a 16-byte boundary
    cr.gemm(f16_codes_from_np(qa), torch.from_numpy(sa).to(DEV), f16_codes_from_np(qw),
            torch.from_numpy(sw).to(DEV), view, K_p=Kp)
    b = big.float().cpu().numpy()
    assert np.all(b[:, 0] == -7) and np.all(b[:, N + 1:] == -7) and np.all(b[M] == -7)
    ref = oracle.dequantize(oracle.int_gemm(qa, qw), sa, sw, out_dtype)
    assert_output_match(b[:M, 1:N + 1], ref)


def test_empty_calls_launch_nothing():
    import rotated_w4a8_int8_gb300 as cr
    lib = cr.load_library()
    y = torch.full((4, 4), 3.0, device=DEV)
    assert lib.convrot_gemm(16, 512, 16, None, 16, 512, 16, None, None, 0, 4, 512, y.data_ptr(), 2, 4, 0) == 0
    assert lib.convrot_quant_act(16, 0, 512, 0, 512, 0, None, 16, 1, 512, 16, None, 0) == 0
    torch.cuda.synchronize()
    assert torch.all(y == 3.0)


# ---------------------------------------------------------------- whole layer
LAYER_CASES = [
    ("tiny", synth.WORKLOADS["tiny"]),
    ("qkv", small("qkv", 300, 600)),
    ("ffn_down", small("ffn_down", 200, 300)),
    ("ffn_up", small("ffn_up", 150, 700)),
    ("ragged", small("ragged", 129, 517)),
    ("wide_k", small("wide_k", 130, 260)),
]


def run_layer(wl, x, packed, scales, t, xdev=None):
    Kp = oracle.padded_k(wl.K)
    qw, sw = gpu_prepare_weight(packed, scales, t, wl.K)
    qa, sa = gpu_quant_act(x, wl.x_dtype, wl.K, wl.swiglu, xdev=xdev)
    y = gpu_gemm(qa, sa, qw, sw, wl.out_dtype, Kp)
    return y, (qa, sa, qw, sw)


@pytest.mark.parametrize("case,wl", LAYER_CASES, ids=[c[0] for c in LAYER_CASES])
def test_layer_matches_oracle(case, wl):
    x = synth.make_activations(wl)
    packed, scales, t = synth.make_nvfp4_weight(wl)
    y, (qa, sa, qw, sw) = run_layer(wl, x, packed, scales, t)
    ref, mid = oracle.convrot_linear(x, wl.x_dtype, packed, scales, t, wl.K, wl.out_dtype, wl.swiglu)
    Kp = oracle.padded_k(wl.K)
    assert_codes_match(codes_to_np(qa, Kp), mid["qa"])
    assert_codes_match(codes_to_np(qw, Kp), mid["qw"])
    assert_output_match(y.float().cpu().numpy(), ref)


PS_CASES = [
    ("bf16_swiglu", synth.Workload("ps1", 70, 1000, 300, "bf16", "bf16", True, 0.0, 1.0, 23)),
    ("fp16_plain", synth.Workload("ps2", 130, 768, 520, "fp16", "fp32", False, 0.02, 20.0, 24)),
    ("fp32_in", synth.Workload("ps3", 33, 512, 257, "fp32", "fp16", False, 0.0, 1.0, 25)),
    ("split_rows", synth.Workload("ps4", 9, 20000, 130, "bf16", "bf16", False, 0.01, 20.0, 28)),
]


@pytest.mark.parametrize("case,wl", PS_CASES, ids=[c[0] for c in PS_CASES])
def test_layer_with_channel_pre_scale_and_bias(case, wl):
    rng = np.random.default_rng(wl.seed)
    pre = np.exp(rng.uniform(-1.5, 1.5, wl.K)).astype(np.float32)
    bias = (rng.standard_normal(wl.N) * 0.5).astype(np.float32)
    x = synth.make_activations(wl)
    packed, scales, t = synth.make_nvfp4_weight(wl)
    Kp = oracle.padded_k(wl.K)
    qw, sw = gpu_prepare_weight(packed, scales, t, wl.K)
    xd = storage_to_dev(x, wl.x_dtype)
    qa = torch.empty(wl.M, Kp, dtype=torch.float16, device=DEV)
    sa = torch.empty(wl.M, dtype=torch.float32, device=DEV)
    import rotated_w4a8_int8_gb300 as cr
    cr.quant_act(xd, wl.K, qa, sa, swiglu=wl.swiglu, pre_scale=torch.from_numpy(pre).to(DEV))
    from gpu_util import TORCH_DT
    y = torch.empty(wl.M, wl.N, dtype=TORCH_DT[wl.out_dtype], device=DEV)
    cr.gemm(qa, sa, qw, sw, y, bias=torch.from_numpy(bias).to(DEV))
    ref, mid = oracle.convrot_linear(x, wl.x_dtype, packed, scales, t, wl.K, wl.out_dtype, wl.swiglu,
                                     pre_scale=pre, bias=bias)
    assert_codes_match(codes_to_np(qa, Kp), mid["qa"])
    assert_scales_match(sa.cpu().numpy(), mid["sa"])
    assert_output_match(y.float().cpu().numpy(), ref)


def test_widen_codes_is_exact():
    import rotated_w4a8_int8_gb300 as cr
    rng = np.random.default_rng(51)
    src = rng.integers(-128, 128, (37, 272)).astype(np.int8)
    src[0, :255] = np.arange(-127, 128)
    s = torch.from_numpy(src).to(DEV)
    d = torch.full((37, 280), 7.0, dtype=torch.float16, device=DEV)
    cr.widen_codes(s, d, cols=272)
    got = d.cpu().numpy()
    assert np.array_equal(got[:, :272].astype(np.int32), src.astype(np.int32))
    assert np.all(got[:, 272:] == 7.0)


def test_w8a8_resident_s8_weights_match_the_w4a8_layer():
    # weights prepared once into S8 storage, widened per call: same outputs
    import rotated_w4a8_int8_gb300 as cr
    wl = small("qkv", 200, 300)
    x = synth.make_activations(wl)
    packed, scales, t = synth.make_nvfp4_weight(wl)
    Kp = oracle.padded_k(wl.K)
    q16, sw = gpu_prepare_weight(packed, scales, t, wl.K, fmt="f16")
    q8, sw8 = gpu_prepare_weight(packed, scales, t, wl.K, fmt="s8")
    wide = torch.empty(wl.N, Kp, dtype=torch.float16, device=DEV)
    cr.widen_codes(q8, wide, cols=Kp)
    assert torch.equal(wide, q16) and torch.equal(sw8, sw)
    qa, sa = gpu_quant_act(x, wl.x_dtype, wl.K)
    y1 = gpu_gemm(qa, sa, q16, sw, "bf16", Kp)
    y2 = gpu_gemm(qa, sa, wide, sw8, "bf16", Kp)
    assert torch.equal(y1, y2)
