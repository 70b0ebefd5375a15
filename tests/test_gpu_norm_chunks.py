"""Code-norm bounds and the GEMM's single-chunk path.

convrot_quant_act and convrot_prepare_weight can write, per row, an upper
bound on the Euclidean norm of the row's codes.  convrot_gemm uses them to run
a 256 x 256 tile's whole K loop as one FP32 chunk when max bound(A rows) x
max bound(B rows) < 2^24: by Cauchy-Schwarz every partial sum is then below
2^24, so FP32 accumulation of the integer products stays exact.  These tests
check that the bounds hold, that the single-chunk path is exact where the
bound is tight, that it is taken on ordinary data, and that outputs are
bit-identical with and without the bounds.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import DEV, TORCH_DT, codes_to_np, ensure_built, f16_codes_from_np, storage_to_dev

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

LIMIT = 2.0 ** 24


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    import rotated_w4a8_int8_gb300 as cr
    yield
    assert cr.device_error() == 0


def small(name, M, N):
    wl = synth.WORKLOADS[name]
    return synth.Workload(f"{name}_n", M, wl.K, N, wl.x_dtype, wl.out_dtype, wl.swiglu,
                          wl.outlier_frac, wl.outlier_mult, wl.seed)


def check_bounds(q, bound, Kp):
    true = np.sqrt(np.sum(q.astype(np.float64) ** 2, axis=1))
    b = bound.astype(np.float64)
    assert np.all(b >= true), f"bound below the norm by {np.max(true - b)}"
    assert np.all(b <= 1.002 * true + np.sqrt(Kp)), "bound far too loose"


ACT = [small("qkv", 150, 8), small("ffn_down", 40, 8), small("ragged", 33, 8), small("wide_k", 12, 8),
       synth.Workload("deg", 4, 512, 8, "bf16", "bf16", False, 0.0, 1.0, 31)]


@pytest.mark.parametrize("wl", ACT, ids=[w.name for w in ACT])
def test_activation_code_norm_bounds_hold(wl):
    import rotated_w4a8_int8_gb300 as cr
    x = synth.make_activations(wl)
    if wl.name == "deg":
        x[1] = 0                                     # degenerate row: bound 0
    Kp = oracle.padded_k(wl.K)
    q = torch.empty(wl.M, Kp, dtype=torch.float16, device=DEV)
    s = torch.empty(wl.M, dtype=torch.float32, device=DEV)
    nrm = torch.full((wl.M,), -1.0, dtype=torch.float32, device=DEV)
    cr.quant_act(storage_to_dev(x, wl.x_dtype), wl.K, q, s, swiglu=wl.swiglu, a_norm=nrm)
    qn, bn = codes_to_np(q, Kp), nrm.cpu().numpy()
    check_bounds(qn, bn, Kp)
    if wl.name == "deg":
        assert bn[1] == 0


WTS = [small("qkv", 8, 130), small("ffn_down", 8, 40), small("ragged", 8, 33), small("wide_k", 8, 12),
       synth.Workload("maxkp", 8, 65536, 3, "bf16", "bf16", False, 0.0, 1.0, 19)]


@pytest.mark.parametrize("wl", WTS, ids=[w.name for w in WTS])
def test_weight_code_norm_bounds_hold(wl):
    import rotated_w4a8_int8_gb300 as cr
    packed, scales, t = synth.make_nvfp4_weight(wl)
    Kp = oracle.padded_k(wl.K)
    q = torch.empty(wl.N, Kp, dtype=torch.float16, device=DEV)
    s = torch.empty(wl.N, dtype=torch.float32, device=DEV)
    nrm = torch.full((wl.N,), -1.0, dtype=torch.float32, device=DEV)
    cr.prepare_weight(torch.from_numpy(packed).to(DEV), torch.from_numpy(scales).to(DEV),
                      torch.tensor([float(t)], dtype=torch.float32, device=DEV), wl.K, q, s, w_norm=nrm)
    check_bounds(codes_to_np(q, Kp), nrm.cpu().numpy(), Kp)


def exact_bounds(q):
    """Bounds a caller may pass: the true norms, rounded up."""
    n = np.sqrt(np.sum(q.astype(np.float64) ** 2, axis=1))
    return torch.from_numpy(np.nextafter(n.astype(np.float32), np.float32(np.inf))).to(DEV)


def run_i32(qa, qw, with_norms):
    import rotated_w4a8_int8_gb300 as cr
    acc = torch.full((qa.shape[0], qw.shape[0]), 7, dtype=torch.int32, device=DEV)
    kw = dict(a_norm=exact_bounds(qa), w_norm=exact_bounds(qw)) if with_norms else {}
    cr.gemm_i32(f16_codes_from_np(qa), f16_codes_from_np(qw), acc, **kw)
    return acc.cpu().numpy().astype(np.int64)


@pytest.mark.parametrize("pattern", ["max_half", "odd_half", "small_random", "over_bound"])
def test_single_chunk_path_is_exact(pattern):
    # max_half / odd_half: 1024 of 2048 entries at 127 in both operands, so the
    # bound 127^2 * 1024 = 16,516,096 sits just below 2^24 and the tile runs as
    # one 2048-deep chunk whose running sums reach the bound; odd_half makes
    # every running sum odd.  small_random: codes in [-20, 20] over K = 5376.
    # over_bound: all 127 over 20480, far above the bound: 1024-deep chunks.
    rng = np.random.default_rng(7)
    M, N = 300, 260
    if pattern in ("max_half", "odd_half"):
        Kp = 2048
        qa = np.zeros((M, Kp), np.int8)
        qw = np.zeros((N, Kp), np.int8)
        qa[:, :1024] = 127
        qw[:, :1024] = 127
        qa[1::2, :1024] = -127
        if pattern == "odd_half":
            qw[:, 15:1024:16] = 126
    elif pattern == "small_random":
        Kp = 5376
        qa = rng.integers(-20, 21, (M, Kp)).astype(np.int8)
        qw = rng.integers(-20, 21, (N, Kp)).astype(np.int8)
    else:
        Kp = 20480
        qa = np.full((M, Kp), 127, np.int8)
        qw = np.full((N, Kp), 127, np.int8)
        qw[:, 1::2] = -127
    na = np.sqrt(np.sum(qa.astype(np.float64) ** 2, axis=1)).max()
    nw = np.sqrt(np.sum(qw.astype(np.float64) ** 2, axis=1)).max()
    assert (na * nw < LIMIT) == (pattern != "over_bound")
    ref = oracle.int_gemm(qa, qw)
    assert np.array_equal(run_i32(qa, qw, True), ref)
    assert np.array_equal(run_i32(qa, qw, False), ref)


LAYERS = [small("qkv", 300, 600), small("ffn_down", 200, 300), small("ffn_up", 150, 520)]


@pytest.mark.parametrize("wl", LAYERS, ids=[w.name for w in LAYERS])
def test_layer_identical_with_and_without_norm_bounds(wl):
    import rotated_w4a8_int8_gb300 as cr
    x = synth.make_activations(wl)
    packed, scales, t = synth.make_nvfp4_weight(wl)
    Kp = oracle.padded_k(wl.K)
    qw = torch.empty(wl.N, Kp, dtype=torch.float16, device=DEV)
    sw = torch.empty(wl.N, dtype=torch.float32, device=DEV)
    nw = torch.empty(wl.N, dtype=torch.float32, device=DEV)
    qa = torch.empty(wl.M, Kp, dtype=torch.float16, device=DEV)
    sa = torch.empty(wl.M, dtype=torch.float32, device=DEV)
    na = torch.empty(wl.M, dtype=torch.float32, device=DEV)
    cr.prepare_weight(torch.from_numpy(packed).to(DEV), torch.from_numpy(scales).to(DEV),
                      torch.tensor([float(t)], dtype=torch.float32, device=DEV), wl.K, qw, sw, w_norm=nw)
    cr.quant_act(storage_to_dev(x, wl.x_dtype), wl.K, qa, sa, swiglu=wl.swiglu, a_norm=na)
    # at K_p = 5376 the bounds of ordinary codes allow one chunk, so the fast
    # path is what runs; at K_p = 14336 they exceed 2^24 (about 4200 each) and
    # the tile keeps its exact chunks
    assert (float(na.max()) * float(nw.max()) < LIMIT) == (Kp <= 8192)
    y1 = torch.empty(wl.M, wl.N, dtype=TORCH_DT[wl.out_dtype], device=DEV)
    y2 = torch.empty_like(y1)
    cr.gemm(qa, sa, qw, sw, y1)
    cr.gemm(qa, sa, qw, sw, y2, a_norm=na, w_norm=nw)
    assert torch.equal(y1, y2)
    acc1 = torch.empty(wl.M, wl.N, dtype=torch.int32, device=DEV)
    acc2 = torch.empty_like(acc1)
    cr.gemm_i32(qa, qw, acc1)
    cr.gemm_i32(qa, qw, acc2, a_norm=na, w_norm=nw)
    assert torch.equal(acc1, acc2)
    ref = oracle.int_gemm(codes_to_np(qa, Kp), codes_to_np(qw, Kp))
    assert np.array_equal(acc2.cpu().numpy().astype(np.int64), ref)


def test_mixed_items_and_ring_reuse():
    # 8192 x 5376 outputs = 32 x 21 = 672 work items of 256 x 256, about nine
    # per CTA pair, so the chunk counts handed to the MMA issuer pass through
    # every slot of its ring more than once.  K_p = 1280 (two exact chunks by
    # default).  Rows of three 256-row A blocks and two 256-row B blocks hold
    # +-127 everywhere: items where both meet have bounds 127^2 * 1280 above
    # 2^24 and keep their chunks; every other item runs as one chunk.
    rng = np.random.default_rng(11)
    M, N, Kp = 8192, 5376, 1280
    qa = rng.integers(-20, 21, (M, Kp)).astype(np.int8)
    qw = rng.integers(-20, 21, (N, Kp)).astype(np.int8)
    for m2 in (0, 5, 17):
        qa[m2 * 256:(m2 + 1) * 256] = rng.choice(np.array([-127, 127], np.int8), (256, Kp))
    for nt in (2, 9):
        qw[nt * 256:(nt + 1) * 256] = rng.choice(np.array([-127, 127], np.int8), (256, Kp))
    big = 127.0 * np.sqrt(Kp)
    assert big * big >= LIMIT and big * np.sqrt(np.sum(qw[:256].astype(np.float64) ** 2, axis=1)).max() < LIMIT
    ref = oracle.int_gemm(qa, qw)
    assert np.array_equal(run_i32(qa, qw, True), ref)


@pytest.mark.parametrize("t", [-3.7, 1e-6, 2.0e4])
def test_weight_bounds_hold_on_random_nvfp4_bytes(t):
    # any stored bytes (all 16 E2M1 codes, random non-NaN E4M3 scales with
    # subnormals and sign bits) and tensor scales of either sign and far from
    # 1: the bound comes from the decoded row before the rotation, scaled by |t|
    import rotated_w4a8_int8_gb300 as cr
    rng = np.random.default_rng(23)
    N, K = 64, 5000
    Ks = (K + 15) // 16 * 16
    Kp = oracle.padded_k(K)
    packed = rng.integers(0, 256, (N, Ks // 2), dtype=np.uint8)
    scales = rng.integers(0, 256, (N, Ks // 16), dtype=np.uint8)
    scales[(scales & 0x7F) == 0x7F] = 0x38                  # no NaN scale bytes
    q = torch.empty(N, Kp, dtype=torch.float16, device=DEV)
    s = torch.empty(N, dtype=torch.float32, device=DEV)
    nrm = torch.full((N,), -1.0, dtype=torch.float32, device=DEV)
    cr.prepare_weight(torch.from_numpy(packed).to(DEV), torch.from_numpy(scales).to(DEV),
                      torch.tensor([t], dtype=torch.float32, device=DEV), K, q, s, w_norm=nrm)
    check_bounds(codes_to_np(q, Kp), nrm.cpu().numpy(), Kp)


CODE_CASES = [small("qkv", 64, 8), small("ffn_down", 48, 8), small("wide_k", 16, 8),
              synth.Workload("pre", 40, 3000, 8, "bf16", "bf16", False, 0.0, 1.0, 41),
              synth.Workload("swpre", 40, 3000, 8, "bf16", "bf16", True, 0.0, 1.0, 43)]


@pytest.mark.parametrize("wl", CODE_CASES, ids=[w.name for w in CODE_CASES])
def test_codes_do_not_depend_on_asking_for_bounds(wl):
    # the bounds are a side result: codes and scales are bit-identical with and
    # without them (SwiGLU, channel pre-scales, split rows, and the weights)
    import rotated_w4a8_int8_gb300 as cr
    Kp = oracle.padded_k(wl.K)
    x = storage_to_dev(synth.make_activations(wl), wl.x_dtype)
    pre = None
    if wl.name in ("pre", "swpre"):
        gen = torch.Generator(device="cpu").manual_seed(5)
        pre = torch.exp(torch.rand(wl.K, generator=gen) * 2 - 1).to(DEV)
    outs = []
    for with_norm in (False, True):
        q = torch.empty(wl.M, Kp, dtype=torch.float16, device=DEV)
        s = torch.empty(wl.M, dtype=torch.float32, device=DEV)
        nrm = torch.empty(wl.M, dtype=torch.float32, device=DEV) if with_norm else None
        cr.quant_act(x, wl.K, q, s, swiglu=wl.swiglu, pre_scale=pre, a_norm=nrm)
        outs.append((q, s))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    ww = small(wl.name if wl.name in synth.WORKLOADS else "qkv", 8, 40)   # 40 weight rows, the same K
    packed, scales, t = synth.make_nvfp4_weight(ww)
    Kpw = oracle.padded_k(ww.K)
    wouts = []
    for with_norm in (False, True):
        q = torch.empty(ww.N, Kpw, dtype=torch.float16, device=DEV)
        s = torch.empty(ww.N, dtype=torch.float32, device=DEV)
        nrm = torch.empty(ww.N, dtype=torch.float32, device=DEV) if with_norm else None
        cr.prepare_weight(torch.from_numpy(packed).to(DEV), torch.from_numpy(scales).to(DEV),
                          torch.tensor([float(t)], dtype=torch.float32, device=DEV), ww.K, q, s, w_norm=nrm)
        wouts.append((q, s))
    assert torch.equal(wouts[0][0], wouts[1][0]) and torch.equal(wouts[0][1], wouts[1][1])


@pytest.mark.parametrize("out_dtype", ["bf16", "fp16", "fp32"])
def test_bias_and_output_dtypes_identical_with_and_without_norm_bounds(out_dtype):
    # the one-chunk epilogue (FP32 accumulator bits kept) against the chunked
    # one (int32 sums converted once), with a per-channel bias, every output type
    import rotated_w4a8_int8_gb300 as cr
    wl = small("qkv", 200, 300)
    x = synth.make_activations(wl)
    packed, scales, t = synth.make_nvfp4_weight(wl)
    Kp = oracle.padded_k(wl.K)
    qw = torch.empty(wl.N, Kp, dtype=torch.float16, device=DEV)
    sw = torch.empty(wl.N, dtype=torch.float32, device=DEV)
    nw = torch.empty(wl.N, dtype=torch.float32, device=DEV)
    qa = torch.empty(wl.M, Kp, dtype=torch.float16, device=DEV)
    sa = torch.empty(wl.M, dtype=torch.float32, device=DEV)
    na = torch.empty(wl.M, dtype=torch.float32, device=DEV)
    cr.prepare_weight(torch.from_numpy(packed).to(DEV), torch.from_numpy(scales).to(DEV),
                      torch.tensor([float(t)], dtype=torch.float32, device=DEV), wl.K, qw, sw, w_norm=nw)
    cr.quant_act(storage_to_dev(x, wl.x_dtype), wl.K, qa, sa, a_norm=na)
    assert float(na.max()) * float(nw.max()) < LIMIT
    bias = (torch.randn(wl.N, generator=torch.Generator().manual_seed(9)) * 0.1).to(DEV)
    y1 = torch.empty(wl.M, wl.N, dtype=TORCH_DT[out_dtype], device=DEV)
    y2 = torch.empty_like(y1)
    cr.gemm(qa, sa, qw, sw, y1, bias=bias)
    cr.gemm(qa, sa, qw, sw, y2, bias=bias, a_norm=na, w_norm=nw)
    assert torch.equal(y1, y2)
