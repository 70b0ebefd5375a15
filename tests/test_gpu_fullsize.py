"""Parity at the workloads' full sizes, through the same three C-ABI calls the
benchmark times (with the code-norm bounds where the benchmark asks for
them), checked on sampled outputs that the oracle can compute.

Per workload: every weight row's S8 codes and scale against the oracle; a
sample of token rows (first, last, M-tile boundaries, random) for the
activation codes and scales; the final outputs of those rows over all N
columns; and the raw int32 accumulators of those rows, given the GPU's own S8
operands, bit-exact against the oracle's integer GEMM.
"""
import numpy as np
import pytest
import torch

import bench
import oracle
import synth
from gpu_util import (DEV, TORCH_DT, assert_codes_match, assert_output_match, assert_scales_match,
                      codes_to_np, ensure_built, storage_to_dev)

pytestmark = [pytest.mark.gpu, pytest.mark.slow,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


def sample_rows(M, seed):
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 127, 128, 129, 255, 256, M // 2, M - 2, M - 1]
    rows = set(r for r in fixed if 0 <= r < M)
    rows.update(int(r) for r in rng.choice(M, size=min(M, 22), replace=False))
    return np.array(sorted(rows))


@pytest.mark.parametrize("name", ["qkv", "ffn_down", "ffn_up", "ragged", "wide_k"])
def test_full_size_layer(name):
    ensure_built()
    import rotated_w4a8_int8_gb300 as cr
    wl = synth.WORKLOADS[name]
    Kp = oracle.padded_k(wl.K)
    x = synth.make_activations(wl)
    packed, scales, t = synth.make_nvfp4_weight(wl)

    # the layer on the GPU, as timed by the benchmark: with the code-norm
    # bounds where the benchmark asks for them
    use_norms = bench.norms_pay(Kp)
    xd = storage_to_dev(x, wl.x_dtype)
    qw = torch.empty(wl.N, Kp, dtype=torch.float16, device=DEV)
    sw = torch.empty(wl.N, dtype=torch.float32, device=DEV)
    qa = torch.empty(wl.M, Kp, dtype=torch.float16, device=DEV)
    sa = torch.empty(wl.M, dtype=torch.float32, device=DEV)
    nw = torch.empty(wl.N, dtype=torch.float32, device=DEV) if use_norms else None
    na = torch.empty(wl.M, dtype=torch.float32, device=DEV) if use_norms else None
    cr.prepare_weight(torch.from_numpy(packed).to(DEV), torch.from_numpy(scales).to(DEV),
                      torch.tensor([float(t)], dtype=torch.float32, device=DEV), wl.K, qw, sw, w_norm=nw)
    cr.quant_act(xd, wl.K, qa, sa, swiglu=wl.swiglu, a_norm=na)
    y = torch.empty(wl.M, wl.N, dtype=TORCH_DT[wl.out_dtype], device=DEV)
    cr.gemm(qa, sa, qw, sw, y, K_p=Kp, a_norm=na, w_norm=nw)
    rows = sample_rows(wl.M, wl.seed)
    rows_t = torch.from_numpy(rows).to(DEV)
    acc = torch.empty(len(rows), wl.N, dtype=torch.int32, device=DEV)
    na_s = na.index_select(0, rows_t).contiguous() if use_norms else None
    cr.gemm_i32(qa.index_select(0, rows_t).contiguous(), qw, acc, K_p=Kp, a_norm=na_s, w_norm=nw)
    torch.cuda.synchronize()
    assert cr.device_error() == 0
    g_qw = codes_to_np(qw, Kp)
    g_sw = sw.cpu().numpy()
    g_qa = codes_to_np(qa.index_select(0, rows_t), Kp)
    g_sa = sa.cpu().numpy()[rows]
    g_y = y.index_select(0, rows_t).float().cpu().numpy().astype(np.float64)
    g_acc = acc.cpu().numpy().astype(np.int64)
    if use_norms:
        # the bounds hold: every weight row, the sampled token rows
        for q, b in ((g_qw, nw.cpu().numpy()), (g_qa, na_s.cpu().numpy())):
            true = np.sqrt(np.sum(q.astype(np.float64) ** 2, axis=1))
            assert np.all(b.astype(np.float64) >= true)
    del xd, qa, qw, y, acc
    torch.cuda.empty_cache()

    # oracle: the whole weight, the sampled token rows
    o_qw, o_sw = oracle.prepare_weight(packed, scales, t, wl.K)
    assert_codes_match(g_qw, o_qw)
    assert_scales_match(g_sw, o_sw)
    o_qa, o_sa = oracle.quant_act(x[rows], wl.x_dtype, wl.K, wl.swiglu)
    assert_codes_match(g_qa, o_qa)
    assert_scales_match(g_sa, o_sa)
    # identical S8 operands -> identical int32 accumulators
    assert np.array_equal(g_acc, oracle.int_gemm(g_qa, g_qw.astype(np.int8)))
    # the outputs against the oracle's own layer
    o_y = oracle.dequantize(oracle.int_gemm(o_qa, o_qw), o_sa, o_sw, wl.out_dtype)
    assert_output_match(g_y, o_y)
