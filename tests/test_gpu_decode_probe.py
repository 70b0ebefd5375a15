"""The decode-inside-GEMM producer probe (a measurement aid beside the layer).

For one chosen work unit, the codes that the probe's producer warps build in
shared memory, in the GEMM's swizzled B-operand layout, must equal the weight
kernel's FP16 codes for the same 128 weight rows bit for bit: the same NVFP4
decode, rotation, products (t/16, then the reciprocal of the row scale) and
rounding.  Rows past N come out zero, and no wait runs out.  Both NVFP4 sources
are used: the synthetic encoder and uniformly random bytes over the whole code
space (the ComfyUI-native checkpoints of the Load ConvRot DiT entry, ComfyUI
Turing Utils page, node list).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import DEV, assert_codes_match, ensure_built, gpu_prepare_weight
from test_gpu_edge_codes import random_nvfp4

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

ROWS = 128


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def synth_weight():
    # ragged N (the last 128-row half holds 44 rows) and ragged K (K_s / 2 not
    # a multiple of 16: the 8-byte load path)
    wl = synth.Workload("probe", 8, 5000, 300, "bf16", "bf16", False, 0.0, 1.0, 31)
    packed, scales, t = synth.make_nvfp4_weight(wl)
    return packed, scales, t, wl.K


def random_weight():
    # whole NVFP4 code space at the QKV width (16-byte loads); rows 0..5 hold
    # the special scales and the all -0 row
    packed, scales = random_nvfp4(256, 5376, seed=5)
    return packed, scales, np.float32(0.37), 5376


def probe_dump(packed, scales, t, K, w_scale, m_strips, pw, unit):
    import rotated_w4a8_int8_gb300 as cr
    Kp = cr.padded_k(K)
    pd = torch.from_numpy(packed).to(DEV)
    sd = torch.from_numpy(scales).to(DEV)
    td = torch.tensor([float(t)], dtype=torch.float32, device=DEV)
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    dump = torch.full((ROWS, Kp), 77.0, dtype=torch.float16, device=DEV)   # sentinel: every entry is written
    cr.decode_gemm_probe(pd, sd, td, w_scale, K, m_strips, pw, status, dump=dump, dump_unit=unit)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return dump


@pytest.mark.parametrize("pw", [8, 16])
@pytest.mark.parametrize("source,m_strips,units", [("synth", 3, (2, 7)), ("random", 2, (3, 0))])
def test_probe_codes_equal_the_weight_kernels(source, m_strips, units, pw):
    packed, scales, t, K = synth_weight() if source == "synth" else random_weight()
    N = packed.shape[0]
    Kp = oracle.padded_k(K)
    q, s = gpu_prepare_weight(packed, scales, t, K, fmt="f16")
    n_halves = -(-N // ROWS)
    for unit in units:                                      # two calls in a row
        r0 = (unit % n_halves) * ROWS
        nv = min(ROWS, N - r0)
        dump = probe_dump(packed, scales, t, K, s, m_strips, pw, unit)
        assert torch.equal(dump[:nv], q[r0:r0 + nv, :Kp]), (unit, nv)
        assert torch.count_nonzero(dump[nv:]).item() == 0
    if source == "random":
        # degenerate rows (zero scales in every block; every element -0) give zero codes here too
        dump = probe_dump(packed, scales, t, K, s, m_strips, pw, 0)
        assert torch.count_nonzero(dump[2]).item() == 0 and torch.count_nonzero(dump[5]).item() == 0


def test_probe_codes_against_the_oracle():
    # the same codes held to the oracle at the parity bars, independent of the weight kernel
    packed, scales, t, K = synth_weight()
    rq, _ = oracle.prepare_weight(packed, scales, t, K)
    _, s = gpu_prepare_weight(packed, scales, t, K, fmt="f16")
    dump = probe_dump(packed, scales, t, K, s, 1, 16, 1)
    assert_codes_match(dump.to(torch.int32).cpu().numpy(), rq[ROWS:2 * ROWS])


def test_probe_without_dump_runs_a_full_schedule():
    # QKV-width rows over many units per CTA (no dump): the waits all complete
    import rotated_w4a8_int8_gb300 as cr
    packed, scales, t, K = random_weight()
    _, s = gpu_prepare_weight(packed, scales, t, K, fmt="f16")
    pd = torch.from_numpy(packed).to(DEV)
    sd = torch.from_numpy(scales).to(DEV)
    td = torch.tensor([float(t)], dtype=torch.float32, device=DEV)
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    for pw in (8, 16):
        cr.decode_gemm_probe(pd, sd, td, s, K, 500, pw, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
