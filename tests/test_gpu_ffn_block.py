"""The FFN block fc1 -> SwiGLU + rotation + S8 -> fc2 (MiniMax-H3 explainer on
modelpad.app, MLP section; the FFN-down entry of the ConvRot layer fuses the
SwiGLU into the activation quantisation), composed from the three C-ABI
calls, against the oracle's chain computed from the same original inputs."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import (DEV, assert_output_match, ensure_built, gpu_prepare_weight, storage_to_dev)

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


def test_ffn_block_matches_oracle_chain():
    ensure_built()
    import rotated_w4a8_int8_gb300 as cr
    M, H, F = 150, 512, 768                     # tokens, hidden, FFN width (fc1 out = 2F)
    up = synth.Workload("fc1", M, H, 2 * F, "bf16", "bf16", False, 0.01, 20.0, 31)
    down = synth.Workload("fc2", M, F, H, "bf16", "bf16", True, 0.0, 1.0, 32)
    x = synth.make_activations(up)
    p1, s1, t1 = synth.make_nvfp4_weight(up, std=0.05)
    p2, s2, t2 = synth.make_nvfp4_weight(down, std=0.05)

    # GPU: fc1 (BF16 out) -> SwiGLU + rotation + S8 -> fc2
    Hp, Fp = oracle.padded_k(H), oracle.padded_k(F)
    w1, sw1 = gpu_prepare_weight(p1, s1, t1, H)
    w2, sw2 = gpu_prepare_weight(p2, s2, t2, F)
    xq = torch.empty(M, Hp, dtype=torch.float16, device=DEV)
    sx = torch.empty(M, dtype=torch.float32, device=DEV)
    cr.quant_act(storage_to_dev(x, "bf16"), H, xq, sx)
    h2 = torch.empty(M, 2 * F, dtype=torch.bfloat16, device=DEV)
    cr.gemm(xq, sx, w1, sw1, h2)
    hq = torch.empty(M, Fp, dtype=torch.float16, device=DEV)
    sh = torch.empty(M, dtype=torch.float32, device=DEV)
    cr.quant_act(h2, F, hq, sh, swiglu=True)
    y = torch.empty(M, H, dtype=torch.bfloat16, device=DEV)
    cr.gemm(hq, sh, w2, sw2, y)
    torch.cuda.synchronize()

    # oracle chain from the original inputs; the fc1 output is stored in BF16
    # between the two layers, as on the GPU
    h2_ref, _ = oracle.convrot_linear(x, "bf16", p1, s1, t1, H, "bf16")
    h2_bits = synth.bf16_bits_from_f32(h2_ref.astype(np.float32))
    y_ref, _ = oracle.convrot_linear(h2_bits, "bf16", p2, s2, t2, F, "bf16", swiglu_flag=True)
    # the intermediate may differ by one BF16 unit where the two roundings
    # tie differently; the final outputs still meet the layer tolerance
    assert_output_match(h2.float().cpu().numpy(), h2_ref)
    assert_output_match(y.float().cpu().numpy(), y_ref)
