"""Failure detection on the GPU without a fault: a bounded wait runs out.

The GEMM kernel is launched with its TMA producer switched off, so the MMA
issuer's wait for operand tiles never completes.  After its time limit the
kernel records an error code, every role leaves its loop, the CTA pair meets
at the cluster barrier, frees tensor memory and returns.  The host then reads
the code, and the same context keeps computing correct results.
"""
import time

import numpy as np
import pytest
import torch

import oracle
from gpu_util import DEV, ensure_built, f16_codes_from_np

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


def test_gemm_wait_timeout_is_reported_and_context_survives():
    ensure_built()
    import rotated_w4a8_int8_gb300 as cr
    assert cr.device_error() == 0
    rng = np.random.default_rng(31)
    qa = rng.integers(-127, 128, (128, 256)).astype(np.int8)
    qw = rng.integers(-127, 128, (256, 256)).astype(np.int8)
    a, w = f16_codes_from_np(qa), f16_codes_from_np(qw)
    acc = torch.zeros((128, 256), dtype=torch.int32, device=DEV)
    t0 = time.time()
    cr.gemm_timeout_selftest(a, w, acc)
    code = cr.device_error()              # synchronises
    waited = time.time() - t0
    assert code != 0
    assert 1.0 < waited < 30.0
    assert cr.device_error() == 0         # reading clears the word
    cr.gemm_i32(a, w, acc)
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), oracle.int_gemm(qa, qw))
    assert cr.device_error() == 0


def test_gemm_wait_timeout_with_the_chunk_ring():
    # With norm bounds and K_p > 1024 the chunking warp runs beside the MMA
    # issuer: 2560 x 10240 outputs are 400 work items, more than five per CTA
    # pair, so after the issuer gives up the chunking warp is left waiting on
    # a slot that is never released and must leave on the abort as well.
    ensure_built()
    import rotated_w4a8_int8_gb300 as cr
    assert cr.device_error() == 0
    M, N, Kp = 2560, 10240, 2048
    a = torch.zeros((M, Kp), dtype=torch.float16, device=DEV)
    w = torch.zeros((N, Kp), dtype=torch.float16, device=DEV)
    na = torch.zeros(M, dtype=torch.float32, device=DEV)
    nw = torch.zeros(N, dtype=torch.float32, device=DEV)
    acc = torch.zeros((M, N), dtype=torch.int32, device=DEV)
    t0 = time.time()
    cr.gemm_timeout_selftest(a, w, acc, a_norm=na, w_norm=nw)
    code = cr.device_error()
    waited = time.time() - t0
    assert code != 0
    assert 1.0 < waited < 30.0
    assert cr.device_error() == 0
    # the context still computes: the same shape with real codes, exact
    rng = np.random.default_rng(5)
    qa = rng.integers(-127, 128, (M, Kp)).astype(np.int8)
    qw = rng.integers(-127, 128, (N, Kp)).astype(np.int8)
    cr.gemm_i32(f16_codes_from_np(qa), f16_codes_from_np(qw), acc)
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), oracle.int_gemm(qa, qw))
    assert cr.device_error() == 0
