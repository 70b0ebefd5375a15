"""Host-side pieces of bench.py that the reported numbers rest on (CPU only).

The roofline fractions divide algorithmic bytes and FLOP by measured times;
these tests pin the per-workload counts to the formulas the measurement
section states (one read of the kernel's inputs, one write of its outputs),
the replica aggregation, and the source hash that decides whether a stored
ncu traffic figure still applies (bench.py reports null traffic otherwise).
"""
import pytest

import bench
import synth


def test_qkv_algorithmic_counts():
    sz = bench.layer_sizes(synth.WORKLOADS["qkv"])
    M, K, N = 19989, 5376, 21504
    assert sz["Kp"] == 5376 and sz["Ks"] == 5376
    # BF16 input once, FP16 codes once, one FP32 scale per row
    assert sz["act_bytes"] == M * K * 2 + M * K * 2 + 4 * M == 429923412
    # packed NVFP4 + E4M3 scales + the tensor scale once, FP16 codes once, one FP32 scale per row
    assert sz["w_bytes"] == N * K // 2 + N * K // 16 + 4 + N * K * 2 + 4 * N == 296325124
    assert sz["gemm_flops"] == 2.0 * M * N * K
    assert abs(sz["gemm_flops"] - 4.6217e12) / 4.6217e12 < 1e-4


def test_ragged_and_swiglu_counts():
    rg = bench.layer_sizes(synth.WORKLOADS["ragged"])
    assert rg["Kp"] == 5120 and rg["Ks"] == 5008
    # effective TOPS use the logical K, the GEMM's FLOP the padded K
    assert rg["ops"] == 2.0 * 4097 * 21500 * 5000 and rg["gemm_flops"] == 2.0 * 4097 * 21500 * 5120
    fd = bench.layer_sizes(synth.WORKLOADS["ffn_down"])
    # the SwiGLU kernel reads gate and value (2K BF16 per token) and writes K codes
    assert fd["act_bytes"] == 19989 * 28672 * 2 + 19989 * 14336 * 2 + 4 * 19989


def test_replica_aggregation():
    # two replicas of a 10-step job timed at 20 ms (max over ranks): 2 * 10 * ops / 0.02 s
    assert bench.aggregate_tops(1e12, 10, 20.0, 2) == pytest.approx(1000.0)


def test_source_hash_ignores_comments(tmp_path):
    a = tmp_path / "a.cu"
    b = tmp_path / "b.cu"
    c = tmp_path / "c.cu"
    a.write_text("int f(int x) {\n  return x + 1;  // add one\n}\n")
    b.write_text("/* header */\nint f(int x) {\n\n  return x + 1;\n}\n")
    c.write_text("int f(int x) {\n  return x + 2;\n}\n")
    assert bench.code_sha16(str(a)) == bench.code_sha16(str(b))
    assert bench.code_sha16(str(a)) != bench.code_sha16(str(c))
