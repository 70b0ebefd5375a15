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
    # algorithmic bytes: BF16 input once, one-byte S8 codes once, one FP32 scale per row
    assert sz["act_alg"] == M * K * 2 + M * K + 4 * M == 322462548
    # packed NVFP4 + E4M3 scales once, one-byte codes once, one FP32 scale per row
    assert sz["w_alg"] == N * K // 2 + N * K // 16 + N * K + 4 * N == 180719616
    # bytes moved with the codes held as FP16 for the GEMM (and the tensor scale read)
    # QKV (K_p = 5376) asks for the code-norm bounds: 4 more bytes per row
    assert sz["act_bytes"] == M * K * 2 + M * K * 2 + 8 * M == 430003368
    assert sz["w_bytes"] == N * K // 2 + N * K // 16 + 4 + N * K * 2 + 8 * N == 296411140
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
    assert fd["act_alg"] == 19989 * 28672 * 2 + 19989 * 14336 + 4 * 19989
    assert abs(fd["act_alg"] - 1432.9e6) / 1432.9e6 < 1e-3
    # ragged weights: K_s = 5008 stored, K_p = 5120 codes
    assert rg["w_alg"] == 21500 * 5008 // 2 + 21500 * 5008 // 16 + 21500 * 5120 + 4 * 21500


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


def test_single_gpu_guard_refuses_more_than_one_gpu():
    bench.single_gpu_guard(1, 1)
    for n, world in ((2, 1), (1, 2), (8, 8)):
        with pytest.raises(SystemExit) as e:
            bench.single_gpu_guard(n, world)
        assert "one GPU" in str(e.value)


def test_tensor_pipe_peak_formula():
    # 152 SMs at 1920 MHz: 8192 FLOP per clock per SM
    assert bench.tensor_pipe_peak(152, 1920.0) == pytest.approx(2390.8, rel=1e-4)


def test_reference_arm_shares_the_workload_config():
    wl = synth.WORKLOADS["qkv"]
    c = bench.bench_config(wl, 0)
    assert c["workload"] == "qkv M=19989 K=5376 N=21504 bf16->bf16"
    assert c == bench.bench_config(wl, 0)


def test_norm_bounds_requested_where_they_can_pay():
    # QKV / FFN-up (K_p = 5376) ask for them; FFN-down (14336) and wide K do not
    assert bench.norms_pay(5376) and bench.norms_pay(8192)
    assert not bench.norms_pay(14336) and not bench.norms_pay(20480)
