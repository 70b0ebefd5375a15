"""Helpers of the GPU parity tests: move seeded inputs to the device, run the
three C-ABI calls through the binding, bring results back, compare."""
import numpy as np
import torch

import rotated_w4a8_int8_gb300 as cr

DEV = torch.device("cuda:0")
TORCH_DT = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}


def ensure_built():
    import __graft_entry__
    __graft_entry__.build()


def storage_to_dev(x: np.ndarray, dtype: str) -> torch.Tensor:
    if dtype == "fp32":
        return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(DEV)
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(DEV).view(TORCH_DT[dtype])


def codes_tensor(rows, Kp, fmt="f16", ld=None):
    dt = torch.float16 if fmt == "f16" else torch.int8
    ld = Kp if ld is None else ld
    return torch.empty(rows, ld, dtype=dt, device=DEV)


def codes_to_np(q: torch.Tensor, Kp: int) -> np.ndarray:
    return q[:, :Kp].to(torch.int32).cpu().numpy()


def gpu_prepare_weight(packed, scales, t, K, fmt="f16", ld=None):
    N = packed.shape[0]
    Kp = cr.padded_k(K)
    pd = torch.from_numpy(packed).to(DEV)
    sd = torch.from_numpy(scales).to(DEV)
    td = torch.tensor([float(t)], dtype=torch.float32, device=DEV)
    q = codes_tensor(N, Kp, fmt, ld)
    s = torch.empty(N, dtype=torch.float32, device=DEV)
    cr.prepare_weight(pd, sd, td, K, q, s)
    return q, s


def gpu_quant_act(x, dtype, K, swiglu=False, fmt="f16", ld=None, xdev=None):
    xd = storage_to_dev(x, dtype) if xdev is None else xdev
    M = xd.shape[0]
    Kp = cr.padded_k(K)
    q = codes_tensor(M, Kp, fmt, ld)
    s = torch.empty(M, dtype=torch.float32, device=DEV)
    cr.quant_act(xd, K, q, s, swiglu=swiglu)
    return q, s


def gpu_gemm(qa, sa, qw, sw, out_dtype, Kp):
    y = torch.empty(qa.shape[0], qw.shape[0], dtype=TORCH_DT[out_dtype], device=DEV)
    cr.gemm(qa, sa, qw, sw, y, K_p=Kp)
    return y


def f16_codes_from_np(q: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(q).astype(np.float16)).to(DEV)


def assert_codes_match(got: np.ndarray, ref: np.ndarray, min_equal=0.9999):
    assert got.shape == ref.shape
    d = np.abs(got.astype(np.int64) - ref.astype(np.int64))
    frac = float(np.mean(d == 0))
    assert d.max() <= 1, f"code differs by {d.max()}"
    assert frac >= min_equal, f"only {frac:.6f} of codes equal"
    return frac


def assert_scales_match(got: np.ndarray, ref: np.ndarray, rtol=1e-6):
    got = got.astype(np.float64)
    ref = ref.astype(np.float64)
    assert np.all((got == 0) == (ref == 0))
    nz = ref != 0
    assert np.all(np.abs(got[nz] - ref[nz]) <= rtol * np.abs(ref[nz]))


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    x = np.maximum(np.abs(x), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(x)) - 7)


def assert_output_match(got: np.ndarray, ref: np.ndarray, rel_l2=1e-3, ulps=2.0):
    got = got.astype(np.float64)
    ref = ref.astype(np.float64)
    assert np.all(np.isfinite(got))
    den = np.linalg.norm(ref)
    rel = float(np.linalg.norm(got - ref) / den) if den > 0 else float(np.linalg.norm(got))
    assert rel <= rel_l2, f"relative L2 {rel:.3e}"
    rowmax = np.max(np.abs(ref), axis=1, keepdims=True)
    lim = ulps * bf16_ulp(rowmax)
    err = np.abs(got - ref)
    assert np.all(err <= lim), f"max element error {np.max(err / lim):.2f} x the limit"
    return rel
