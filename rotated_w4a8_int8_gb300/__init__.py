"""Python binding of the ConvRot W4A8 C ABI (libconvrot.so).

Argument marshalling only: every step of the layer runs in the CUDA kernels
behind the C ABI declared in include/convrot.h.  Tensors are torch CUDA
tensors (PyTorch supplies device memory and streams); each function passes
their device pointers and the current stream to the library.  There is no
CPU fallback: if the library is missing or a call fails, an exception says
so.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "load_library", "padded_k", "status_string", "last_error", "prepare_weight", "quant_act", "gemm",
    "gemm_i32", "widen_codes", "gemm_timeout_selftest", "int8_mma_probe", "decode_gemm_probe",
    "device_error", "ConvRotError", "BF16", "FP16",
    "FP32", "CODES_S8",
    "CODES_F16", "LIB_PATH", "EXPORTS",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libconvrot.so")
BF16, FP16, FP32 = 0, 1, 2
CODES_S8, CODES_F16 = 0, 1
EXPORTS = ("convrot_padded_k", "convrot_status_string", "convrot_prepare_weight",
           "convrot_quant_act", "convrot_gemm", "convrot_gemm_i32", "convrot_device_error",
           "convrot_last_error", "convrot_gemm_timeout_selftest", "convrot_widen_codes", "convrot_int8_mma_probe",
           "convrot_decode_gemm_probe")

_lib = None


class ConvRotError(RuntimeError):
    def __init__(self, fn: str, status: int):
        detail = last_error() if status == 4 else ""
        msg = f"{fn} failed: {status_string(status)} (status {status})"
        super().__init__(msg + (f": {detail}" if detail else ""))
        self.status = status


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libconvrot.so (built by build()); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} not found: run __graft_entry__.build() (nvcc, sm_103a) first")
    lib = ctypes.CDLL(path)
    i32, i64, vp, f = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p, None
    lib.convrot_padded_k.argtypes = [i32]
    lib.convrot_padded_k.restype = i32
    lib.convrot_status_string.argtypes = [i32]
    lib.convrot_status_string.restype = ctypes.c_char_p
    lib.convrot_prepare_weight.argtypes = [vp, vp, vp, i32, i32, vp, i32, i64, vp, vp, vp]
    lib.convrot_prepare_weight.restype = i32
    lib.convrot_quant_act.argtypes = [vp, i32, i64, i32, i32, i32, vp, vp, i32, i64, vp, vp, vp]
    lib.convrot_quant_act.restype = i32
    lib.convrot_gemm.argtypes = [vp, i64, vp, vp, vp, i64, vp, vp, vp, i32, i32, i32, vp, i32, i64, vp]
    lib.convrot_gemm.restype = i32
    lib.convrot_gemm_i32.argtypes = [vp, i64, vp, vp, i64, vp, i32, i32, i32, vp, i64, vp]
    lib.convrot_gemm_i32.restype = i32
    lib.convrot_widen_codes.argtypes = [vp, i64, i32, i32, vp, i64, vp]
    lib.convrot_widen_codes.restype = i32
    lib.convrot_gemm_timeout_selftest.argtypes = [vp, i64, vp, vp, i64, vp, i32, i32, i32, vp, i64, vp]
    lib.convrot_gemm_timeout_selftest.restype = i32
    lib.convrot_int8_mma_probe.argtypes = [i32, i32, vp, vp]
    lib.convrot_int8_mma_probe.restype = i32
    lib.convrot_decode_gemm_probe.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, vp, i64, i32, vp, vp]
    lib.convrot_decode_gemm_probe.restype = i32
    lib.convrot_last_error.argtypes = []
    lib.convrot_last_error.restype = ctypes.c_char_p
    lib.convrot_device_error.argtypes = [vp, ctypes.POINTER(i32)]
    lib.convrot_device_error.restype = i32
    del f
    _lib = lib
    return lib


def padded_k(K: int) -> int:
    return load_library().convrot_padded_k(int(K))


def status_string(status: int) -> str:
    return load_library().convrot_status_string(int(status)).decode()


def last_error() -> str:
    """Text of the CUDA error behind the calling thread's last CONVROT_ERR_CUDA."""
    return load_library().convrot_last_error().decode()


def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


def _ld(t) -> int:
    """Row pitch in elements.  Torch may report any stride (often 0) for a
    dimension of size 1; a single row has no pitch, so its own width is
    passed instead (rows must be contiguous)."""
    if t.dim() >= 2 and t.shape[0] <= 1:
        return max(int(t.stride(0)), int(t.shape[1]))
    return int(t.stride(0))


def _stream(stream) -> int:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    return int(getattr(stream, "cuda_stream", stream))


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise ConvRotError(fn, status)


def _dtype_code(t) -> int:
    import torch
    return {torch.bfloat16: BF16, torch.float16: FP16, torch.float32: FP32}[t.dtype]


def _codes_fmt(t) -> int:
    import torch
    return {torch.int8: CODES_S8, torch.float16: CODES_F16}[t.dtype]


def prepare_weight(w_fp4, w_sf, w_tensor_scale, K: int, w_q, w_scale, w_norm=None, stream=None) -> None:
    """convrot_prepare_weight: w_fp4 uint8 [N, K_s/2], w_sf uint8 [N, K_s/16],
    w_tensor_scale float32 [1], w_q int8 or float16 [N, >=K_p], w_scale float32 [N],
    w_norm None or float32 [N] (bounds on the rows' code norms, for gemm)."""
    N = w_fp4.shape[0]
    _check("convrot_prepare_weight", load_library().convrot_prepare_weight(
        _ptr(w_fp4), _ptr(w_sf), _ptr(w_tensor_scale), N, int(K), _ptr(w_q), _codes_fmt(w_q),
        _ld(w_q), _ptr(w_scale), _ptr(w_norm), _stream(stream)))


def quant_act(x, K: int, a_q, a_scale, swiglu: bool = False, pre_scale=None, a_norm=None, stream=None) -> None:
    """convrot_quant_act: x bf16/fp16/fp32 [M, >=K or 2K], a_q int8 or float16
    [M, >=K_p], a_scale float32 [M], pre_scale None or float32 [K], a_norm None
    or float32 [M] (bounds on the rows' code norms, for gemm)."""
    M = x.shape[0]
    _check("convrot_quant_act", load_library().convrot_quant_act(
        _ptr(x), _dtype_code(x), _ld(x), M, int(K), int(bool(swiglu)), _ptr(pre_scale),
        _ptr(a_q), _codes_fmt(a_q), _ld(a_q), _ptr(a_scale), _ptr(a_norm), _stream(stream)))


def gemm(a_q, a_scale, w_q, w_scale, out, K_p: int | None = None, bias=None, a_norm=None, w_norm=None,
         stream=None) -> None:
    """convrot_gemm: a_q float16 codes [M, >=K_p], w_q float16 codes [N, >=K_p],
    out bf16/fp16/fp32 [M, >=N] (N = w_q rows), bias None or float32 [N],
    a_norm / w_norm None or the code-norm bounds from quant_act / prepare_weight."""
    M, N = a_q.shape[0], w_q.shape[0]
    K_p = a_q.shape[1] if K_p is None else K_p
    _check("convrot_gemm", load_library().convrot_gemm(
        _ptr(a_q), _ld(a_q), _ptr(a_scale), _ptr(a_norm), _ptr(w_q), _ld(w_q), _ptr(w_scale), _ptr(w_norm),
        _ptr(bias), M, N, int(K_p), _ptr(out), _dtype_code(out), _ld(out), _stream(stream)))


def gemm_i32(a_q, w_q, acc, K_p: int | None = None, a_norm=None, w_norm=None, stream=None) -> None:
    """convrot_gemm_i32: raw int32 accumulators into acc int32 [M, >=N]."""
    M, N = a_q.shape[0], w_q.shape[0]
    K_p = a_q.shape[1] if K_p is None else K_p
    _check("convrot_gemm_i32", load_library().convrot_gemm_i32(
        _ptr(a_q), _ld(a_q), _ptr(a_norm), _ptr(w_q), _ld(w_q), _ptr(w_norm), M, N, int(K_p), _ptr(acc),
        _ld(acc), _stream(stream)))


def widen_codes(src, dst, cols: int | None = None, stream=None) -> None:
    """convrot_widen_codes: int8 S8 codes [rows, >=cols] -> float16 codes [rows, >=cols]."""
    rows = src.shape[0]
    cols = src.shape[1] if cols is None else cols
    _check("convrot_widen_codes", load_library().convrot_widen_codes(
        _ptr(src), _ld(src), rows, int(cols), _ptr(dst), _ld(dst), _stream(stream)))


def gemm_timeout_selftest(a_q, w_q, acc, K_p: int | None = None, a_norm=None, w_norm=None, stream=None) -> None:
    """convrot_gemm_timeout_selftest: the GEMM with its producer off (a wait runs out)."""
    M, N = a_q.shape[0], w_q.shape[0]
    K_p = a_q.shape[1] if K_p is None else K_p
    _check("convrot_gemm_timeout_selftest", load_library().convrot_gemm_timeout_selftest(
        _ptr(a_q), _ld(a_q), _ptr(a_norm), _ptr(w_q), _ld(w_q), _ptr(w_norm), M, N, int(K_p), _ptr(acc),
        _ld(acc), _stream(stream)))


def int8_mma_probe(blocks: int, iters: int, out, stream=None) -> None:
    """convrot_int8_mma_probe: out int32 [blocks * 4]; each entry becomes 8 * 32 * iters."""
    _check("convrot_int8_mma_probe", load_library().convrot_int8_mma_probe(
        int(blocks), int(iters), _ptr(out), _stream(stream)))


def decode_gemm_probe(w_fp4, w_sf, w_tensor_scale, w_scale, K: int, m_strips: int, producer_warps: int, status,
                      dump=None, dump_unit: int = 0, stream=None) -> None:
    """convrot_decode_gemm_probe: the producer of a decode-inside-GEMM over m_strips token strips.

    status: int32 [1] (device); dump: optional FP16 [128, >= K_p] receiving unit dump_unit's codes.
    """
    N = w_fp4.shape[0]
    _check("convrot_decode_gemm_probe", load_library().convrot_decode_gemm_probe(
        _ptr(w_fp4), _ptr(w_sf), _ptr(w_tensor_scale), _ptr(w_scale), N, int(K), int(m_strips),
        int(producer_warps), _ptr(dump), _ld(dump) if dump is not None else 0, int(dump_unit), _ptr(status),
        _stream(stream)))


def device_error(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device failure word."""
    code = ctypes.c_int(0)
    load_library().convrot_device_error(_stream(stream), ctypes.byref(code))
    return code.value
