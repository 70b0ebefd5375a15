"""Host-side checks of the C ABI: the library loads, exports every declared
symbol, and rejects bad arguments before touching the GPU."""
import ctypes
import os
import re

import pytest

import rotated_w4a8_int8_gb300 as cr

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "convrot.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return cr.load_library()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+(convrot_\w+)\s*\(", text, re.M)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 7
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(cr.EXPORTS)


def test_padded_k(lib):
    assert [cr.padded_k(k) for k in (1, 255, 256, 257, 5000, 5376, 20480, 0, -3)] == \
        [256, 256, 256, 512, 5120, 5376, 20480, 0, 0]


def test_status_strings(lib):
    for s in range(6):
        assert cr.status_string(s)
    assert cr.status_string(99) == "unknown status"


def test_quant_act_rejects_bad_arguments(lib):
    f = lib.convrot_quant_act
    P = 1 << 20    # fake, never dereferenced: every call below fails validation first
    assert f(P, 0, 512, 4, 0, 0, None, P, 1, 512, P, None, 0) == 1                 # K <= 0
    assert f(P, 0, 512, -1, 512, 0, None, P, 1, 512, P, None, 0) == 1              # M < 0
    assert f(P, 7, 512, 4, 512, 0, None, P, 1, 512, P, None, 0) == 3               # dtype
    assert f(P, 0, 512, 4, 512, 0, None, P, 5, 512, P, None, 0) == 3               # code format
    assert f(P, 0, 511, 4, 512, 0, None, P, 1, 512, P, None, 0) == 1               # ld_x < K
    assert f(P, 0, 1023, 4, 512, 1, None, P, 1, 512, P, None, 0) == 1              # ld_x < 2K (SwiGLU)
    assert f(P, 0, 512, 4, 300, 0, None, P, 1, 300, P, None, 0) == 1               # ld_aq < K_p
    assert f(None, 0, 512, 4, 512, 0, None, P, 1, 512, P, None, 0) == 1            # null x
    assert f(P + 1, 0, 512, 4, 512, 0, None, P, 1, 512, P, None, 0) == 2           # misaligned bf16
    assert f(P, 0, 512, 4, 512, 0, P + 4, P, 1, 512, P, None, 0) == 2              # pre_scale not 16-byte aligned
    assert f(P, 0, 70000, 4, 70000, 0, None, P, 1, 70144, P, None, 0) == 3         # K_p too large
    assert f(P, 0, 512, 4, 512, 0, None, P, 1, 512, P, P + 2, 0) == 2        # a_norm misaligned
    assert f(P, 0, 512, 0, 512, 0, None, P, 1, 512, P, None, 0) == 0               # empty: no launch


def test_prepare_weight_rejects_bad_arguments(lib):
    f = lib.convrot_prepare_weight
    P = 1 << 20
    assert f(P, P, P, 4, 0, P, 1, 512, P, None, 0) == 1                      # K <= 0
    assert f(P, P, P, 4, 512, P, 1, 256, P, None, 0) == 1                    # ld_wq < K_p
    assert f(P + 4, P, P, 4, 512, P, 1, 512, P, None, 0) == 2                # w_fp4 not 8-aligned
    assert f(P, P, P, 4, 512, P + 1, 1, 512, P, None, 0) == 2                # f16 codes misaligned
    assert f(P, None, P, 4, 512, P, 1, 512, P, None, 0) == 1                 # null scales
    assert f(P, P, P, 4, 512, P, 1, 512, P, P + 1, 0) == 2             # w_norm misaligned
    assert f(P, P, P, 0, 512, P, 1, 512, P, None, 0) == 0                    # empty


def test_gemm_rejects_bad_arguments(lib):
    f = lib.convrot_gemm
    P = 1 << 20
    ok = dict(a=P, lda=512, sa=P, w=P, ldw=512, sw=P, M=4, N=4, Kp=512, o=P, dt=0, ldo=4)

    def call(**kw):
        d = dict(ok, **kw)
        return f(d["a"], d["lda"], d["sa"], d.get("an"), d["w"], d["ldw"], d["sw"], d.get("wn"), d.get("b"),
                 d["M"], d["N"], d["Kp"], d["o"], d["dt"], d["ldo"], 0)
    assert call(Kp=500) == 1                 # K_p not a multiple of 256
    assert call(Kp=0) == 1
    assert call(lda=256) == 1                # ld < K_p
    assert call(ldo=3) == 1                  # ld_out < N
    assert call(dt=9) == 3
    assert call(a=P + 8) == 2                # TMA base alignment
    assert call(lda=520 + 4) == 2            # TMA pitch alignment
    assert call(a=None) == 1
    assert call(Kp=65536 + 256, lda=70000, ldw=70000) == 3
    assert call(M=0) == 0 and call(N=0) == 0
    assert call(sw=P + 4) == 2               # w_scale read four at a time
    assert call(b=P + 4) == 2                # bias read four at a time
    assert call(an=P + 2, wn=P) == 2         # norm bounds 4-byte aligned
    g = lib.convrot_gemm_i32
    assert g(P, 512, None, P, 512, None, 4, 4, 512, None, 4, 0) == 1
    assert g(P, 512, None, P, 512, None, 4, 4, 512, P + 2, 4, 0) == 2
    assert g(P, 512, P + 1, P, 512, P, 4, 4, 512, P, 4, 0) == 2


def test_binding_fails_loudly_without_library(tmp_path):
    saved = cr._lib
    cr._lib = None
    try:
        with pytest.raises(ImportError):
            cr.load_library(str(tmp_path / "missing.so"))
    finally:
        cr._lib = saved


def test_widen_codes_rejects_bad_arguments(lib):
    f = lib.convrot_widen_codes
    P = 1 << 20
    assert f(P, 64, 4, 40, P, 64, 0) == 1           # cols not a multiple of 16
    assert f(P, 32, 4, 48, P, 64, 0) == 1           # ld_src < cols
    assert f(P + 8, 64, 4, 48, P, 64, 0) == 2       # src not 16-byte aligned
    assert f(P, 64, 4, 48, P, 60, 0) == 2           # ld_dst not a multiple of 8
    assert f(None, 64, 4, 48, P, 64, 0) == 1
    assert f(P, 64, 0, 48, P, 64, 0) == 0           # empty


def test_single_row_tensors_pass_their_width_as_pitch():
    # torch reports stride 0 for a leading dimension of size 1 (e.g. a numpy
    # view with a new axis); the binding passes the row width instead
    import numpy as np
    import torch
    t = torch.from_numpy(np.ascontiguousarray(np.zeros(512)[None, :])).to(torch.float16)
    assert t.stride(0) in (0, 512)
    assert cr._ld(t) == 512
    assert cr._ld(torch.zeros(3, 40)[:, :16]) == 40


def test_int8_probe_rejects_bad_arguments(lib):
    f = lib.convrot_int8_mma_probe
    P = 1 << 20
    assert f(0, 10, P, 0) == 1                      # no blocks
    assert f(4, 0, P, 0) == 1                       # no iterations
    assert f(4, (1 << 22) + 1, P, 0) == 1           # the per-warp sum would overflow int32
    assert f(4, 10, None, 0) == 1
    assert f(4, 10, P + 2, 0) == 2                  # int32 output misaligned


def test_decode_gemm_probe_rejects_bad_arguments(lib):
    f = lib.convrot_decode_gemm_probe
    P = 1 << 20                                     # aligned fake device addresses: no call reaches the GPU
    ok = dict(w=P, sf=P, t=P, s=P, N=256, K=5376, ms=2, pw=16, dump=None, ld=0, unit=0, st=P)

    def call(**kw):
        a = {**ok, **kw}
        return f(a["w"], a["sf"], a["t"], a["s"], a["N"], a["K"], a["ms"], a["pw"], a["dump"], a["ld"],
                 a["unit"], a["st"], None)
    assert call(N=0) == 1
    assert call(K=0) == 1
    assert call(ms=0) == 1
    assert call(pw=4) == 3                          # 8 or 16 producer warps
    assert call(K=65537) == 3                       # K_p beyond the limit
    assert call(w=None) == 1
    assert call(s=None) == 1
    assert call(st=None) == 1
    assert call(w=P + 4) == 2
    assert call(s=P + 2) == 2
    assert call(st=P + 2) == 2
    assert call(dump=P, ld=5120) == 1               # ld_dump below K_p
    assert call(dump=P, ld=5376, unit=4) == 1       # 2 strips x 2 halves: units 0..3
    assert call(dump=P, ld=5376, unit=-1) == 1
    assert call(dump=P + 2, ld=5376) == 2
    assert call(dump=P, ld=5378 + 1) == 2            # odd pitch
