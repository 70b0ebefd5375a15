"""The layer's three calls captured in one CUDA graph.

Every call only enqueues kernels on the given stream and allocates nothing, so
a caller can capture weight preparation, activation quantisation and the GEMM
once and replay them (the pages run the layer as one path per call, ComfyUI
Turing Utils page, node list, the ConvRot loaders' NVFP4 entry).  A replay
must give the eager result bit for bit, also after new inputs are copied into
the captured buffers; the code-norm bounds and the fused SwiGLU take part.
"""
import pytest
import torch

import synth
from gpu_util import DEV, TORCH_DT, ensure_built, storage_to_dev

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

CASES = [
    # (name, workload, tokens, weight rows, code-norm bounds)
    ("qkv_rows", synth.Workload("g_qkv", 1000, 5376, 1024, "bf16", "bf16", False, 0.01, 20.0, 41), True),
    ("swiglu", synth.Workload("g_sw", 700, 2048, 520, "bf16", "fp32", True, 0.0, 1.0, 42), False),
]


class StaticLayer:
    """Device buffers that stay put, so a captured graph can be replayed on new contents."""

    def __init__(self, wl, norms):
        import rotated_w4a8_int8_gb300 as cr
        self.cr, self.wl = cr, wl
        packed, scales, t = synth.make_nvfp4_weight(wl)
        self.x = storage_to_dev(synth.make_activations(wl), wl.x_dtype)
        self.p = torch.from_numpy(packed).to(DEV)
        self.s = torch.from_numpy(scales).to(DEV)
        self.t = torch.tensor([float(t)], dtype=torch.float32, device=DEV)
        Kp = cr.padded_k(wl.K)
        self.wq = torch.empty(wl.N, Kp, dtype=torch.float16, device=DEV)
        self.sw = torch.empty(wl.N, dtype=torch.float32, device=DEV)
        self.aq = torch.empty(wl.M, Kp, dtype=torch.float16, device=DEV)
        self.sa = torch.empty(wl.M, dtype=torch.float32, device=DEV)
        self.nw = torch.empty(wl.N, dtype=torch.float32, device=DEV) if norms else None
        self.na = torch.empty(wl.M, dtype=torch.float32, device=DEV) if norms else None
        self.y = torch.empty(wl.M, wl.N, dtype=TORCH_DT[wl.out_dtype], device=DEV)

    def run(self):
        cr, wl = self.cr, self.wl
        cr.prepare_weight(self.p, self.s, self.t, wl.K, self.wq, self.sw, w_norm=self.nw)
        cr.quant_act(self.x, wl.K, self.aq, self.sa, swiglu=wl.swiglu, a_norm=self.na)
        cr.gemm(self.aq, self.sa, self.wq, self.sw, self.y, a_norm=self.na, w_norm=self.nw)


@pytest.mark.parametrize("name,wl,norms", CASES, ids=[c[0] for c in CASES])
def test_layer_replays_from_a_cuda_graph(name, wl, norms):
    ensure_built()
    import rotated_w4a8_int8_gb300 as cr
    L = StaticLayer(wl, norms)
    L.run()                                             # eager result (and first-call set-up)
    torch.cuda.synchronize()
    y_eager = L.y.clone()

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        L.run()                                         # warm-up on the capturing stream's side
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        L.run()
    L.y.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(L.y, y_eager)

    # new contents in the captured buffers: the replay follows them
    g = torch.Generator(device=DEV).manual_seed(7)
    L.x.copy_((torch.randn(L.x.shape, generator=g, device=DEV) * 2).to(L.x.dtype))
    L.p.copy_(torch.randint(0, 256, L.p.shape, generator=g, device=DEV, dtype=torch.uint8))
    L.s.copy_(torch.randint(0x30, 0x40, L.s.shape, generator=g, device=DEV, dtype=torch.uint8))
    graph.replay()
    torch.cuda.synchronize()
    y_graph = L.y.clone()
    L.run()
    torch.cuda.synchronize()
    assert torch.equal(y_graph, L.y)
    assert not torch.equal(y_graph, y_eager)
    assert cr.device_error() == 0
