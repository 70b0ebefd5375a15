"""The INT8 tensor-rate probe (a measurement aid beside the layer): each warp's
8 chains of mma.sync m16n8k32 on all-ones s8 operands add 32 per iteration."""
import pytest
import torch

from gpu_util import DEV, ensure_built

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


@pytest.mark.parametrize("blocks,iters", [(1, 1), (3, 1000), (300, 4096)])
def test_int8_mma_probe_counts(blocks, iters):
    ensure_built()
    import rotated_w4a8_int8_gb300 as cr
    out = torch.full((blocks * 4,), -1, dtype=torch.int32, device=DEV)
    cr.int8_mma_probe(blocks, iters, out)
    assert torch.equal(out.cpu(), torch.full((blocks * 4,), 8 * 32 * iters, dtype=torch.int32))
