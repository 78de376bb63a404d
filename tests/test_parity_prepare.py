"""GPU prepare vs the oracle: bf16 products and fp8 codes/scales bit-exact."""
import numpy as np
import pytest
import torch

from mixture_experts_layer_tokens_gb300 import moe
from mixture_experts_layer_tokens_gb300.inputs import CONFIGS, make_inputs, scaled
from oracle import moe_ref

pytestmark = pytest.mark.gpu


def _a1(T, H, seed, wide=False):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((T, H), generator=g)
    if wide:  # magnitudes from 2^-24 to 2^20 so E4M3 subnormals and saturation edges appear
        x = x * torch.exp2(torch.randint(-24, 21, (T, H), generator=g).float())
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("quant,won", [("fp8", False), ("fp8", True), ("bf16", True), ("fp8_token", False),
                                       ("fp8_token", True), ("fp8_tensor", False), ("fp8_tensor", True)])
@pytest.mark.parametrize("T,H", [(1, 128), (37, 512), (4096, 7168), (64, 5120)])
def test_prepare_bit_exact(cuda_dev, quant, won, T, H):
    a1 = _a1(T, H, T + H)
    g = torch.Generator().manual_seed(5)
    w = torch.rand((T, 1), generator=g) if won else torch.rand((T, 8), generator=g)
    k = w.shape[1]
    q, s = moe.moe_prepare(a1.to(cuda_dev), w.to(cuda_dev), k, won, quant)
    torch.cuda.synchronize()
    rq, rs = moe_ref.prepare(a1, w, won, quant)
    assert torch.equal(q.cpu(), rq)
    if quant != "bf16":
        assert torch.equal(s.cpu(), rs)


def test_prepare_fp8_edge_groups(cuda_dev):
    a1 = _a1(8, 1024, 3, wide=True)
    a1[0, :128] = 0                     # all-zero group
    a1[1, 128:256] = -0.0
    a1[2, :128] = 1e-30                 # tiny constant group
    a1[3, 256:384] = 3.0e38             # near bf16 max
    q, s = moe.moe_prepare(a1.to(cuda_dev), None, 1, False, "fp8")
    torch.cuda.synchronize()
    rq, rs = moe_ref.prepare(a1, None, False, "fp8")
    assert torch.equal(s.cpu(), rs)
    assert torch.equal(q.cpu(), rq)


def test_prepare_bf16_passthrough_and_copy(cuda_dev):
    a1 = _a1(16, 256, 1).to(cuda_dev)
    q, _ = moe.moe_prepare(a1, None, 2, False, "bf16", a1q=a1)
    assert q.data_ptr() == a1.data_ptr()
    q2, _ = moe.moe_prepare(a1, None, 2, False, "bf16")
    torch.cuda.synchronize()
    assert torch.equal(q2, a1) and q2.data_ptr() != a1.data_ptr()
