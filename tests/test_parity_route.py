"""GPU router vs the oracle: ids bit-exact, weights within 2^-20 relative."""
import numpy as np
import pytest
import torch

from mixture_experts_layer_tokens_gb300 import moe
from mixture_experts_layer_tokens_gb300.inputs import CONFIGS, make_logits
from oracle import moe_ref

pytestmark = pytest.mark.gpu


def _check(logits, k, scoring, dev):
    ids, w = moe.moe_route(logits.to(dev), k, scoring)
    torch.cuda.synchronize()
    if scoring == moe.MOE_SCORING_SIGMOID:
        rid, rw = moe_ref.route_sigmoid_top1(logits)
    else:
        rid, rw = moe_ref.route_softmax_renorm(logits, k)
    assert torch.equal(ids.cpu(), rid)
    assert torch.allclose(w.cpu().double(), rw.double(), rtol=2.0 ** -20, atol=0)


@pytest.mark.parametrize("name", ["tiny", "mixtral", "deepseek", "finalize512", "llama512"])
def test_route_configs(cuda_dev, name):
    cfg = CONFIGS[name]
    logits = make_logits(cfg)
    k = cfg.top_k
    scoring = moe.MOE_SCORING_SIGMOID if cfg.scoring == "sigmoid" else moe.MOE_SCORING_SOFTMAX_RENORM
    _check(logits, k, scoring, cuda_dev)


@pytest.mark.parametrize("T,E,k", [(64, 8, 2), (200, 256, 8), (33, 1024, 32), (7, 1, 1), (50, 33, 5), (9, 64, 64 // 2)])
def test_route_ties_go_to_lower_index(cuda_dev, T, E, k):
    g = torch.Generator().manual_seed(T + E + k)
    logits = torch.randint(-3, 4, (T, E), generator=g).float()  # heavy ties
    _check(logits, k, moe.MOE_SCORING_SOFTMAX_RENORM, cuda_dev)
    if k == 1:
        _check(logits, 1, moe.MOE_SCORING_SIGMOID, cuda_dev)


def test_route_signed_zero_and_infinities(cuda_dev):
    # (a row whose chosen logits are all -inf has no softmax: outside the contract)
    logits = torch.tensor([[0.0, -0.0, 1.0, float("-inf")], [-0.0, 0.0, -0.0, 0.0], [float("-inf"), 2.0, 3.0, 1.0]])
    _check(logits, 3, moe.MOE_SCORING_SOFTMAX_RENORM, cuda_dev)


def test_route_k_equals_e_and_empty(cuda_dev):
    g = torch.Generator().manual_seed(11)
    _check(torch.randn((40, 16), generator=g), 16, moe.MOE_SCORING_SOFTMAX_RENORM, cuda_dev)
    ids, w = moe.moe_route(torch.empty((0, 8), device=cuda_dev), 2)
    assert ids.shape == (0, 2)
