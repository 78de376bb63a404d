"""GPU align/permute vs the oracle: every output bit-exact."""
import pytest
import torch

from mixture_experts_layer_tokens_gb300 import moe
from mixture_experts_layer_tokens_gb300.inputs import CONFIGS, make_logits
from oracle import moe_ref

pytestmark = pytest.mark.gpu


def _check(ids, E, dev, block_m=128):
    al = moe.moe_align(ids.to(dev), E, block_m)
    torch.cuda.synchronize()
    ref = moe_ref.align(ids, E, block_m)
    S = ids.numel()
    assert torch.equal(al.expert_offsets.cpu(), ref.expert_offsets)
    assert torch.equal(al.sorted_slot.cpu()[:S], ref.sorted_slot)
    assert torch.equal(al.inv_slot.cpu()[:S], ref.inv_slot)
    n = int(al.num_tiles.item())
    assert n == ref.num_tiles
    assert torch.equal(al.tile_map.cpu()[:n], ref.tile_map)
    assert moe.moe_device_status() == moe.MOE_OK


def _random_ids(T, k, E, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.argsort(torch.rand((T, E), generator=g), dim=1)[:, :k].to(torch.int32).contiguous()


@pytest.mark.parametrize("name", ["tiny", "mixtral", "deepseek", "llama512"])
def test_align_configs(cuda_dev, name):
    cfg = CONFIGS[name]
    ids, _ = moe_ref.route_softmax_renorm(make_logits(cfg), cfg.top_k) if cfg.scoring == "softmax" else \
        moe_ref.route_sigmoid_top1(make_logits(cfg))
    _check(ids, cfg.E, cuda_dev)


@pytest.mark.parametrize("T,k,E,bm", [(1, 1, 1, 128), (3, 2, 4, 1), (999, 3, 7, 128), (5000, 8, 1024, 128),
                                      (2049, 1, 16, 64), (16384, 8, 256, 128),
                                      # one-block path (at most 2048 slots): 1024 experts, exactly 2048 slots
                                      (700, 2, 1024, 128), (1024, 2, 64, 16)])
def test_align_random(cuda_dev, T, k, E, bm):
    _check(_random_ids(T, k, E, T + E), E, cuda_dev, bm)


def test_align_skewed_and_empty_experts(cuda_dev):
    ids = torch.zeros((6000, 2), dtype=torch.int32)
    ids[:, 1] = 5
    ids[::7, 0] = 3
    _check(ids, 8, cuda_dev)                         # experts 1, 2, 4, 6, 7 empty; expert 0 has many tiles
    _check(torch.zeros((0, 2), dtype=torch.int32), 8, cuda_dev)


def test_align_out_of_range_ids_are_reported_not_faulted(cuda_dev):
    ids = _random_ids(100, 2, 8, 1)
    ids[3, 1] = 8
    al = moe.moe_align(ids.to(cuda_dev), 8)
    assert moe.moe_device_status(clear=True) == moe.MOE_ERR_INVALID_ARG
    assert int(al.expert_offsets[-1]) == 199
    assert moe.moe_device_status() == moe.MOE_OK
