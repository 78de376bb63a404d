"""Pins of the oracle alignment/permutation (CPU only): invariants only."""
import numpy as np
import pytest
import torch

from oracle import moe_ref


def _check(ids, E, bm):
    al = moe_ref.align(ids, E, bm)
    flat = ids.reshape(-1).numpy()
    S = flat.size
    off = al.expert_offsets.numpy()
    srt = al.sorted_slot.numpy()
    inv = al.inv_slot.numpy()
    assert off[0] == 0 and off[-1] == S
    assert (np.diff(off) == np.bincount(flat, minlength=E)).all()
    assert sorted(srt.tolist()) == list(range(S))           # a permutation
    assert (inv[srt] == np.arange(S)).all()                  # inverse
    for e in range(E):
        seg = srt[off[e]:off[e + 1]]
        assert (flat[seg] == e).all()                        # grouped by expert
        assert (np.diff(seg) > 0).all()                      # stable: ascending slot
    tm = al.tile_map.numpy()
    exp_tiles = []
    for e in range(E):
        c = off[e + 1] - off[e]
        exp_tiles += [(e, off[e] + i * bm) for i in range((c + bm - 1) // bm)]
    assert al.num_tiles == len(exp_tiles) == tm.shape[0]
    assert [tuple(r) for r in tm.tolist()] == exp_tiles
    return al


@pytest.mark.parametrize("T,k,E,bm", [(16, 2, 8, 128), (37, 3, 5, 4), (100, 8, 256, 128), (1, 1, 16, 128), (64, 1, 1, 16)])
def test_align_invariants_random(T, k, E, bm):
    g = torch.Generator().manual_seed(T * 7 + k)
    ids = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).to(torch.int32) if T else torch.zeros((0, k), dtype=torch.int32)
    _check(ids, E, bm)


def test_align_skewed_and_empty_experts():
    ids = torch.tensor([[3, 0]] * 40 + [[0, 3]] * 9, dtype=torch.int32)
    al = _check(ids, 6, 8)
    assert al.expert_offsets.tolist() == [0, 49, 49, 49, 98, 98, 98]


def test_align_empty_input():
    al = _check(torch.zeros((0, 2), dtype=torch.int32), 4, 128)
    assert al.num_tiles == 0
