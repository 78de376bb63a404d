"""Pins of the oracle router (CPU only)."""
import itertools
import os

import numpy as np
import torch

from mixture_experts_layer_tokens_gb300.inputs import CONFIGS, make_inputs
from oracle import moe_ref

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_route_brute_force_tiny():
    inp = make_inputs(CONFIGS["tiny"])
    L = inp.logits.double().numpy()
    ids, w = moe_ref.route_softmax_renorm(inp.logits, 2)
    T, E = L.shape
    for t in range(T):
        key = lambda i: (L[t, i], -i)
        winners = [S for S in itertools.combinations(range(E), 2)
                   if min(key(i) for i in S) > max(key(i) for i in range(E) if i not in S)]
        assert len(winners) == 1
        assert set(ids[t].tolist()) == set(winners[0])
        assert key(int(ids[t, 0])) > key(int(ids[t, 1]))  # slot 0 holds the larger logit


def test_route_weights_equal_renormalised_full_softmax():
    g = torch.Generator().manual_seed(3)
    logits = torch.randn((64, 32), generator=g)
    for k in (1, 2, 5, 8):
        ids, w = moe_ref.route_softmax_renorm(logits, k)
        p = torch.softmax(logits.double(), dim=1)
        sel = torch.gather(p, 1, ids.long())
        ref = sel / sel.sum(1, keepdim=True)
        assert torch.allclose(w.double(), ref, rtol=2 ** -23, atol=0)
        assert (w.double().sum(1) - 1).abs().max() <= k * 2 ** -24


def test_route_k_equals_e_is_full_softmax():
    g = torch.Generator().manual_seed(4)
    logits = torch.randn((16, 8), generator=g)
    ids, w = moe_ref.route_softmax_renorm(logits, 8)
    p = torch.softmax(logits.double(), dim=1)
    srt, order = torch.sort(p, dim=1, descending=True, stable=True)
    assert torch.equal(ids.long(), order)
    assert torch.allclose(w.double(), srt, rtol=2 ** -23, atol=0)


def test_route_golden_ties():
    for line in open(os.path.join(GOLD, "route_ties.txt")):
        if line.startswith("#") or not line.strip():
            continue
        head, lg, eid, ew = [s.strip() for s in line.split("|")]
        kind, k = head.split()
        logits = torch.tensor([[float(v) for v in lg.split()]], dtype=torch.float32)
        if kind == "softmax":
            ids, w = moe_ref.route_softmax_renorm(logits, int(k))
        else:
            ids, w = moe_ref.route_sigmoid_top1(logits)
        assert ids[0].tolist() == [int(v) for v in eid.split()]
        assert np.allclose(w[0].double().numpy(), [float(v) for v in ew.split()], rtol=1e-7, atol=0)


def test_sigmoid_top1_is_sigmoid_of_argmax():
    g = torch.Generator().manual_seed(5)
    logits = torch.randn((50, 16), generator=g)
    ids, w = moe_ref.route_sigmoid_top1(logits)
    assert torch.equal(ids[:, 0].long(), torch.argmax(logits, dim=1))
    ref = torch.sigmoid(logits.double().max(1).values)
    assert torch.allclose(w[:, 0].double(), ref, rtol=2 ** -23, atol=0)
