"""Pins of the oracle's batched activation format (CPU only).

"Fused MoE Kernel Features", section "Fused MoE Modular All2All backends": a
prepare step outputs "standard" or "batched" activations and the finalize
takes the same format back to standard.  The layout read here: one slab per
expert [E, max_tokens, H] holding the expert's slots in ascending slot order,
with a count per expert.  Pinned by a layout derived by hand, by brute force
over the sort key (expert, slot), and by the standard path (itself pinned
elsewhere): computing in the batched format and reading the rows back must give
the standard path's rows exactly, in every quantisation format.
"""
import numpy as np
import pytest
import torch

from mixture_experts_layer_tokens_gb300.inputs import CONFIGS, make_inputs, scaled
from oracle import moe_ref


def test_positions_of_a_hand_example():
    # tokens 0..2, top-2: slots f = 0..5 choose experts 1,0 | 1,2 | 0,1
    ids = torch.tensor([[1, 0], [1, 2], [0, 1]], dtype=torch.int32)
    e, rank, counts = moe_ref.batched_positions(ids, 3)
    # expert 0 gets slots 1 (token 0) and 4 (token 2); expert 1 slots 0, 2, 5; expert 2 slot 3
    assert counts.tolist() == [2, 3, 1]
    assert e.tolist() == [1, 0, 1, 2, 0, 1]
    assert rank.tolist() == [0, 0, 1, 0, 1, 2]
    a1 = torch.arange(3 * 8, dtype=torch.float32).reshape(3, 8).to(torch.bfloat16)
    q, s, n = moe_ref.prepare_batched(a1, ids, None, False, "bf16", 3, 4)
    assert s is None and n.tolist() == [2, 3, 1]
    assert torch.equal(q[0, :2], a1[[0, 2]]) and torch.equal(q[1, :3], a1[[0, 1, 2]]) and torch.equal(q[2, :1], a1[[1]])
    assert (q[0, 2:] == 0).all() and (q[2, 1:] == 0).all()


def test_positions_match_sorting_by_expert_then_slot():
    g = torch.Generator().manual_seed(4)
    ids = torch.argsort(torch.rand((37, 9), generator=g), dim=1)[:, :3].to(torch.int32)
    e, rank, counts = moe_ref.batched_positions(ids, 9)
    flat = ids.reshape(-1).tolist()
    order = sorted(range(len(flat)), key=lambda f: (flat[f], f))
    assert counts.tolist() == np.bincount(flat, minlength=9).tolist()
    start = np.concatenate([[0], np.cumsum(counts)[:-1]])
    for p, f in enumerate(order):                 # the standard alignment's row p of slot f
        assert e[f] == flat[f] and start[e[f]] + rank[f] == p
    # a bijection onto the counted rows of the slabs
    assert len({(int(a), int(b)) for a, b in zip(e, rank)}) == len(flat)


def test_overflow_is_an_error():
    ids = torch.zeros((5, 1), dtype=torch.int32)
    with pytest.raises(ValueError):
        moe_ref.prepare_batched(torch.zeros((5, 128), dtype=torch.bfloat16), ids, None, False, "bf16", 2, 4)


@pytest.mark.parametrize("quant", ["bf16", "fp8", "fp8_token", "fp8_tensor"])
def test_batched_path_equals_standard_path(quant):
    base = CONFIGS["tiny"] if quant == "bf16" else CONFIGS["deepseek"]
    cfg = scaled(base, T=40, H=256, I=256, E=5, top_k=2, shared_I=0, quant=quant)
    inp = make_inputs(cfg)
    ids, w = moe_ref.route_softmax_renorm(inp.logits, 2)
    al = moe_ref.align(ids, 5, 128)
    a1q, sc = moe_ref.prepare(inp.a1, w, False, quant)
    y_std = moe_ref.experts(a1q, sc, inp.w13, inp.w13_scale, inp.w2, inp.w2_scale, al, 2, quant)
    qb, sb, n = moe_ref.prepare_batched(inp.a1, ids, w, False, quant, 5, 40)
    # every prepared slab row is the standard prepared row of its token, bit for bit
    e, rank, _ = moe_ref.batched_positions(ids, 5)
    for f in range(80):
        assert torch.equal(qb[e[f], rank[f]], a1q[f // 2])
    yb = moe_ref.experts_batched(qb, sb, n, inp.w13, inp.w13_scale, inp.w2, inp.w2_scale, quant)
    assert torch.equal(moe_ref.unbatch(yb, ids), y_std)
    fb = moe_ref.finalize_batched(yb, ids, w, 2, False)
    assert np.array_equal(fb.out, moe_ref.finalize(y_std, w, 2, False).out)
