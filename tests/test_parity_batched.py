"""The batched activation format on the GPU against the oracle and the standard path.

Layout (the reading stated in include/moe.h and oracle.moe_ref): one slab per
expert [E, max_tokens, H] holding the expert's slots in ascending slot order
and a count per expert.  prepare is bit-exact on every counted row; the experts
match the oracle's batched experts at the bf16 / fp8 bounds; and the whole
batched step (prepare -> experts -> finalize) gives exactly the standard
step's output, since every expert row is the same computation in both layouts."""
import numpy as np
import pytest
import torch

from mixture_experts_layer_tokens_gb300 import moe
from mixture_experts_layer_tokens_gb300.inputs import CONFIGS, make_inputs, scaled
from oracle import moe_ref
from parity_util import check_bf16, check_fp8, half_ulp_bf16

pytestmark = pytest.mark.gpu


def _setup(quant, T, H, I, E, k, seed=0, act="silu"):
    base = CONFIGS["tiny"] if quant == "bf16" else CONFIGS["deepseek"]
    cfg = scaled(base, T=T, H=H, I=I, E=E, top_k=k, shared_I=0, quant=quant, activation=act)
    inp = make_inputs(cfg, seed=seed)
    ids, w = moe_ref.route_softmax_renorm(inp.logits, k)
    return cfg, inp, ids, w


@pytest.mark.parametrize("quant", ["bf16", "fp8", "fp8_token", "fp8_tensor"])
def test_prepare_batched_bit_exact(cuda_dev, quant):
    cfg, inp, ids, w = _setup(quant, 300, 512, 256, 6, 2)
    al = moe.moe_align(ids.to(cuda_dev), 6)
    M = 160
    qb, sb, n = moe.moe_prepare_batched(inp.a1.to(cuda_dev), w.to(cuda_dev), al, 6, M, False, quant)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == moe.MOE_OK
    rq, rs, rn = moe_ref.prepare_batched(inp.a1, ids, w, False, quant, 6, M)
    assert torch.equal(n.cpu(), rn)
    for e in range(6):
        c = int(rn[e])
        assert torch.equal(qb[e, :c].cpu(), rq[e, :c])
        if quant in ("fp8", "fp8_token"):
            assert torch.equal(sb[e, :c].cpu(), rs[e, :c])
    if quant == "fp8_tensor":
        assert torch.equal(sb.cpu(), rs)


def test_prepare_batched_weight_on_input(cuda_dev):
    cfg = scaled(CONFIGS["llama8"], T=40, H=256, I=256, E=4, shared_I=0)
    inp = make_inputs(cfg)
    ids, w = moe_ref.route_sigmoid_top1(inp.logits)
    al = moe.moe_align(ids.to(cuda_dev), 4)
    qb, _, n = moe.moe_prepare_batched(inp.a1.to(cuda_dev), w.to(cuda_dev), al, 4, 40, True, "bf16")
    torch.cuda.synchronize()
    rq, _, rn = moe_ref.prepare_batched(inp.a1, ids, w, True, "bf16", 4, 40)
    assert torch.equal(n.cpu(), rn)
    for e in range(4):
        assert torch.equal(qb[e, :int(rn[e])].cpu(), rq[e, :int(rn[e])])


def test_prepare_batched_overflow_is_reported_not_written(cuda_dev):
    # every token on expert 0: 50 slots into slabs of 32 rows
    T, H = 50, 256
    a1 = torch.randn((T, H)).to(torch.bfloat16).to(cuda_dev)
    ids = torch.zeros((T, 1), dtype=torch.int32, device=cuda_dev)
    al = moe.moe_align(ids, 2)
    guard = torch.full((2, 33, H), -3.0, dtype=torch.bfloat16, device=cuda_dev)  # one row past slab 1
    qb = guard[:, :32]
    moe.moe_device_status(clear=True)
    qc = moe.QUANT_CONFIGS["bf16"]
    counts = torch.empty((2,), dtype=torch.int32, device=cuda_dev)
    slab = torch.empty((2, 32, H), dtype=torch.bfloat16, device=cuda_dev)
    import ctypes
    st = moe.lib().moe_prepare_batched(a1.data_ptr(), None, al.expert_offsets.data_ptr(), al.sorted_slot.data_ptr(),
                                       T, H, 1, 2, 32, 0, ctypes.byref(qc), slab.data_ptr(), None, counts.data_ptr(),
                                       None, 0, None)
    assert st == moe.MOE_OK
    assert moe.moe_device_status(clear=True) == moe.MOE_ERR_INVALID_ARG
    assert counts.tolist() == [32, 0]
    assert torch.equal(slab[0], a1[:32])
    assert moe.moe_device_status(clear=False) == moe.MOE_OK


@pytest.mark.parametrize("quant,act,T,H,I,E,k", [
    ("bf16", "silu", 300, 512, 384, 6, 2),
    ("bf16", "gelu_no_mul", 200, 256, 256, 4, 2),
    ("fp8", "silu", 300, 512, 384, 6, 2),
    ("fp8", "swigluoai", 100, 1024, 512, 16, 4),
    ("fp8_token", "silu", 300, 512, 384, 6, 2),
    ("fp8_tensor", "silu", 300, 512, 384, 6, 2),
])
def test_experts_batched(cuda_dev, quant, act, T, H, I, E, k):
    cfg, inp, ids, w = _setup(quant, T, H, I, E, k, seed=T + E, act=act)
    w13, w13_scale = inp.w13, inp.w13_scale
    al = moe.moe_align(ids.to(cuda_dev), E)
    M = int(torch.bincount(ids.reshape(-1).long(), minlength=E).max()) + 5
    qb, sb, n = moe.moe_prepare_batched(inp.a1.to(cuda_dev), w.to(cuda_dev), al, E, M, False, quant)
    d = lambda t: None if t is None else t.to(cuda_dev)
    yb = moe.moe_experts_batched(qb, sb, d(w13), d(w13_scale), d(inp.w2), d(inp.w2_scale), n, quant, activation=act)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == moe.MOE_OK
    rq, rs, rn = moe_ref.prepare_batched(inp.a1, ids, w, False, quant, E, M)
    ref = moe_ref.experts_batched(rq, rs, rn, w13, w13_scale, inp.w2, inp.w2_scale, quant, act)
    counted = torch.cat([yb[e, :int(rn[e])].double().cpu() for e in range(E)])
    counted_ref = torch.cat([ref[e, :int(rn[e])] for e in range(E)])
    if quant == "bf16":
        check_bf16(counted, counted_ref, f"batched experts {quant} {act}", slack=half_ulp_bf16(counted_ref.numpy()))
    else:
        check_fp8(counted, counted_ref, f"batched experts {quant} {act}")


@pytest.mark.parametrize("quant", ["bf16", "fp8", "fp8_tensor"])
def test_batched_step_equals_standard_step(cuda_dev, quant):
    """route -> align -> prepare -> experts -> finalize in both formats: every expert row is
    the same computation, so the outputs agree bit for bit."""
    cfg, inp, ids, w = _setup(quant, 256, 512, 256, 16, 4, seed=3)
    d = lambda t: None if t is None else t.to(cuda_dev)
    ids_d, w_d = ids.to(cuda_dev), w.to(cuda_dev)
    al = moe.moe_align(ids_d, 16)
    a1q, sc = moe.moe_prepare(d(inp.a1), w_d, 4, False, quant)
    y = moe.moe_experts(a1q, sc, d(inp.w13), d(inp.w13_scale), d(inp.w2), d(inp.w2_scale), al, quant)
    out_std, _ = moe.moe_finalize(y, w_d, 4, False)
    M = 96
    qb, sb, n = moe.moe_prepare_batched(d(inp.a1), w_d, al, 16, M, False, quant)
    yb = moe.moe_experts_batched(qb, sb, d(inp.w13), d(inp.w13_scale), d(inp.w2), d(inp.w2_scale), n, quant)
    out_b = moe.moe_finalize_batched(yb, w_d, ids_d, al, False)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == moe.MOE_OK
    assert torch.equal(out_b, out_std)
    # and the batched finalize is the oracle's finalize of the rows it reads
    fo = moe_ref.finalize_batched(yb.cpu(), ids, w, 4, False)
    check_bf16(out_b, fo.out, "batched finalize", slack=0.0)
