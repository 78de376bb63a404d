"""Pins of the oracle experts and whole-layer composition (CPU only)."""
import numpy as np
import torch
import torch.nn.functional as F

from mixture_experts_layer_tokens_gb300.inputs import CONFIGS, make_inputs, scaled
from oracle import codecs, moe_ref


def _dense(x, w13, w2):
    """Dense SwiGLU MLP written with torch's own silu, bf16 intermediate/out."""
    I = w13.shape[0] // 2
    xd = x.double()
    h = F.silu(xd @ w13[:I].double().T) * (xd @ w13[I:].double().T)
    h = h.to(torch.float32).to(torch.bfloat16).double()
    return (h @ w2.double().T).to(torch.float32).to(torch.bfloat16).double()


def _layer(inp, top_k):
    cfg = inp.cfg
    ids, w = moe_ref.route_softmax_renorm(inp.logits, top_k)
    al = moe_ref.align(ids, cfg.E, 128)
    a1q, sc = moe_ref.prepare(inp.a1, w, False, cfg.quant)
    y = moe_ref.experts(a1q, sc, inp.w13, inp.w13_scale, inp.w2, inp.w2_scale, al, top_k, cfg.quant)
    return moe_ref.finalize(y, w, top_k, False), y, ids


def test_identical_experts_reduce_to_dense_mlp():
    inp = make_inputs(scaled(CONFIGS["tiny"], T=24))
    inp.w13[:] = inp.w13[0]
    inp.w2[:] = inp.w2[0]
    fo, y, _ = _layer(inp, 2)
    dense = _dense(inp.a1, inp.w13[0], inp.w2[0])
    # every slot row is the dense MLP row; the weighted sum of equal rows with sum(w)=1 is that row
    assert torch.equal(y.reshape(24, 2, -1)[:, 0], dense) or (y.reshape(24, 2, -1)[:, 0] - dense).abs().max() < 2e-2
    rel = np.linalg.norm(fo.out - dense.numpy()) / np.linalg.norm(dense.numpy())
    assert rel < 1e-6


def test_one_expert_top1_is_dense_mlp():
    inp = make_inputs(scaled(CONFIGS["tiny"], T=20, E=1, top_k=1))
    fo, y, ids = _layer(inp, 1)
    assert (ids == 0).all()
    dense = _dense(inp.a1, inp.w13[0], inp.w2[0])
    diff = (y - dense).abs()
    assert (diff <= dense.abs() * 2 ** -7 + 1e-6).all()   # at most a bf16 rounding flip of h or y
    assert diff.max() < 0.05 and (diff > 0).float().mean() < 0.02


def test_slot_rows_are_token_major_and_unweighted():
    inp = make_inputs(CONFIGS["tiny"])
    fo, y, ids = _layer(inp, 2)
    for t in (0, 7, 15):
        rows = moe_ref.token_expert_rows(inp.a1, None, inp.w13, None, inp.w2, None, ids, t, "bf16")
        assert torch.equal(rows, y[t * 2:(t + 1) * 2])


def test_weight_on_input_differs_from_weight_on_output():
    cfg = scaled(CONFIGS["llama1"], T=8, H=256, I=256, E=4, shared_I=0)
    inp = make_inputs(cfg)
    ids, w = moe_ref.route_sigmoid_top1(inp.logits)
    al = moe_ref.align(ids, 4, 128)
    a1q, _ = moe_ref.prepare(inp.a1, w, True, "bf16")
    y_in = moe_ref.experts(a1q, None, inp.w13, None, inp.w2, None, al, 1, "bf16")
    out_in = moe_ref.finalize(y_in, w, 1, True).out
    a1q2, _ = moe_ref.prepare(inp.a1, w, False, "bf16")
    y_out = moe_ref.experts(a1q2, None, inp.w13, None, inp.w2, None, al, 1, "bf16")
    out_out = moe_ref.finalize(y_out, w, 1, False).out
    assert np.linalg.norm(out_in - out_out) / np.linalg.norm(out_out) > 0.05
    # finalize ignores the weights when they were applied on the input
    assert np.array_equal(out_in, y_in.numpy())


def test_fp8_experts_with_exact_scales_equal_bf16_on_dequantised_values():
    # power-of-two scales and grid-valued inputs: prepare is exact, GEMM1 is exact in fp64
    cfg = scaled(CONFIGS["tiny"], H=256, I=256, E=2, top_k=1, quant="fp8")
    inp = make_inputs(cfg)
    rng = np.random.default_rng(1)
    codes = rng.integers(0, 256, size=(16, 256)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x30
    codes[:, 0] = 0x7E
    codes[:, 128] = 0x7E
    a1 = torch.from_numpy(codecs.e4m3_decode(codes) * 2.0 ** -6).to(torch.float32).to(torch.bfloat16)
    a1q, s = moe_ref.prepare(a1, None, False, "fp8")
    assert np.array_equal(moe_ref.dequant_fp8_g128(a1q.numpy(), s.numpy()), a1.double().numpy())
    inp.w13_scale[:] = 2.0 ** -9
    W = moe_ref.dequant_weight_block(inp.w13[0].numpy(), inp.w13_scale[0].numpy())
    assert np.array_equal(W, codecs.e4m3_decode(inp.w13[0].numpy()) * 2.0 ** -9)
    # per-block scales land on their own 128x128 block
    sc = np.arange(1, 5, dtype=np.float32).reshape(2, 2)
    Wb = moe_ref.dequant_weight_block(np.full((256, 256), 0x38, np.uint8), sc)
    assert Wb[0, 0] == 1 and Wb[0, 200] == 2 and Wb[200, 0] == 3 and Wb[255, 255] == 4
