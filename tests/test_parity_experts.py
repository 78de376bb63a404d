"""GPU grouped expert GEMMs vs the oracle, fed identical prepared inputs.

Sizes span several M, N and K tiles with ragged tails: experts of 0, 1, <128,
>128 and many-tile row counts, N tiles that run past H, deep K loops.  The
decode-sized bf16 cases (at most 16 slots per expert, K of 32+ blocks, fewer
units than half the SMs) split their K loops across many CTAs and finish each
unit through the fp32 partials (stream-K): one or many valid rows per tile,
units cut into 2 to 20 segments.  The 64-expert cases have at least four units
per CTA and run the round-robin schedule."""
import numpy as np
import pytest
import torch

from mixture_experts_layer_tokens_gb300 import moe
from mixture_experts_layer_tokens_gb300.inputs import CONFIGS, make_inputs, scaled
from oracle import moe_ref
from parity_util import (E4M3_VALUES, check_bf16, check_fp8, check_fp8_intermediate, fp8_row_scales, half_ulp_bf16,
                         to64)

pytestmark = pytest.mark.gpu


def _run(inp, ids, dev, quant, identity=False, act="silu", w13=None, w13_scale=None, stages=False):
    cfg = inp.cfg
    E, k = cfg.E, ids.shape[1]
    T, H = inp.a1.shape
    I = inp.w2.shape[2]
    w13 = inp.w13 if w13 is None else w13
    w13_scale = inp.w13_scale if w13_scale is None else w13_scale
    al = moe.moe_align(ids.to(dev), E)
    a1q, sc = moe.moe_prepare(inp.a1.to(dev), None, k, False, quant)
    d = lambda t: None if t is None else t.to(dev)
    ws = torch.empty(max(moe.workspace_size(T, H, I, E, k, quant), 16), dtype=torch.uint8, device=dev)
    y = moe.moe_experts(a1q, sc, d(w13), d(w13_scale), d(inp.w2), d(inp.w2_scale), al, quant,
                        identity=identity, activation=act, ws=ws)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == moe.MOE_OK
    ral = moe_ref.align(ids, E, 128)
    rq, rs = moe_ref.prepare(inp.a1, None, False, quant)
    assert torch.equal(a1q.cpu(), rq)
    yref = moe_ref.experts(rq, rs, w13, w13_scale, inp.w2, inp.w2_scale, ral, k, quant, act)
    if stages:
        _fp8_stages(inp, ral, rq, rs, w13, w13_scale, quant, act, ws, y, f"experts {quant} {act}")
    return y, yref


def _fp8_stages(inp, ral, rq, rs, w13, w13_scale, quant, act, ws, y, what):
    """The fp8 experts stage by stage: the GPU's intermediate (codes and scales left in
    the workspace) against the oracle's quantisation of its own h, then the GPU's
    expert rows against the oracle's second GEMM applied to the GPU's intermediate, at
    the bf16 bound (both sides then hold the same h)."""
    T, H = inp.a1.shape
    E, k, I = w13.shape[0], int(ral.sorted_slot.numel()) // max(T, 1), inp.w2.shape[2]
    h_gpu, hs_gpu = moe.experts_intermediate(ws, T, H, I, E, k, quant)
    offs, order = ral.expert_offsets.numpy(), ral.sorted_slot.numpy()
    S = int(offs[-1])
    codes = h_gpu[:S].cpu().numpy()
    scales = fp8_row_scales(hs_gpu, quant, np.arange(S), I // 128)
    h_ref = np.zeros((S, I))
    for e in range(E):
        p0, p1 = int(offs[e]), int(offs[e + 1])
        if p0 < p1:
            A = moe_ref._act64(rq, rs, order[p0:p1] // k, quant)
            h_ref[p0:p1] = moe_ref.activation(A @ moe_ref._weights64(w13, w13_scale, e, quant).T, act).numpy()
    check_fp8_intermediate(codes, scales, h_ref, quant, what)
    h_deq = E4M3_VALUES[codes] * np.repeat(scales, 128, axis=1)
    y2 = torch.zeros((S, H), dtype=torch.float64)
    for e in range(E):
        p0, p1 = int(offs[e]), int(offs[e + 1])
        if p0 < p1:
            y2[torch.from_numpy(order[p0:p1].astype(np.int64))] = moe_ref._expert_out(
                h_deq[p0:p1], moe_ref._weights64(inp.w2, inp.w2_scale, e, quant))
    check_bf16(y, y2, what + ": second GEMM on the GPU's intermediate", slack=_stored_pair_slack(y2))


def _stored_pair_slack(yref):
    """Both sides store y (and h) as bf16, so the oracle's stored value and the GPU's
    can be neighbouring bf16 numbers: one ulp in all, half from each rounding."""
    return half_ulp_bf16(to64(yref))


def _ids(T, k, E, seed, skew=False):
    g = torch.Generator().manual_seed(seed)
    if skew:
        p = torch.tensor([0.5 ** i for i in range(E)])
        p[E // 2] = 0  # one empty expert
        ids = torch.stack([torch.multinomial(p, k, replacement=False, generator=g) for _ in range(T)])
    else:
        ids = torch.argsort(torch.rand((T, E), generator=g), dim=1)[:, :k]
    return ids.to(torch.int32).contiguous()


@pytest.mark.parametrize("T,H,I,E,k,skew", [
    (16, 256, 512, 8, 2, False),      # the tiny layer
    (300, 512, 384, 4, 2, False),     # 2 M tiles per expert, ragged tails
    (700, 384, 256, 6, 2, True),      # skewed: a 5-tile expert, an empty one; GEMM2 N tile past H
    (130, 2048, 256, 3, 1, False),    # deep K (32 stages)
    (1, 256, 128, 8, 2, False),       # single token
    (256, 256, 2048, 64, 4, False),   # 1024 units >= 4 per CTA: round-robin schedule
    (4, 2048, 2048, 16, 1, False),    # stream-K in both GEMMs, single-row tiles
    (1, 4096, 1024, 8, 1, False),     # stream-K GEMM1: 8 units cut into ~19 segments each
    (16, 2048, 4096, 1, 1, False),    # stream-K, 16 valid rows in one tile (the shared-expert shape)
    (12, 2048, 2048, 8, 2, True),     # stream-K with skewed routing: one expert holds most rows
    # two-tile units (on 152 SMs): 96 GEMM1 / 128 GEMM2 units of two 128-row tiles fill one
    # wave, experts of ~128 rows give groups of one and of two tiles
    (512, 4096, 1536, 8, 2, False),
    # one dense expert of 16 tiles: 160 two-tile GEMM1 units (more than a wave: the dense
    # expert's rule), 80 two-tile GEMM2 units (one wave)
    (2048, 2560, 2560, 1, 1, False),
])
def test_experts_bf16(cuda_dev, T, H, I, E, k, skew):
    inp = make_inputs(scaled(CONFIGS["tiny"], T=T, H=H, I=I, E=E, top_k=k))
    y, yref = _run(inp, _ids(T, k, E, T + H, skew), cuda_dev, "bf16")
    check_bf16(y, yref, "experts bf16", slack=_stored_pair_slack(yref))


@pytest.mark.parametrize("T,H,I,E,k,skew", [
    (16, 256, 256, 8, 2, False),
    (300, 512, 384, 4, 2, False),
    (500, 384, 256, 6, 2, True),
    (100, 1024, 512, 16, 4, False),
    (256, 256, 2048, 64, 4, False),   # round-robin schedule
])
def test_experts_fp8(cuda_dev, T, H, I, E, k, skew):
    inp = make_inputs(scaled(CONFIGS["deepseek"], T=T, H=H, I=I, E=E, top_k=k, shared_I=0))
    y, yref = _run(inp, _ids(T, k, E, T + I, skew), cuda_dev, "fp8", stages=True)
    rel, _ = check_fp8(y, yref, "experts fp8")
    print(f"experts fp8 T{T} H{H} I{I} E{E} k{k}: relative Frobenius vs the oracle {rel:.2e} (bound 3e-2)")


def test_experts_identity_permutation(cuda_dev):
    # one expert, top-1, NULL sorted_slot: the shared-expert call
    inp = make_inputs(scaled(CONFIGS["tiny"], T=200, H=512, I=256, E=1, top_k=1))
    ids = torch.zeros((200, 1), dtype=torch.int32)
    y, yref = _run(inp, ids, cuda_dev, "bf16", identity=True)
    check_bf16(y, yref, "identity", slack=_stored_pair_slack(yref))


@pytest.mark.parametrize("quant,identity", [("fp8", False), ("bf16", False), ("bf16", True)])
def test_experts_reused_dirty_workspace(cuda_dev, quant, identity):
    """Units dealt round-robin are taken from counters in the workspace; every call clears
    them (in its gather or plan launch, or a memset for the identity case with neither), so
    a workspace that starts as garbage and serves call after call gives the same bits, and
    those agree with the oracle."""
    E, k = (1, 1) if identity else (8, 2)
    base = CONFIGS["deepseek"] if quant == "fp8" else CONFIGS["tiny"]
    inp = make_inputs(scaled(base, T=600, H=512, I=384, E=E, top_k=k, shared_I=0))
    ids = torch.zeros((600, 1), dtype=torch.int32) if identity else _ids(600, k, E, 5)
    T, H, I = 600, 512, 384
    al = moe.moe_align(ids.to(cuda_dev), E)
    a1q, sc = moe.moe_prepare(inp.a1.to(cuda_dev), None, k, False, quant)
    d = lambda t: None if t is None else t.to(cuda_dev)
    ws = torch.full((max(moe.workspace_size(T, H, I, E, k, quant), 16),), 0xFF, dtype=torch.uint8, device=cuda_dev)
    ys = [moe.moe_experts(a1q, sc, d(inp.w13), d(inp.w13_scale), d(inp.w2), d(inp.w2_scale), al, quant,
                          identity=identity, ws=ws).clone() for _ in range(3)]
    torch.cuda.synchronize()
    assert moe.moe_device_status() == moe.MOE_OK
    assert torch.equal(ys[0], ys[1]) and torch.equal(ys[1], ys[2])
    rq, rs = moe_ref.prepare(inp.a1, None, False, quant)
    yref = moe_ref.experts(rq, rs, inp.w13, inp.w13_scale, inp.w2, inp.w2_scale, moe_ref.align(ids, E, 128), k, quant,
                           "silu")
    if quant == "bf16":
        check_bf16(ys[0], yref, "reused workspace", slack=_stored_pair_slack(yref))
    else:
        check_fp8(ys[0], yref, "reused workspace")


def test_experts_twice_same_bits(cuda_dev):
    inp = make_inputs(scaled(CONFIGS["tiny"], T=300, H=512, I=384, E=4))
    ids = _ids(300, 2, 4, 3)
    y1, _ = _run(inp, ids, cuda_dev, "bf16")
    y2, _ = _run(inp, ids, cuda_dev, "bf16")
    assert torch.equal(y1, y2)


@pytest.mark.parametrize("T,H,I,E,k,quant,act", [
    (300, 512, 384, 4, 2, "bf16", "gelu"),
    (300, 512, 384, 4, 2, "bf16", "gelu_tanh"),
    (300, 512, 384, 4, 2, "bf16", "swigluoai"),
    (300, 512, 384, 4, 2, "bf16", "silu_no_mul"),   # 384 gate rows: N tiles of 256 and 128
    (300, 512, 384, 4, 2, "bf16", "gelu_no_mul"),
    (4, 2048, 2048, 16, 1, "bf16", "swigluoai"),     # stream-K in both GEMMs
    (4, 2048, 2048, 16, 1, "bf16", "gelu_no_mul"),   # stream-K, gate-only units
    (256, 256, 2048, 64, 4, "bf16", "silu_no_mul"),  # round-robin schedule
    (300, 512, 384, 4, 2, "fp8", "gelu"),
    (300, 512, 384, 4, 2, "fp8", "swigluoai"),
    (300, 512, 384, 4, 2, "fp8", "silu_no_mul"),    # three G(128) groups of h, the last alone in its tile
    (100, 1024, 512, 16, 4, "fp8", "gelu_no_mul"),
    # per-token ("A") and per-tensor ("T") activation scales: h stored bf16, then quantised
    (300, 512, 384, 4, 2, "fp8_token", "silu"),
    (300, 512, 384, 4, 2, "fp8_tensor", "silu"),
    (100, 1024, 512, 16, 4, "fp8_token", "gelu_no_mul"),
    (100, 1024, 512, 16, 4, "fp8_tensor", "swigluoai"),
    (256, 256, 2048, 64, 4, "fp8_token", "silu"),    # round-robin schedule
    (500, 384, 256, 6, 2, "fp8_tensor", "silu_no_mul"),
])
def test_experts_activations(cuda_dev, T, H, I, E, k, quant, act):
    base = CONFIGS["deepseek"] if quant != "bf16" else CONFIGS["tiny"]
    inp = make_inputs(scaled(base, T=T, H=H, I=I, E=E, top_k=k, shared_I=0, quant=quant))
    w13, w13_scale = inp.w13, inp.w13_scale
    if act == "swigluoai" and quant == "bf16":
        # gate and up values of a few units, so that both clamps at +-7 are reached
        w13 = (w13.float() * 4).to(torch.bfloat16)
    if act.endswith("_no_mul"):
        w13 = w13[:, :I].contiguous()
        w13_scale = None if w13_scale is None else w13_scale[:, :I // 128].contiguous()
    y, yref = _run(inp, _ids(T, k, E, T + I + 7), cuda_dev, quant, act=act, w13=w13, w13_scale=w13_scale,
                   stages=quant != "bf16")
    if quant != "bf16":
        rel, _ = check_fp8(y, yref, f"experts {quant} {act}")
        print(f"experts {quant} {act}: relative Frobenius vs the oracle {rel:.2e} (bound 3e-2)")
    else:
        check_bf16(y, yref, f"experts bf16 {act}", slack=_stored_pair_slack(yref))


def test_experts_act_silu_is_moe_experts(cuda_dev):
    # moe_experts is moe_experts_act with MOE_ACT_SILU: the same bits
    inp = make_inputs(scaled(CONFIGS["tiny"], T=64, H=256, I=256, E=4, top_k=2))
    ids = _ids(64, 2, 4, 99).to(cuda_dev)
    al = moe.moe_align(ids, 4)
    a1q, sc = moe.moe_prepare(inp.a1.to(cuda_dev), None, 2, False, "bf16")
    w13, w2 = inp.w13.to(cuda_dev), inp.w2.to(cuda_dev)
    y_act = moe.moe_experts(a1q, None, w13, None, w2, None, al, "bf16", activation="silu")
    out = torch.empty_like(y_act)
    ws = torch.empty(moe.workspace_size(64, 256, 256, 4, 2, "bf16"), dtype=torch.uint8, device=cuda_dev)
    import ctypes
    st = moe.lib().moe_experts(a1q.data_ptr(), None, w13.data_ptr(), None, w2.data_ptr(), None,
                               al.expert_offsets.data_ptr(), al.sorted_slot.data_ptr(), al.tile_map.data_ptr(),
                               al.num_tiles.data_ptr(), 64, 256, 256, 4, 2, ctypes.byref(moe.QC_BF16),
                               out.data_ptr(), ws.data_ptr(), ws.numel(), None)
    torch.cuda.synchronize()
    assert st == moe.MOE_OK
    assert torch.equal(out, y_act)



@pytest.mark.parametrize("T,H,I,E,k", [
    (1, 2048, 2048, 16, 1),    # decode: both problems' units split across CTAs (stream-K)
    (8, 2048, 2048, 16, 1),
    (200, 512, 384, 6, 2),     # round-robin: routed tiles and the shared expert's tiles side by side
])
def test_experts_multi_routed_and_shared(cuda_dev, T, H, I, E, k):
    # the routed experts and a shared expert (E = 1, identity rows) in the same launches
    inp = make_inputs(scaled(CONFIGS["llama8"], T=T, H=H, I=I, E=E, top_k=k, shared_I=I, scoring="softmax",
                             weight_on_input=False))
    ids = _ids(T, k, E, T + H + 11)
    d = lambda t: t.to(cuda_dev)
    al = moe.moe_align(d(ids), E)
    al_s = moe.moe_align(torch.zeros((T, 1), dtype=torch.int32, device=cuda_dev), 1)
    a1 = d(inp.a1)
    y = torch.empty((T * k, H), dtype=torch.bfloat16, device=cuda_dev)
    ysh = torch.empty((T, H), dtype=torch.bfloat16, device=cuda_dev)
    probs = [moe.experts_problem(a1, None, d(inp.w13), None, d(inp.w2), None, al, y),
             moe.experts_problem(a1, None, d(inp.shared_w13), None, d(inp.shared_w2), None, al_s, ysh, identity=True)]
    ws = torch.empty(moe.workspace_size_multi(probs, H, "bf16"), dtype=torch.uint8, device=cuda_dev)
    moe.moe_experts_multi(probs, H, "bf16", ws)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == moe.MOE_OK
    yref = moe_ref.experts(inp.a1, None, inp.w13, None, inp.w2, None, moe_ref.align(ids, E, 128), k, "bf16")
    shref = moe_ref.dense_mlp(inp.a1, inp.shared_w13[0], inp.shared_w2[0])
    check_bf16(y, yref, "multi: routed", slack=_stored_pair_slack(yref))
    check_bf16(ysh, shref, "multi: shared", slack=_stored_pair_slack(shref))
