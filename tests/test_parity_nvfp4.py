"""GPU NVFP4 prepare and grouped experts vs the oracle.

prepare: bit-exact scale codes and values of the codes (+0 and -0 both decode to
0).  experts: the GPU-prepared codes (checked equal to the oracle's first) feed
both sides; shapes span several M, N and K tiles with ragged tails, empty
experts, a single token, the round-robin schedule (>= 4 units per CTA) and the
decode-sized stream-K schedule (units split across CTAs), the gated and the
gate-only activations and the identity permutation."""
import numpy as np
import pytest
import torch

from mixture_experts_layer_tokens_gb300 import moe
from mixture_experts_layer_tokens_gb300.inputs import CONFIGS, NVFP4_A1_GSCALE, NVFP4_H_GSCALE, make_inputs, scaled
from oracle import codecs, moe_ref
from parity_util import check_bf16, check_nvfp4, half_ulp_bf16, ulp_bf16

pytestmark = pytest.mark.gpu


def _ids(T, k, E, seed, skew=False):
    g = torch.Generator().manual_seed(seed)
    if skew:
        p = torch.tensor([0.5 ** i for i in range(E)])
        p[E // 2] = 0  # one empty expert
        ids = torch.stack([torch.multinomial(p, k, replacement=False, generator=g) for _ in range(T)])
    else:
        ids = torch.argsort(torch.rand((T, E), generator=g), dim=1)[:, :k]
    return ids.to(torch.int32).contiguous()


def _same_codes(gpu_q, gpu_sf, ref_q, ref_sf):
    assert torch.equal(gpu_sf.cpu(), ref_sf), "block-scale codes differ"
    lo = lambda q: codecs.e2m1_decode(q.numpy() & 15)
    hi = lambda q: codecs.e2m1_decode(q.numpy() >> 4)
    g = gpu_q.cpu()
    assert np.array_equal(lo(g), lo(ref_q)) and np.array_equal(hi(g), hi(ref_q)), "E2M1 values differ"


@pytest.mark.parametrize("T,H,weight", [(300, 512, False), (5, 7168, True), (1, 256, False), (0, 512, False)])
def test_prepare_nvfp4(cuda_dev, T, H, weight):
    cfg = scaled(CONFIGS["llama1"] if weight else CONFIGS["tiny"], T=T, H=H, I=256, E=4, shared_I=0, quant="nvfp4")
    inp = make_inputs(cfg)
    w = torch.rand((T, 1), generator=torch.Generator().manual_seed(T)) if weight else None
    q, sf = moe.moe_prepare_nvfp4(inp.a1.to(cuda_dev), None if w is None else w.to(cuda_dev), 1, weight,
                                  NVFP4_A1_GSCALE)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == moe.MOE_OK
    rq, rsf = moe_ref.prepare_nvfp4(inp.a1, w, weight, NVFP4_A1_GSCALE)
    _same_codes(q, sf, rq, rsf)


def _run(T, H, I, E, k, ids, dev, act="silu", identity=False, seed=0):
    cfg = scaled(CONFIGS["tiny"], T=T, H=H, I=I, E=E, top_k=k, quant="nvfp4", activation=act)
    inp = make_inputs(cfg, seed=seed)
    d = lambda t: t.to(dev)
    al = moe.moe_align(d(ids), E)
    q, sf = moe.moe_prepare_nvfp4(d(inp.a1), None, k, False, NVFP4_A1_GSCALE)
    ws = torch.empty(max(moe.workspace_size_nvfp4(T, H, I, E, k), 16), dtype=torch.uint8, device=dev)
    y = moe.moe_experts_nvfp4(q, sf, NVFP4_A1_GSCALE, d(inp.w13), d(inp.w13_scale), d(inp.extra["w13_gscale"]),
                              d(inp.w2), d(inp.w2_scale), d(inp.extra["w2_gscale"]), NVFP4_H_GSCALE, al,
                              identity=identity, activation=act, ws=ws)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == moe.MOE_OK
    rq, rsf = moe_ref.prepare_nvfp4(inp.a1, None, False, NVFP4_A1_GSCALE)
    _same_codes(q, sf, rq, rsf)
    ral = moe_ref.align(ids, E, 128)
    yref, h_ref = moe_ref.experts_nvfp4(rq, rsf, NVFP4_A1_GSCALE, inp.w13, inp.w13_scale, inp.extra["w13_gscale"],
                                        inp.w2, inp.w2_scale, inp.extra["w2_gscale"], NVFP4_H_GSCALE, ral, k, act,
                                        return_h=True)
    _stages(inp, ral, ws, y, h_ref, T, H, I, E, k, f"experts nvfp4 T{T} H{H} I{I} E{E} k{k} {act}")
    return y, yref


def _stages(inp, ral, ws, y, h_ref, T, H, I, E, k, what):
    """NVFP4 experts stage by stage.  GEMM1: the GPU's bf16 h (left in the workspace)
    against the oracle's fp64 h, within one bf16 step (plus 1e-3 of the row's RMS for
    the fp32 summation order).  Quantisation: the GPU's codes and scale codes equal the
    oracle quantiser's on the GPU's own bf16 h, bit for bit.  GEMM2: the expert rows
    against the oracle's second GEMM on the GPU's codes, at the bf16 bound."""
    hb, hq, hsf = moe.experts_intermediate_nvfp4(ws, T, H, I, E, k)
    offs, order = ral.expert_offsets.numpy(), ral.sorted_slot.numpy()
    S = int(offs[-1])
    if S == 0:
        return
    hb64 = hb[:S].double().cpu().numpy()
    rms = np.sqrt((h_ref ** 2).mean(axis=1, keepdims=True))
    over = np.abs(hb64 - h_ref) > ulp_bf16(h_ref) + 1e-3 * rms
    assert not over.any(), f"{what}: {int(over.sum())} elements of the bf16 intermediate beyond one bf16 step"
    rq, rsf = moe_ref.nvfp4_quantize_fp32(hb64, NVFP4_H_GSCALE)
    _same_codes(hq[:S], hsf[:S], torch.from_numpy(rq), torch.from_numpy(rsf))
    hdeq = moe_ref.nvfp4_dequantize(hq[:S].cpu().numpy(), hsf[:S].cpu().numpy(), NVFP4_H_GSCALE)
    g2 = inp.extra["w2_gscale"].double().numpy().reshape(-1)
    y2 = torch.zeros((S, H), dtype=torch.float64)
    for e in range(E):
        p0, p1 = int(offs[e]), int(offs[e + 1])
        if p0 < p1:
            W2 = moe_ref.nvfp4_dequantize(inp.w2[e].numpy(), inp.w2_scale[e].numpy(), g2[e])
            y2[torch.from_numpy(order[p0:p1].astype(np.int64))] = moe_ref._expert_out(hdeq[p0:p1],
                                                                                        torch.from_numpy(W2))
    check_bf16(y, y2, what + ": second GEMM on the GPU's intermediate", slack=half_ulp_bf16(y2.numpy()))


@pytest.mark.parametrize("T,H,I,E,k,skew", [
    (16, 256, 512, 8, 2, False),      # the tiny layer
    (300, 512, 512, 4, 2, False),     # 2 M tiles per expert, ragged tails
    (700, 512, 256, 6, 2, True),      # skewed: a many-tile expert, an empty one
    (130, 2048, 256, 3, 1, False),    # deep K (8 stages of 256)
    (1, 256, 256, 8, 2, False),       # single token
    (256, 256, 2048, 64, 4, False),   # >= 4 units per CTA: round-robin schedule
    (4, 2048, 2048, 16, 1, False),    # stream-K in both GEMMs, single-row tiles
    (1, 4096, 1024, 8, 1, False),     # stream-K GEMM1: few units cut into many segments
    (12, 2048, 2048, 8, 2, True),     # stream-K with skewed routing
    (512, 4096, 2048, 8, 2, False),   # the Mixtral-like shape at a smaller I: ~190 gemm2 units, 1.3 waves
    (600, 4096, 2048, 8, 2, True),    # the same with skewed routing (a many-tile expert, an empty one)
])
def test_experts_nvfp4(cuda_dev, T, H, I, E, k, skew):
    y, yref = _run(T, H, I, E, k, _ids(T, k, E, T + H, skew), cuda_dev)
    check_nvfp4(y, yref, "experts nvfp4")


@pytest.mark.parametrize("T,H,I,E,k,act", [
    (300, 512, 512, 4, 2, "gelu"),
    (300, 512, 512, 4, 2, "swigluoai"),
    (300, 512, 512, 4, 2, "silu_no_mul"),    # 512 gate rows: two 256-row N tiles
    (4, 2048, 2048, 16, 1, "gelu_no_mul"),   # stream-K, gate-only units
])
def test_experts_nvfp4_activations(cuda_dev, T, H, I, E, k, act):
    y, yref = _run(T, H, I, E, k, _ids(T, k, E, T + I), cuda_dev, act=act)
    check_nvfp4(y, yref, f"experts nvfp4 {act}")


def test_experts_nvfp4_identity_permutation(cuda_dev):
    ids = torch.zeros((200, 1), dtype=torch.int32)
    y, yref = _run(200, 512, 256, 1, 1, ids, cuda_dev, identity=True)
    check_nvfp4(y, yref, "experts nvfp4 identity")


def test_experts_nvfp4_rejects_bad_shapes(cuda_dev):
    cfg = scaled(CONFIGS["tiny"], T=4, H=384, I=256, E=2, top_k=1, quant="nvfp4")   # H % 256 != 0
    inp = make_inputs(cfg)
    d = lambda t: t.to(cuda_dev)
    al = moe.moe_align(torch.zeros((4, 1), dtype=torch.int32, device=cuda_dev), 2)
    q, sf = moe.moe_prepare_nvfp4(d(inp.a1), None, 1, False, NVFP4_A1_GSCALE)
    with pytest.raises(moe.MoeError):
        moe.moe_experts_nvfp4(q, sf, NVFP4_A1_GSCALE, d(inp.w13), d(inp.w13_scale), d(inp.extra["w13_gscale"]),
                              d(inp.w2), d(inp.w2_scale), d(inp.extra["w2_gscale"]), NVFP4_H_GSCALE, al,
                              ws=torch.empty(16, dtype=torch.uint8, device=cuda_dev))
