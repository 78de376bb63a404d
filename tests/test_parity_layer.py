"""Whole-layer parity: route -> align -> prepare -> experts (+ shared) -> finalize
through the C ABI against the oracle.

Small shapes of every configuration are checked on every token; the full-size
configurations are run exactly as the bench runs them and checked on sampled
tokens, which the oracle computes one expert at a time."""
import numpy as np
import pytest
import torch

from mixture_experts_layer_tokens_gb300 import moe
from mixture_experts_layer_tokens_gb300.inputs import CONFIGS, make_inputs, scaled
from mixture_experts_layer_tokens_gb300.layer import MoELayer
from oracle import moe_ref
from parity_util import check_bf16, check_fp8, check_nvfp4, ulp_bf16

pytestmark = pytest.mark.gpu


def oracle_tokens(inp, tokens, gpu_ids, gpu_w):
    """Oracle output rows (fp64) of the given tokens and the rounding slack of
    the bf16 intermediates (see parity_util).  The router is checked bit-exact
    against the oracle's; the weights fed on are the GPU's (same inputs for
    every stage)."""
    cfg = inp.cfg
    k = cfg.top_k
    logits = inp.logits[tokens].cpu()
    if cfg.scoring == "sigmoid":
        ids, _ = moe_ref.route_sigmoid_top1(logits)
    else:
        ids, _ = moe_ref.route_softmax_renorm(logits, k)
    assert torch.equal(ids, gpu_ids[tokens].cpu())
    w = gpu_w[tokens].cpu()
    a1 = inp.a1[tokens].cpu()
    n, H = len(tokens), cfg.H
    y = torch.zeros((n * k, H), dtype=torch.float64)
    if cfg.quant == "nvfp4":
        # every row quantises on its own: the sampled tokens' rows are exact
        a1q, sc = moe_ref.prepare_nvfp4(a1, w, cfg.weight_on_input, inp.extra["a1_gscale"])
        x = inp.extra
        y = moe_ref.experts_nvfp4(a1q, sc, x["a1_gscale"], inp.w13.cpu(), inp.w13_scale.cpu(),
                                  x["w13_gscale"].cpu(), inp.w2.cpu(), inp.w2_scale.cpu(), x["w2_gscale"].cpu(),
                                  x["h_gscale"], moe_ref.align(ids, cfg.E, 128), k, cfg.activation)
    else:
        a1q, sc = moe_ref.prepare(a1, w, cfg.weight_on_input, cfg.quant)
    if cfg.quant == "fp8_tensor":
        # one scale over every expert's intermediate: the whole layer at once (all tokens)
        assert n == cfg.T
        y = moe_ref.experts(a1q, sc, inp.w13, inp.w13_scale, inp.w2, inp.w2_scale, moe_ref.align(ids, cfg.E, 128),
                            k, cfg.quant, cfg.activation)
    for e in ([] if cfg.quant in ("fp8_tensor", "nvfp4") else sorted(set(ids.reshape(-1).tolist()))):
        slots = [(i, j) for i in range(n) for j in range(k) if int(ids[i, j]) == e]
        rows = np.array([i for i, _ in slots])
        A = moe_ref._act64(a1q, sc, rows, cfg.quant)
        W13 = moe_ref._weights64(inp.w13, inp.w13_scale, e, cfg.quant)
        W2 = moe_ref._weights64(inp.w2, inp.w2_scale, e, cfg.quant)
        ye = moe_ref.expert_rows(A, W13, W2, cfg.quant, cfg.activation)
        for r, (i, j) in enumerate(slots):
            y[i * k + j] = ye[r]
    shared = moe_ref.dense_mlp(a1, inp.shared_w13[0], inp.shared_w2[0]) if cfg.shared_I else None
    res = inp.residual[tokens].cpu() if inp.residual is not None else None
    gm = None if inp.rms_weight is None else inp.rms_weight.cpu()
    fo = moe_ref.finalize(y, w, k, cfg.weight_on_input, shared=shared, residual=res, rms_weight=gm)
    yw = y.numpy().reshape(n, k, H)
    ww = np.ones((n, k)) if cfg.weight_on_input else w.double().numpy()
    slack = (np.abs(ww)[:, :, None] * ulp_bf16(yw)).sum(axis=1)
    if shared is not None:
        slack = slack + ulp_bf16(shared.numpy())
    if gm is not None:
        pre = moe_ref.finalize(y, w, k, cfg.weight_on_input, shared=shared, residual=res).out
        slack = slack / np.sqrt((pre ** 2).mean(axis=1, keepdims=True) + 1e-6) * np.abs(gm.double().numpy())[None]
    return fo.out, slack


def _check(cfg, out, ref, what):
    ref, slack = ref
    if cfg.quant == "nvfp4":
        return check_nvfp4(out, ref, what)
    if cfg.quant != "bf16":
        return check_fp8(out, ref, what)
    return check_bf16(out, ref, what, slack=slack)


SMALL = {
    "tiny": CONFIGS["tiny"],
    "mixtral_small": scaled(CONFIGS["mixtral"], T=200, H=512, I=768),
    "deepseek_small": scaled(CONFIGS["deepseek"], T=256, H=512, I=256, E=32, shared_I=256),
    "deepseek_small_token": scaled(CONFIGS["deepseek"], T=256, H=512, I=256, E=32, shared_I=256, quant="fp8_token"),
    "deepseek_small_tensor": scaled(CONFIGS["deepseek"], T=256, H=512, I=256, E=32, shared_I=256, quant="fp8_tensor"),
    "llama_small": scaled(CONFIGS["llama8"], T=100, H=384, I=512, shared_I=256),
    "llama_small_T1": scaled(CONFIGS["llama1"], H=384, I=512, shared_I=256),
    # shared expert with the routed experts' I: both in the same launches (moe_experts_multi)
    "llama_small_fused": scaled(CONFIGS["llama8"], T=100, H=384, I=512, shared_I=512),
    "llama_small_fused_T1": scaled(CONFIGS["llama1"], H=2048, I=2048, shared_I=2048),
    "residual_rms": scaled(CONFIGS["mixtral"], T=64, H=256, I=256, residual=True, rms=True),
    "mixtral_small_gelu_tanh": scaled(CONFIGS["mixtral"], T=200, H=512, I=768, activation="gelu_tanh"),
    "deepseek_small_gelu_no_mul": scaled(CONFIGS["deepseek"], T=256, H=512, I=256, E=32, shared_I=256,
                                         activation="gelu_no_mul"),
    "mixtral_small_nvfp4": scaled(CONFIGS["mixtral"], T=200, H=512, I=768, quant="nvfp4"),
    # the whole step as one launch (moe_layer_fused): round-robin and split GEMM schedules,
    # with and without the shared expert, residual and RMSNorm
    "llama_small_single": scaled(CONFIGS["llama8_fused"], T=100, H=384, I=512, shared_I=512),
    "llama_small_single_T1": scaled(CONFIGS["llama1_fused"], H=2048, I=2048, shared_I=2048),
    # at most 32 slots (decode stages: 32-row A boxes) with residual and RMSNorm
    "llama_small_single_T24": scaled(CONFIGS["llama8_fused"], T=24, H=1024, I=1024, shared_I=1024, residual=True,
                                     rms=True),
    "llama_small_fused_T24": scaled(CONFIGS["llama8"], T=24, H=1024, I=1024, shared_I=1024),
    "mixtral_small_single": scaled(CONFIGS["mixtral_fused"], T=200, H=512, I=768),
    "residual_rms_single": scaled(CONFIGS["mixtral_fused"], T=64, H=256, I=256, residual=True, rms=True),
    # the single launch's limits: E = 256 with top-8 (eight logits per lane, many small experts),
    # and T * top_k = 2048 slots
    "single_e256_top8": scaled(CONFIGS["mixtral_fused"], T=64, H=256, I=256, E=256, top_k=8),
    "single_max_slots": scaled(CONFIGS["mixtral_fused"], T=256, H=256, I=256, E=64, top_k=8),
    # weight on the input before the NVFP4 quantisation, bf16 shared expert beside the NVFP4 experts
    "llama_small_nvfp4": scaled(CONFIGS["llama8"], T=100, H=512, I=512, shared_I=256, quant="nvfp4"),
    # the Qwen3-MoE-like expert shape (H 2048, I 768: six 128-column groups of h) with 16 rows per
    # expert on average over 128 experts
    "qwen3_small": scaled(CONFIGS["qwen3"], T=256),
    "qwen3_small_fp8": scaled(CONFIGS["qwen3_fp8"], T=256),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_layer_small_all_tokens(cuda_dev, name):
    cfg = SMALL[name]
    inp = make_inputs(cfg)
    layer = MoELayer(inp.to(cuda_dev))
    out = layer.forward(layer.inp.logits, layer.inp.a1)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == moe.MOE_OK
    ref = oracle_tokens(inp, list(range(cfg.T)), layer.topk_ids, layer.topk_weights)
    _check(cfg, out, ref, name)


@pytest.mark.parametrize("name,sample", [("mixtral", 12), ("mixtral_T4096", 4), ("deepseek", 3), ("deepseek_T16384", 3),
                                         ("qwen3", 8), ("qwen3_fp8", 8),
                                         ("llama1", 1), ("llama8", 8),
                                         ("llama64", 6), ("llama512", 6), ("llama_shared512", 6), ("mixtral_nvfp4", 12),
                                         ("llama1_nvfp4", 1), ("llama1_fused", 1), ("llama64_fused", 6),
                                         ("mixtral_fused", 12)])
def test_layer_full_size_sampled_tokens(cuda_dev, name, sample):
    cfg = CONFIGS[name]
    inp = make_inputs(cfg, device=cuda_dev)   # full-size weights drawn on the device
    layer = MoELayer(inp)
    for _ in range(2):                        # the second run checks reuse of every buffer
        out = layer.forward(inp.logits, inp.a1)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == moe.MOE_OK
    g = torch.Generator().manual_seed(1)
    tokens = sorted(torch.randperm(cfg.T, generator=g)[:sample].tolist())
    if cfg.T - 1 not in tokens:
        tokens[-1] = cfg.T - 1                # always include the last token (ragged tail)
    ref = oracle_tokens(inp, tokens, layer.topk_ids, layer.topk_weights)
    _check(cfg, out[tokens], ref, name)
    # properties that hold at any size: finite everywhere, every routed expert row written
    assert torch.isfinite(out.float()).all()
    if not cfg.single_launch:
        assert int(layer.al.expert_offsets[-1]) == cfg.T * cfg.top_k


@pytest.mark.parametrize("T", [40, 20])  # 20 slots: both sides with the decode stages
def test_single_launch_matches_the_separate_calls(cuda_dev, T):
    """The one-launch step routes exactly like moe_route and, its GEMMs being the same
    units in the same order, gives the separate calls' output up to the finalize's fp32
    summation order."""
    cfg = scaled(CONFIGS["llama8_fused"], T=T, H=1024, I=1024, shared_I=1024, residual=True, rms=True)
    inp = make_inputs(cfg, device=cuda_dev)
    single = MoELayer(inp)
    sep = MoELayer(make_inputs(scaled(cfg, single_launch=False), device=cuda_dev))
    o1 = single.forward(inp.logits, inp.a1).clone()
    o2 = sep.forward(inp.logits, inp.a1)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == moe.MOE_OK
    assert torch.equal(single.topk_ids, sep.topk_ids) and torch.equal(single.topk_weights, sep.topk_weights)
    check_bf16(o1, o2.double(), "single launch vs separate calls", slack=ulp_bf16(o2.double().cpu().numpy()))


def test_deepseek_full_size_sampled_expert_rows(cuda_dev):
    """The DeepSeek-V3-like layer at full size (T 4096, 256 experts of ~128 rows, fp8
    G(128)), run as the bench runs it, checked stage by stage on one sorted row of each
    of 48 experts: the last row of 24 experts that have a second, partial 128-row tile,
    and a row of 24 experts with one tile (their first and last rows among them).  For
    each row: prepare bit-exact for its token; the intermediate h (codes and scales left
    in the workspace) against the oracle's quantisation of its own h; the expert row
    against the oracle's second GEMM on the GPU's intermediate, at the bf16 bound."""
    from parity_util import E4M3_VALUES, check_fp8_intermediate, fp8_row_scales, half_ulp_bf16
    cfg = CONFIGS["deepseek"]
    T, H, I, E, k = cfg.T, cfg.H, cfg.I, cfg.E, cfg.top_k
    inp = make_inputs(cfg, device=cuda_dev)
    layer = MoELayer(inp)
    layer.forward(inp.logits, inp.a1)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == moe.MOE_OK
    offs = layer.al.expert_offsets.cpu().numpy()
    order = layer.al.sorted_slot.cpu().numpy()
    counts = np.diff(offs)
    rng = np.random.default_rng(7)
    two = [e for e in range(E) if counts[e] > 128]
    one = [e for e in range(E) if 0 < counts[e] <= 128]
    assert len(two) >= 24 and len(one) >= 24
    picks = [(int(e), int(offs[e + 1] - 1)) for e in rng.choice(two, 24, replace=False)]
    singles = rng.choice(one, 24, replace=False)
    for i, e in enumerate(singles):
        r = 0 if i == 0 else (counts[e] - 1 if i == 1 else int(rng.integers(0, counts[e])))
        picks.append((int(e), int(offs[e] + r)))
    h_gpu, hs_gpu = moe.experts_intermediate(layer.ws, T, H, I, E, k, "fp8")
    rows = np.array([p for _, p in picks])
    codes = h_gpu[torch.from_numpy(rows).to(cuda_dev)].cpu().numpy()
    scales = fp8_row_scales(hs_gpu, "fp8", rows, I // 128)
    h_ref = np.zeros((len(picks), I))
    y_gpu = torch.zeros((len(picks), H), dtype=torch.float64)
    y_ref = torch.zeros((len(picks), H), dtype=torch.float64)
    h_deq = E4M3_VALUES[codes] * np.repeat(scales, 128, axis=1)
    for i, (e, p) in enumerate(picks):
        f = int(order[p])
        t = f // k
        rq, rs = moe_ref.prepare(inp.a1[t:t + 1].cpu(), None, False, "fp8")
        assert torch.equal(layer.a1q[t:t + 1].cpu(), rq) and torch.equal(layer.a1q_scale[t:t + 1].cpu(), rs)
        A = moe_ref._act64(rq, rs, np.array([0]), "fp8")
        h_ref[i] = moe_ref.silu_and_mul(A @ moe_ref._weights64(inp.w13, inp.w13_scale, e, "fp8").T).numpy()[0]
        y_ref[i] = moe_ref._expert_out(h_deq[i:i + 1], moe_ref._weights64(inp.w2, inp.w2_scale, e, "fp8"))[0]
        y_gpu[i] = layer.y[f].double().cpu()
    check_fp8_intermediate(codes, scales, h_ref, "fp8", "deepseek full size: sampled rows")
    check_bf16(y_gpu, y_ref, "deepseek full size: second GEMM on the GPU's intermediate",
               slack=half_ulp_bf16(y_ref.numpy()))
