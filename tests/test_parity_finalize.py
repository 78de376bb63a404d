"""GPU finalize vs the oracle (weighted sum, shared, residual, RMSNorm, NVFP4)."""
import numpy as np
import pytest
import torch

from mixture_experts_layer_tokens_gb300 import moe
from mixture_experts_layer_tokens_gb300.inputs import CONFIGS, make_inputs, scaled
from mixture_experts_layer_tokens_gb300.layer import FinalizeStep
from oracle import codecs, moe_ref
from parity_util import check_bf16, to64

pytestmark = pytest.mark.gpu


def _nvfp4_check(packed, sf, ref64, g):
    """Each dequantised element lies within one E2M1 step (at its magnitude, in
    units of the group scale) of the exact value; scales within one E4M3 step."""
    packed, sf = packed.cpu().numpy(), sf.cpu().numpy()
    deq = moe_ref.nvfp4_dequantize(packed, sf, g)
    rp, rsf = moe_ref.nvfp4_quantize(ref64, g)
    unit = np.repeat(codecs.e4m3_decode(rsf) * g, 16, axis=1)
    a = np.abs(ref64) / np.where(unit > 0, unit, 1)
    step = np.where(a < 2, 0.5, np.where(a < 4, 1.0, 2.0)) * unit
    # values a rounded-down block scale pushes past 6 * unit saturate: allow that gap too
    slack = np.maximum(np.abs(ref64) - 6 * unit, 0)
    err = np.abs(deq - ref64)
    assert (err <= step + slack + 1e-30).all(), f"max excess {(err - step - slack).max():.3e}"
    gs = codecs.e4m3_decode(sf).astype(np.float64)
    rs = codecs.e4m3_decode(rsf).astype(np.float64)
    assert (np.abs(gs - rs) <= rs * 2.0 ** -3 + 2.0 ** -9).all()
    exact = np.mean(packed == rp)
    assert exact > 0.99, f"only {exact:.4f} of the packed bytes equal the oracle's"


@pytest.mark.parametrize("name", ["finalize128", "finalize512"])
def test_finalize_configs(cuda_dev, name):
    cfg = CONFIGS[name]
    inp = make_inputs(cfg)
    step = FinalizeStep(inp.to(cuda_dev))
    w = step.weights()
    out, _ = step.finalize(False)
    fp4, sf = step.finalize(True)
    torch.cuda.synchronize()
    ref = moe_ref.finalize(inp.y, w.cpu(), 4, False, shared=inp.extra["shared"], residual=inp.residual,
                           rms_weight=inp.rms_weight, eps=1e-6, nvfp4_global_scale=1.0)
    check_bf16(out, ref.out, name)
    _nvfp4_check(fp4, sf, ref.out, 1.0)


@pytest.mark.parametrize("T,H,k", [(1, 7168, 4), (3, 256, 1), (300, 4096, 2), (40, 2048, 8), (2, 14336, 4),
                                   (600, 264, 2)])
@pytest.mark.parametrize("variant", ["plain", "shared_res", "rms", "won", "all"])
def test_finalize_variants(cuda_dev, T, H, k, variant):
    g = torch.Generator().manual_seed(T * H + k)
    y = torch.randn((T * k, H), generator=g).to(torch.bfloat16)
    w = torch.softmax(torch.randn((T, k), generator=g), 1)
    sh = torch.randn((T, H), generator=g).to(torch.bfloat16) if variant in ("shared_res", "all") else None
    res = torch.randn((T, H), generator=g).to(torch.bfloat16) if variant in ("shared_res", "all") else None
    gm = (torch.rand(H, generator=g) + 0.5).to(torch.bfloat16) if variant in ("rms", "all") else None
    won = variant == "won"
    d = lambda t: None if t is None else t.to(cuda_dev)
    res_out = torch.empty((T, H), dtype=torch.bfloat16, device=cuda_dev)
    out, _ = moe.moe_finalize(d(y), d(w), k, won, shared=d(sh), residual=d(res), rms_weight=d(gm),
                              residual_out=res_out)
    o32, _ = moe.moe_finalize(d(y), d(w), k, won, shared=d(sh), residual=d(res), rms_weight=d(gm),
                              out_dtype=moe.MOE_DT_FP32)
    torch.cuda.synchronize()
    ref = moe_ref.finalize(y, w, k, won, shared=sh, residual=res, rms_weight=gm, eps=1e-6)
    check_bf16(out, ref.out, f"{variant} bf16")
    # fp32 output: the literal bound 1e-2 * RMS(ref) with no output rounding
    g64, r64 = to64(o32), ref.out
    rms = np.sqrt(np.mean(r64 ** 2))
    assert np.abs(g64 - r64).max() <= 1e-2 * rms and np.linalg.norm(g64 - r64) / np.linalg.norm(r64) <= 5e-3
    # residual_out is bf16 of the pre-norm sum
    check_bf16(res_out, ref.residual_out.double(), "residual_out")


@pytest.mark.parametrize("gscale", [1.0, 0.25, 3.0])
def test_finalize_nvfp4_global_scales(cuda_dev, gscale):
    g = torch.Generator().manual_seed(9)
    T, H, k = 64, 7168, 4
    y = torch.randn((T * k, H), generator=g).to(torch.bfloat16)
    w = torch.softmax(torch.randn((T, k), generator=g), 1)
    gm = (torch.rand(H, generator=g) + 0.5).to(torch.bfloat16)
    fp4, sf = moe.moe_finalize(y.to(cuda_dev), w.to(cuda_dev), k, rms_weight=gm.to(cuda_dev),
                               out_dtype=moe.MOE_DT_NVFP4, out_global_scale=gscale)
    torch.cuda.synchronize()
    ref = moe_ref.finalize(y, w, k, False, rms_weight=gm, eps=1e-6, nvfp4_global_scale=gscale)
    _nvfp4_check(fp4, sf, ref.out, gscale)


def test_finalize_empty(cuda_dev):
    y = torch.empty((0, 256), dtype=torch.bfloat16, device=cuda_dev)
    out, _ = moe.moe_finalize(y, torch.empty((0, 2), device=cuda_dev), 2)
    assert out.shape == (0, 256)


@pytest.mark.parametrize("T,H,k", [(300, 4096, 2), (3, 7168, 4), (512, 7168, 4)])
def test_finalize_residual_in_place(cuda_dev, T, H, k):
    """residual_out written over residual (the in-place add + RMSNorm): the outputs are
    those of the out-of-place call and the residual buffer ends up holding the sum."""
    g = torch.Generator().manual_seed(T + H)
    y = torch.randn((T * k, H), generator=g).to(torch.bfloat16)
    w = torch.softmax(torch.randn((T, k), generator=g), 1)
    sh = torch.randn((T, H), generator=g).to(torch.bfloat16)
    res = torch.randn((T, H), generator=g).to(torch.bfloat16)
    gm = (torch.rand(H, generator=g) + 0.5).to(torch.bfloat16)
    d = lambda t: t.to(cuda_dev)
    res_out = torch.empty((T, H), dtype=torch.bfloat16, device=cuda_dev)
    out_sep, _ = moe.moe_finalize(d(y), d(w), k, False, shared=d(sh), residual=d(res), rms_weight=d(gm),
                                  residual_out=res_out)
    res_buf = d(res).clone()
    out_inp, _ = moe.moe_finalize(d(y), d(w), k, False, shared=d(sh), residual=res_buf, rms_weight=d(gm),
                                  residual_out=res_buf)
    torch.cuda.synchronize()
    assert torch.equal(out_inp, out_sep)
    assert torch.equal(res_buf, res_out)
    ref = moe_ref.finalize(y, w, k, False, shared=sh, residual=res, rms_weight=gm, eps=1e-6)
    check_bf16(res_buf, ref.residual_out.double(), "residual in place")
