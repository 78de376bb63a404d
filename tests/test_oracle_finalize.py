"""Pins of the oracle finalize and NVFP4 packing (CPU only)."""
import os

import numpy as np
import torch

from oracle import codecs, moe_ref

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rows(S, H, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn((S, H), generator=g).to(torch.bfloat16)


def test_weighted_sum_closed_form():
    y = _rows(12, 64, 0)
    w = torch.tensor([[1.0, 0.0, 0.0], [0.0, 0.0, 1.0], [0.25, 0.5, 0.25], [0.5, 0.5, 0.0]])
    fo = moe_ref.finalize(y, w, 3, False)
    yd = y.double().numpy().reshape(4, 3, 64)
    assert np.array_equal(fo.out[0], yd[0, 0]) and np.array_equal(fo.out[1], yd[1, 2])
    assert np.array_equal(fo.out[2], 0.25 * yd[2, 0] + 0.5 * yd[2, 1] + 0.25 * yd[2, 2])


def test_shared_and_residual_are_added_unscaled():
    y, sh, res = _rows(8, 32, 1), _rows(4, 32, 2), _rows(4, 32, 3)
    w = torch.full((4, 2), 0.5)
    base = moe_ref.finalize(y, w, 2, False).out
    fo = moe_ref.finalize(y, w, 2, False, shared=sh, residual=res)
    assert np.allclose(fo.out, base + sh.double().numpy() + res.double().numpy(), rtol=0, atol=1e-15)
    assert torch.equal(fo.residual_out, moe_ref.to_bf16_tensor(fo.out))


def test_rmsnorm_closed_forms():
    y = _rows(6, 7168, 4)
    ones = torch.ones(7168, dtype=torch.bfloat16)
    eps = 1e-6
    fo = moe_ref.finalize(y, torch.ones((6, 1)), 1, False, rms_weight=ones, eps=eps)
    yd = y.double().numpy()
    ms = (yd ** 2).mean(1)
    assert np.allclose((fo.out ** 2).mean(1), ms / (ms + eps), rtol=1e-12)
    # scale invariance of the normalised direction (eps = 0)
    f1 = moe_ref.finalize(y, torch.full((6, 1), 1.0), 1, False, rms_weight=ones, eps=0.0).out
    f2 = moe_ref.finalize(y, torch.full((6, 1), 4.0), 1, False, rms_weight=ones, eps=0.0).out
    assert np.allclose(f1, f2, rtol=1e-12, atol=0)
    gm = torch.linspace(0.5, 1.5, 7168).to(torch.bfloat16)
    f3 = moe_ref.finalize(y, torch.ones((6, 1)), 1, False, rms_weight=gm, eps=0.0).out
    assert np.allclose(f3, f1 * gm.double().numpy()[None], rtol=1e-12, atol=0)


def test_nvfp4_golden_group():
    lines = {l.split()[0]: l.split()[1:] for l in open(os.path.join(GOLD, "nvfp4_group.txt")) if not l.startswith("#")}
    x = np.array([[float(v) for v in lines["input"]]])
    packed, sf = moe_ref.nvfp4_quantize(x, 1.0)
    assert sf.tolist() == [[int(lines["scale"][0], 16)]]
    assert packed[0].tolist() == [int(v, 16) for v in lines["packed"]]


def test_nvfp4_grid_values_reproduce_exactly_and_scale_round_trips():
    rng = np.random.default_rng(3)
    R, C = 8, 256
    codes = rng.integers(0, 16, size=(R, C)).astype(np.uint8)
    codes[:, ::16] = 7                                # amax = 6 * sf in every group
    sfv = codecs.e4m3_decode(rng.integers(0x20, 0x60, size=(R, C // 16)).astype(np.uint8))
    for gs in (1.0, 0.5):
        x = codecs.e2m1_decode(codes) * np.repeat(sfv, 16, 1) * gs
        packed, sf = moe_ref.nvfp4_quantize(x, gs)
        assert np.array_equal(codecs.e4m3_decode(sf), sfv)
        assert np.array_equal(moe_ref.nvfp4_dequantize(packed, sf, gs), x)


def test_nvfp4_zero_group_and_error_bound():
    x = np.random.default_rng(4).normal(size=(4, 64))
    x[1, 16:32] = 0
    packed, sf = moe_ref.nvfp4_quantize(x, 1.0)
    assert sf[1, 1] == 0 and (packed[1, 8:16] == 0).all()
    deq = moe_ref.nvfp4_dequantize(packed, sf, 1.0)
    step = np.repeat(codecs.e4m3_decode(sf), 16, 1)   # one unit of the group's scale
    a = np.abs(x) / np.where(step > 0, step, 1)
    half_step = np.where(a < 2, 0.25, np.where(a < 4, 0.5, 1.0)) * step
    # the block scale itself is rounded, so |x| can exceed 6*sf by up to 1/16: allow the saturation gap
    assert (np.abs(deq - x) <= half_step + np.maximum(np.abs(x) - 6 * step, 0) + 1e-12).all()
