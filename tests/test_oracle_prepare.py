"""Pins of the oracle prepare step (CPU only)."""
import numpy as np
import pytest
import torch

from oracle import codecs, moe_ref


def _a1(T=8, H=256, seed=0):
    g = torch.Generator().manual_seed(seed)
    return torch.randn((T, H), generator=g).to(torch.bfloat16)


def test_bf16_passthrough():
    a1 = _a1()
    a1q, s = moe_ref.prepare(a1, torch.ones((8, 1)), False, "bf16")
    assert s is None and torch.equal(a1q, a1)


def test_weight_on_input_exact_cases():
    a1 = _a1()
    for w, f in ((1.0, 1.0), (0.5, 0.5), (-2.0, -2.0)):
        out, _ = moe_ref.prepare(a1, torch.full((8, 1), w), True, "bf16")
        assert torch.equal(out.float(), a1.float() * f)


def test_weight_on_input_casts_weight_to_activation_type_first():
    # 1.5 + 2^-8 is halfway between two bf16 numbers; cast to bf16 it is 1.5 (even), so the
    # product must be bf16(a1 * 1.5), while the fp32 weight would give other values.
    a1 = _a1(T=4, H=512)
    w = torch.full((4, 1), 1.5 + 2.0 ** -8)
    out, _ = moe_ref.prepare(a1, w, True, "bf16")
    assert torch.equal(out, (a1.float() * 1.5).to(torch.bfloat16))
    assert not torch.equal((a1.float() * w).to(torch.bfloat16), out)


def test_weight_on_input_is_correctly_rounded_product():
    a1 = _a1(T=16, H=256, seed=3)
    g = torch.Generator().manual_seed(9)
    w = torch.rand((16, 1), generator=g)
    out, _ = moe_ref.prepare(a1, w, True, "bf16")
    exact = a1.double() * w.to(torch.bfloat16).double()     # bf16 x bf16 is exact in fp64
    err = (out.double() - exact).abs()
    ulp = torch.from_numpy(np.spacing(np.abs(exact.numpy()).astype(np.float32)).astype(np.float64)) * 2 ** 16
    assert (err <= ulp / 2).all()


def test_weight_on_input_needs_top1():
    with pytest.raises(AssertionError):
        moe_ref.prepare(_a1(), torch.ones((8, 2)), True, "bf16")


def test_fp8_codes_match_torch_cast_of_the_ratio():
    a1 = _a1(T=32, H=512, seed=4)
    q, s = moe_ref.prepare(a1, None, False, "fp8")
    x = a1.float().reshape(32, 4, 128)
    amax = x.abs().amax(2)
    s_ref = torch.maximum(amax, torch.tensor(1e-10, dtype=torch.float32)) / 448.0   # fp32 IEEE division
    assert torch.equal(s, s_ref)
    q_ref = (x / s_ref[:, :, None]).to(torch.float8_e4m3fn).view(torch.uint8).reshape(32, 512)
    assert torch.equal(q, q_ref)


def test_fp8_group_extremes():
    a1 = _a1(T=2, H=256, seed=5)
    a1[0, :128] = 0
    q, s = moe_ref.prepare(a1, None, False, "fp8")
    assert (q[0, :128] == 0).all()
    assert s[0, 0].item() == np.float32(np.float32(1e-10) / np.float32(448.0))
    for r, gi in ((0, 1), (1, 0), (1, 1)):
        grp = a1[r, gi * 128:(gi + 1) * 128].float()
        i = int(grp.abs().argmax())
        assert codecs.e4m3_decode(q[r, gi * 128 + i].item()) == (448.0 if grp[i] > 0 else -448.0)
    deq = moe_ref.dequant_fp8_g128(q.numpy(), s.numpy())
    x = a1.double().numpy()
    assert (np.abs(deq - x) <= np.abs(x) * 2.0 ** -4 + np.repeat(s.numpy().astype(np.float64), 128, 1) * 2.0 ** -10).all()


def test_fp8_scale_invariance_under_powers_of_two():
    a1 = _a1(T=4, H=256, seed=6)
    q, s = moe_ref.prepare(a1, None, False, "fp8")
    q2, s2 = moe_ref.prepare((a1.float() * 8).to(torch.bfloat16), None, False, "fp8")
    assert torch.equal(q, q2) and torch.equal(s2, s * 8)


def test_fp8_exact_round_trip_on_grid_values():
    rng = np.random.default_rng(7)
    codes = rng.integers(0, 256, size=(4, 256)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x10
    codes[:, 0] = 0x7E                      # amax = 448 * 2^-5 in every group
    codes[:, 128] = 0xFE
    x = codecs.e4m3_decode(codes) * 2.0 ** -5
    q, s = moe_ref.quantize_fp8_g128(x)
    assert (s == np.float32(2.0 ** -5)).all()
    assert (moe_ref.dequant_fp8_g128(q, s) == x).all()
