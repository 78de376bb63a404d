"""Pins of the oracle's activations between the two expert GEMMs.

The "Fused Experts Kernels" table (vLLM design doc) names the activations
without formulas; the oracle's readings are stated in ``oracle/moe_ref.py``.
These checks tie them to facts outside the oracle: the normal CDF's table
values, the odd-part identities of SiLU and GELU, the clamping structure of the
gpt-oss SwiGLU, and the reduction of a gated layer whose up projection is
exactly 1 to the matching *_no_mul layer."""
import math

import numpy as np
import pytest
import torch

from oracle import moe_ref

F64 = torch.float64


def _act1(name, g):
    """act(g) alone: the *_no_mul form, or the gated form with u = 1."""
    if name.endswith("_no_mul"):
        return moe_ref.activation(g[:, None], name)[:, 0]
    return moe_ref.activation(torch.stack([g, torch.ones_like(g)], 1), name)[:, 0]


@pytest.mark.parametrize("name", ["silu_no_mul", "gelu_no_mul", "gelu_tanh", "silu", "gelu"])
def test_odd_part_identity(name):
    # sigmoid(x) + sigmoid(-x) = 1, Phi(x) + Phi(-x) = 1 and tanh odd give act(x) - act(-x) = x
    x = torch.linspace(-12.0, 12.0, 2001, dtype=F64)
    d = _act1(name, x) - _act1(name, -x)
    assert torch.allclose(d, x, rtol=0, atol=1e-12)


def test_gelu_is_x_times_normal_cdf():
    # Phi(1), Phi(-1), Phi(2), Phi(-3) from the standard normal table
    table = {1.0: 0.8413447460685429, -1.0: 0.15865525393145707, 2.0: 0.9772498680518208,
             -3.0: 0.0013498980316301035}
    x = torch.tensor(list(table), dtype=F64)
    want = torch.tensor([k * v for k, v in table.items()], dtype=F64)
    for name in ("gelu", "gelu_no_mul"):
        assert torch.allclose(_act1(name, x), want, rtol=1e-14, atol=0)


def test_gelu_tanh_is_a_close_approximation_of_gelu():
    x = torch.linspace(-8.0, 8.0, 4001, dtype=F64)
    err = (_act1("gelu_tanh", x) - _act1("gelu", x)).abs()
    assert 1e-5 < err.max().item() < 1e-3   # a different function, within the approximation's error
    assert err[x.abs() > 6].max().item() < 1e-7  # both reach x and 0 in the tails


def test_silu_forms_agree():
    g = torch.randn(64, 32, dtype=F64, generator=torch.Generator().manual_seed(1)) * 4
    u = torch.randn(64, 32, dtype=F64, generator=torch.Generator().manual_seed(2))
    gu = torch.cat([g, u], 1)
    assert torch.equal(moe_ref.activation(gu, "silu"), moe_ref.silu_and_mul(gu))
    assert torch.allclose(moe_ref.activation(g, "silu_no_mul"), g * torch.sigmoid(g), rtol=1e-15, atol=1e-300)


def test_swigluoai_structure():
    L, a = moe_ref.SWIGLUOAI_LIMIT, moe_ref.SWIGLUOAI_ALPHA
    assert (L, a) == (7.0, 1.702)
    h = lambda g, u: moe_ref.activation(torch.tensor([[g, u]], dtype=F64), "swigluoai").item()
    for g in (-3.0, 0.5, 6.9, 12.0):
        assert h(g, -1.0) == 0.0                      # (u + 1) factor
    for u in (-6.0, 0.0, 2.5):
        assert h(10.0, u) == h(7.0, u) and h(50.0, u) == h(7.0, u)  # gate clamped above at the limit
    for g in (-2.0, 1.0, 5.0):
        assert h(g, 9.0) == h(g, 7.0) and h(g, -9.0) == h(g, -7.0)  # up clamped to [-limit, limit]
    assert abs(h(-60.0, 3.0)) < 1e-20                  # no clamp below: the sigmoid closes the gate
    # inside the limits it is (u + 1) * silu(alpha g) / alpha: alpha only scales the sigmoid's argument
    g = torch.linspace(-8, 7, 301, dtype=F64)
    u = torch.linspace(-7, 7, 301, dtype=F64)
    got = moe_ref.activation(torch.stack([g, u], 1), "swigluoai")[:, 0]
    silu_ag = (a * g) * torch.sigmoid(a * g)
    assert torch.allclose(got, (u + 1) * silu_ag / a, rtol=1e-14, atol=1e-300)


@pytest.mark.parametrize("name", ["silu", "gelu"])
def test_gated_layer_with_unit_up_projection_equals_no_mul_layer(name):
    # a1's last channel is 1 and every expert's up rows select it, so u = 1 exactly:
    # the gated layer must equal the *_no_mul layer built from the gate rows alone
    g = torch.Generator().manual_seed(3)
    T, H, I, E, k = 20, 256, 128, 3, 2
    a1 = (torch.randn(T, H, generator=g)).to(torch.bfloat16)
    a1[:, -1] = 1.0
    wg = (torch.randn(E, I, H, generator=g) / 16).to(torch.bfloat16)
    sel = torch.zeros(E, I, H, dtype=torch.bfloat16)
    sel[:, :, -1] = 1.0
    w13 = torch.cat([wg, sel], 1)
    w2 = (torch.randn(E, H, I, generator=g) / 11).to(torch.bfloat16)
    ids = torch.argsort(torch.rand(T, E, generator=g), 1)[:, :k].to(torch.int32)
    al = moe_ref.align(ids, E, 128)
    y_gated = moe_ref.experts(a1, None, w13, None, w2, None, al, k, "bf16", name)
    y_nomul = moe_ref.experts(a1, None, wg, None, w2, None, al, k, "bf16", name + "_no_mul")
    assert torch.equal(y_gated, y_nomul)
    assert not torch.equal(y_gated, moe_ref.experts(a1, None, w13, None, w2, None, al, k, "bf16",
                                                    "gelu" if name == "silu" else "silu"))


def test_unknown_activation_is_rejected():
    with pytest.raises(ValueError):
        moe_ref.activation(torch.zeros(2, 4, dtype=F64), "relu")
