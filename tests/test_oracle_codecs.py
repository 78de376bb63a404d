"""Pins of the oracle's number-format codecs (CPU only)."""
import os

import numpy as np
import pytest
import torch

from oracle import codecs

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_e4m3_matches_ocp_table():
    for line in open(os.path.join(GOLD, "e4m3_ocp.txt")):
        if line.startswith("#") or not line.strip():
            continue
        v, c = line.split()
        assert int(codecs.e4m3_encode(np.array([float(v)]))[0]) == int(c, 16), v
        if abs(float(v)) <= 448:
            assert codecs.e4m3_decode(np.array([int(c, 16)]))[0] == float(v) or float(v) == 0


def test_e4m3_matches_torch_cast_on_all_bf16_values():
    bits = torch.arange(0, 65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    x = bits.float()
    keep = torch.isfinite(x) & (x.abs() < 464)  # torch's cast is not saturating beyond 464
    x = x[keep]
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = codecs.e4m3_encode(x.double().numpy())
    assert (ref == got).all()


def test_e4m3_matches_torch_cast_on_random_fp32():
    g = torch.Generator().manual_seed(1)
    x = (torch.randn(400000, generator=g, dtype=torch.float64) *
         torch.exp(torch.empty(400000, dtype=torch.float64).uniform_(-14, 6, generator=g))).float()
    x = x[x.abs() < 464]
    assert (x.to(torch.float8_e4m3fn).view(torch.uint8).numpy() == codecs.e4m3_encode(x.double().numpy())).all()


def test_e4m3_codes_round_trip_and_saturate():
    codes = np.arange(256, dtype=np.uint8)
    vals = codecs.e4m3_decode(codes)
    finite = ~np.isnan(vals)
    assert finite.sum() == 254  # 0x7F and 0xFF are the only NaNs
    assert (codecs.e4m3_encode(vals[finite]) == codes[finite]).all()
    assert np.nanmax(vals) == 448.0
    big = np.array([448.5, 463.9, 464.0, 480.0, 1e9, np.inf])
    assert (codecs.e4m3_encode(big) == 0x7E).all()
    assert (codecs.e4m3_encode(-big) == 0xFE).all()


def _e2m1_brute(x):
    # nearest table value; ties to the even code index
    a = abs(x)
    best = None
    for i, v in enumerate(codecs.E2M1_VALUES):
        d = abs(a - v)
        if best is None or d < best[0] - 1e-15 or (abs(d - best[0]) <= 1e-15 and i % 2 == 0):
            best = (d, i)
    i = best[1] if a <= 6 else 7
    return i | (8 if np.signbit(x) else 0)


def test_e2m1_brute_force():
    xs = np.concatenate([np.arange(-8 * 64, 8 * 64 + 1) / 64.0, np.random.default_rng(0).normal(0, 3, 2000)])
    got = codecs.e2m1_encode(xs)
    exp = np.array([_e2m1_brute(x) for x in xs], dtype=np.uint8)
    assert (got == exp).all()
    assert (codecs.e2m1_decode(np.arange(16)) == np.concatenate([codecs.E2M1_VALUES, -codecs.E2M1_VALUES])).all()


def test_bf16_rounding_matches_torch_from_fp32():
    g = torch.Generator().manual_seed(2)
    x = (torch.randn(300000, generator=g, dtype=torch.float64) *
         torch.exp(torch.empty(300000, dtype=torch.float64).uniform_(-90, 90, generator=g))).float()
    x = torch.cat([x, torch.tensor([1e-40, -3e-39, 3.3e38, -3.39e38, 0.0, -0.0])])
    ref = x.to(torch.bfloat16).double().numpy()
    got = codecs.round_bf16(x.double().numpy())
    assert np.array_equal(ref, got) or np.allclose(ref, got, rtol=0, atol=0, equal_nan=True)


def test_bf16_rounding_is_a_single_rounding_from_fp64():
    # 1 + 2^-8 + 2^-30: above the halfway point between 1 and 1 + 2^-7, so it
    # rounds up; rounding to fp32 first would land on the tie and go to 1.0.
    x = 1.0 + 2.0 ** -8 + 2.0 ** -30
    assert codecs.round_bf16(np.array([x]))[0] == 1.0 + 2.0 ** -7
    assert codecs.round_bf16(np.array([1.0 + 2.0 ** -8]))[0] == 1.0          # tie -> even
    assert codecs.round_bf16(np.array([1.0 + 3 * 2.0 ** -8]))[0] == 1.0 + 2.0 ** -6  # tie -> even (up)
