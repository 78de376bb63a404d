"""Pins of the oracle's fp8 experts (CPU only): G(128), "A" and "T" formats.

"Fused MoE Kernel Features" (vLLM design doc), section "Fused Experts Kernels":
the fp8 experts take E4M3 activations with one fp32 scale per token per 128
channels ("G(128)"), per token ("A") or per tensor ("T"), and E4M3 weights with
one fp32 scale per 128x128 block; the intermediate between the two GEMMs is
quantised again in the activations' format.

The checks re-derive a tiny layer with scalar code written here from the
format definitions -- an E4M3 value table built from the OCP bit layout
(1 sign, 4 exponent bits with bias 7, 3 mantissa bits, subnormals at exponent
0, 0x7F/0xFF NaN), nearest-value search with ties to the even code, fp32
decision steps written with numpy.float32, and library dot products per
128-deep K block -- and compare the oracle with it.  The inputs make the
plausible mistakes visible: every token has its own scales, the routing sorts
slots out of token order, and the intermediate has values whose fp32 and bf16
roundings quantise to different codes.  Two tests plant such mistakes in the
oracle (monkeypatched, on the CPU) and show that the pin then fails.
"""
import math

import numpy as np
import pytest
import torch

from oracle import codecs, moe_ref


def _e4m3_value(c):
    s = -1.0 if c & 0x80 else 1.0
    e, m = (c >> 3) & 15, c & 7
    if e == 15 and m == 7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


E4M3 = np.array([_e4m3_value(c) for c in range(256)])
E4M3_POS = [(c, E4M3[c]) for c in range(0x7F)]  # non-negative finite codes, 0 .. 448


def _e4m3_code(x):
    """Nearest E4M3 code of a finite number, ties to the even code, saturating at 448."""
    a = abs(x)
    best = None
    for c, v in E4M3_POS:
        d = abs(v - a)
        if best is None or d < best[0] or (d == best[0] and c % 2 == 0):
            best = (d, c)
    c = best[1]
    return c | 0x80 if (x < 0 and c != 0) else c


def _bf16(x):
    """Round-to-nearest-even to 8 significant bits."""
    if x == 0.0 or not math.isfinite(x):
        return x
    m, e = math.frexp(x)
    s = m * 256.0
    r = math.floor(s)
    f = s - r
    if f > 0.5 or (f == 0.5 and r % 2 == 1):
        r += 1
    return math.ldexp(r / 256.0, e)


def _silu_mul(g, u):
    return g / (1.0 + math.exp(-g)) * u


def _quant_group(vals32):
    """fp32 decision steps of one scale group: s = fp32(max(amax, 1e-10) / 448),
    q = e4m3(fp32(x / s)).  Returns (codes, s)."""
    f32 = np.float32
    amax = f32(max(abs(float(v)) for v in vals32))
    s = f32(max(amax, f32(1e-10)) / f32(448.0))
    return [_e4m3_code(float(f32(f32(v) / s))) for v in vals32], s


def _layer(T=3, H=256, I=256, E=3, k=2, fmt="fp8", seed=5):
    """Random codes and scales of a tiny fp8 layer, and a routing whose sorted
    order differs from token order."""
    rng = np.random.default_rng(seed)

    def codes(*shape):
        c = rng.integers(0, 256, size=shape).astype(np.uint8)
        c[(c & 0x7F) == 0x7F] = 0x3A  # no NaN codes
        return c

    a1q = codes(T, H)
    if fmt == "fp8":
        a_s = (2.0 ** -rng.integers(2, 9, size=(T, H // 128)) * rng.uniform(0.8, 1.2, (T, H // 128)))
    elif fmt == "fp8_token":
        a_s = 2.0 ** -rng.integers(2, 9, size=T) * rng.uniform(0.8, 1.2, T)
    else:
        a_s = np.array([0.003])
    a_s = a_s.astype(np.float32)
    w13 = codes(E, 2 * I, H)
    w13_s = (rng.uniform(0.5, 1.5, (E, 2 * I // 128, H // 128)) * 2.0 ** -10).astype(np.float32)
    w2 = codes(E, H, I)
    w2_s = (rng.uniform(0.5, 1.5, (E, H // 128, I // 128)) * 2.0 ** -8).astype(np.float32)
    ids = np.array([[2, 0], [1, 2], [0, 1]], dtype=np.int32)[:T, :k]
    return a1q, a_s, w13, w13_s, w2, w2_s, ids


def _scalar_rows(a1q, a_s, w13, w13_s, w2, w2_s, ids, fmt):
    """The expert rows y[t*k + j] (unrounded fp64, before the final bf16 rounding)
    written out token by token."""
    T, H = a1q.shape
    k = ids.shape[1]
    I = w2.shape[2]
    KB, IB = H // 128, I // 128

    def a_scale(t, kb):
        return float(a_s[t, kb]) if fmt == "fp8" else float(a_s[t] if fmt == "fp8_token" else a_s[0])

    # GEMM1 and the activation, per slot (fp64 sums of 128-deep K blocks)
    h = {}
    for t in range(T):
        x = E4M3[a1q[t]]
        for j in range(k):
            e = int(ids[t, j])
            gu = np.zeros(2 * I)
            for n in range(2 * I):
                wrow = E4M3[w13[e, n]]
                acc = 0.0
                for kb in range(KB):
                    sl = slice(128 * kb, 128 * kb + 128)
                    acc += a_scale(t, kb) * float(w13_s[e, n // 128, kb]) * float(np.dot(x[sl], wrow[sl]))
                gu[n] = acc
            h[(t, j)] = [_silu_mul(gu[i], gu[I + i]) for i in range(I)]
    # the intermediate in the activations' format
    hq, hs = {}, {}
    if fmt == "fp8":          # G(128) from fp32 h
        for key, v in h.items():
            v32 = [np.float32(x) for x in v]
            cs, ss = [], []
            for ib in range(IB):
                c, s = _quant_group(v32[128 * ib:128 * ib + 128])
                cs += c
                ss.append(float(s))
            hq[key], hs[key] = cs, ss
    elif fmt == "fp8_token":  # per row from bf16 h
        for key, v in h.items():
            c, s = _quant_group([np.float32(_bf16(x)) for x in v])
            hq[key], hs[key] = c, [float(s)] * IB
    else:                     # one scale over every row's bf16 h
        allv = {key: [np.float32(_bf16(x)) for x in v] for key, v in h.items()}
        f32 = np.float32
        amax = f32(max(abs(float(x)) for v in allv.values() for x in v))
        s = f32(max(amax, f32(1e-10)) / f32(448.0))
        for key, v in allv.items():
            hq[key] = [_e4m3_code(float(f32(x / s))) for x in v]
            hs[key] = [float(s)] * IB
    # GEMM2, token-major rows f = t*k + j
    y = np.zeros((T * k, H))
    for t in range(T):
        for j in range(k):
            e = int(ids[t, j])
            hv = E4M3[np.array(hq[(t, j)], dtype=np.uint8)]
            for n in range(H):
                wrow = E4M3[w2[e, n]]
                acc = 0.0
                for ib in range(IB):
                    sl = slice(128 * ib, 128 * ib + 128)
                    acc += hs[(t, j)][ib] * float(w2_s[e, n // 128, ib]) * float(np.dot(hv[sl], wrow[sl]))
                y[t * k + j, n] = acc
    return y


def _oracle_rows(a1q, a_s, w13, w13_s, w2, w2_s, ids, fmt):
    al = moe_ref.align(torch.from_numpy(ids), w13.shape[0], 128)
    return moe_ref.experts(torch.from_numpy(a1q), torch.from_numpy(a_s), torch.from_numpy(w13),
                           torch.from_numpy(w13_s), torch.from_numpy(w2), torch.from_numpy(w2_s), al,
                           ids.shape[1], fmt).numpy()


def _agree(got, y_unrounded):
    """The oracle stores y in bf16: every element must be the bf16 rounding of the
    scalar sum (within the fp64 noise of a different summation order)."""
    half = np.array([abs(_bf16(v) - v) for v in y_unrounded.ravel()]).reshape(y_unrounded.shape)
    ulp = np.array([2.0 ** (math.frexp(v)[1] - 8) if v else 0.0 for v in y_unrounded.ravel()]).reshape(
        y_unrounded.shape)
    err = np.abs(got - y_unrounded)
    return bool(np.all(err <= half + 1e-9 * ulp)), float((err / np.maximum(ulp, 1e-300)).max())


@pytest.fixture(scope="module")
def layers():
    out = {}
    for fmt in ("fp8", "fp8_token", "fp8_tensor"):
        inp = _layer(fmt=fmt)
        out[fmt] = (inp, _scalar_rows(*inp, fmt))
    return out


@pytest.mark.parametrize("fmt", ["fp8", "fp8_token", "fp8_tensor"])
def test_fp8_experts_equal_scalar_rederivation(layers, fmt):
    inp, y = layers[fmt]
    ok, worst = _agree(_oracle_rows(*inp, fmt), y)
    assert ok, f"{fmt}: oracle differs from the scalar layer by up to {worst:.3f} bf16 ulp"


def test_fp8_inputs_exercise_the_requant_precision(layers):
    # the pin below is only meaningful if the G(128) intermediate, rounded through
    # bf16 instead of fp32, lands on other codes for some elements
    inp, _ = layers["fp8"]
    a1q, a_s, w13, w13_s, w2, w2_s, ids = inp
    al = moe_ref.align(torch.from_numpy(ids), 3, 128)
    A = moe_ref._act64(torch.from_numpy(a1q), torch.from_numpy(a_s), np.array([0]), "fp8")
    W = torch.from_numpy(moe_ref.dequant_weight_block(w13[ids[0, 0]], w13_s[ids[0, 0]]))
    h = moe_ref.silu_and_mul(A @ W.T).numpy()
    q32, _ = moe_ref.quantize_fp8_g128(codecs.round_fp32(h))
    q16, _ = moe_ref.quantize_fp8_g128(codecs.round_bf16(h))
    assert (q32 != q16).sum() >= 3
    assert int(al.expert_offsets[-1]) == 6


def test_pin_fails_if_intermediate_is_requantised_from_bf16(layers, monkeypatch):
    inp, y = layers["fp8"]
    real = moe_ref.quantize_fp8_g128

    def from_bf16(x64, group=128):
        return real(codecs.round_bf16(x64), group)

    monkeypatch.setattr(moe_ref, "quantize_fp8_g128", from_bf16)
    ok, _ = _agree(_oracle_rows(*inp, "fp8"), y)
    assert not ok


def test_pin_fails_if_scales_are_indexed_by_sorted_row(layers, monkeypatch):
    inp, y = layers["fp8"]
    real = moe_ref._act64

    def by_position(a1q, a1q_scale, rows, quant):
        v = real(a1q, None if a1q_scale is None else a1q_scale, rows, "bf16" if a1q_scale is None else quant)
        sc = moe_ref._np(a1q_scale)
        wrong = sc[np.arange(len(rows)) % sc.shape[0]]
        return torch.from_numpy(moe_ref.dequant_fp8(moe_ref._np(a1q)[rows].astype(np.uint8), wrong, quant))

    monkeypatch.setattr(moe_ref, "_act64", by_position)
    ok, _ = _agree(_oracle_rows(*inp, "fp8"), y)
    assert not ok


def test_fp8_experts_with_unit_scales_match_decoded_matmul():
    # with all scales 1 and codes whose products stay exact, GEMM1 is a plain matmul of
    # the decoded tables (numpy), and G(128) of an h that is already on the E4M3 grid
    # times a power of two reproduces it exactly
    rng = np.random.default_rng(3)
    A = rng.integers(0, 256, size=(4, 128)).astype(np.uint8)
    A[(A & 0x7F) == 0x7F] = 0x38
    W = rng.integers(0, 256, size=(256, 128)).astype(np.uint8)
    W[(W & 0x7F) == 0x7F] = 0x38
    Aq = moe_ref._act64(torch.from_numpy(A), torch.ones((4, 1), dtype=torch.float32), np.arange(4), "fp8")
    Wq = moe_ref.dequant_weight_block(W, np.ones((2, 1), dtype=np.float32))
    assert np.array_equal((Aq @ torch.from_numpy(Wq).T).numpy(), E4M3[A] @ E4M3[W].T)
    grid = np.array([[E4M3[c] * 2.0 ** -5 for c in rng.integers(0, 0x7E, size=128)]])
    grid[0, 7] = 448.0 * 2.0 ** -5  # the group's amax is the top code
    q, s = moe_ref.quantize_fp8_g128(grid)
    assert float(s[0, 0]) == 2.0 ** -5
    assert np.array_equal(E4M3[q[0]] * 2.0 ** -5, grid[0])
