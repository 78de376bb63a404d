"""Pins of the oracle's NVFP4 experts path (CPU only).

NVFP4 here is the finalize page's packed encoding ("[flashinfer] MoE Finalize +
AllReduce fusion", introduction): E2M1 codes (OCP Microscaling Formats v1.0,
section 5.3.3) in pairs, one E4M3 scale per 16 elements and an fp32 global
scale; the experts table of "Fused MoE Kernel Features" lists it as a
quantisation type of the cutlass_fp4 and trtllm experts.  The checks below use
a scalar re-derivation written from those definitions (value tables and a
nearest-value search, not the oracle's codecs), library matmuls, and exact
scaling invariants.
"""
import math
import os

import numpy as np
import torch

from mixture_experts_layer_tokens_gb300.inputs import CONFIGS, make_inputs, scaled
from oracle import codecs, moe_ref

GOLD = os.path.join(os.path.dirname(__file__), "golden")

# E2M1 magnitudes of codes 0..7 (1 sign, 2 exponent, 1 mantissa bit; bias 1)
E2M1_MAG = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _e2m1(c):
    return (-1.0 if c & 8 else 1.0) * E2M1_MAG[c & 7]


def _e4m3(c):
    # sign bit 0 only (block scales are positive); bias 7, subnormals at exponent 0
    e, m = (c >> 3) & 15, c & 7
    return (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)


E4M3_POS = [(c, _e4m3(c)) for c in range(0x7F)]  # 0x7f is NaN


def _nearest(t, table):
    """Code of the nearest table value to t >= 0, ties to the even code, saturating."""
    best = None
    for c, v in table:
        d = abs(v - t)
        if best is None or d < best[0] or (d == best[0] and c % 2 == 0):
            best = (d, c)
    return best[1]


def _bf16_rn(x):
    """Round-to-nearest-even to 8 significant bits (bf16) of a finite fp64 number."""
    if x == 0.0:
        return 0.0
    m, e = math.frexp(x)              # x = m 2^e, 0.5 <= |m| < 1
    s = m * 256.0                     # 8 significant bits above the point
    r = math.floor(s)
    f = s - r
    if f > 0.5 or (f == 0.5 and r % 2 == 1):
        r += 1
    return math.ldexp(r / 256.0, e)


def _quant16(vals, g):
    """One 16-element group in fp32 decision steps -> (codes, scale code)."""
    f32 = np.float32
    amax = max(abs(v) for v in vals)
    t = float(f32(amax) / (f32(6.0) * f32(g)))
    sc = _nearest(t, E4M3_POS)
    d = f32(_e4m3(sc)) * f32(g)
    codes = []
    for v in vals:
        r = float(f32(v) / d) if d > 0 else 0.0
        mag = _nearest(abs(r), list(enumerate(E2M1_MAG)))
        codes.append((8 if r < 0 else 0) | mag)
    return codes, sc


def _deq_row(packed_row, sf_row, g):
    out = []
    for i, b in enumerate(packed_row):
        for c in (int(b) & 15, int(b) >> 4):            # element 2i in the low nibble
            out.append(_e2m1(c))
    return [v * _e4m3(int(sf_row[j // 16])) * g for j, v in enumerate(out)]


def _brute_experts(a1q, a1sf, ga, w13, w13sf, g13, w2, w2sf, g2, gh, ids):
    T, k = ids.shape
    H = a1q.shape[1] * 2
    y = np.zeros((T * k, H))
    for t in range(T):
        x = _deq_row(a1q[t], a1sf[t], ga)
        for j in range(k):
            e = int(ids[t, j])
            W13 = [_deq_row(w13[e][n], w13sf[e][n], float(g13[e])) for n in range(w13.shape[1])]
            I = len(W13) // 2
            gu = [sum(x[c] * W13[n][c] for c in range(H)) for n in range(2 * I)]
            h = [_bf16_rn(gu[n] / (1.0 + math.exp(-gu[n])) * gu[I + n]) for n in range(I)]
            hq = []
            for g0 in range(0, I, 16):
                codes, sc = _quant16(h[g0:g0 + 16], gh)
                hq += [_e2m1(c) * _e4m3(sc) * gh for c in codes]
            for n in range(H):
                w = _deq_row(w2[e][n], w2sf[e][n], float(g2[e]))
                y[t * k + j, n] = _bf16_rn(sum(hq[c] * w[c] for c in range(I)))
    return y


def _tiny(seed=0, T=3, E=2, k=2, H=32, I=32):
    cfg = scaled(CONFIGS["tiny"], T=T, H=H, I=I, E=E, top_k=k, quant="nvfp4")
    inp = make_inputs(cfg, seed=seed)
    g = torch.Generator().manual_seed(seed + 100)
    ids = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).to(torch.int32)
    return cfg, inp, ids


def test_fp32_quantizer_reproduces_the_golden_group():
    lines = {l.split()[0]: l.split()[1:] for l in open(os.path.join(GOLD, "nvfp4_group.txt")) if not l.startswith("#")}
    x = np.array([[float(v) for v in lines["input"]]])
    packed, sf = moe_ref.nvfp4_quantize_fp32(x, 1.0)
    assert sf.tolist() == [[int(lines["scale"][0], 16)]]
    assert packed[0].tolist() == [int(v, 16) for v in lines["packed"]]


def test_fp32_quantizer_matches_scalar_rederivation():
    rng = np.random.default_rng(7)
    x = codecs.round_bf16(rng.normal(size=(6, 64)) * rng.choice([0.01, 1.0, 30.0], size=(6, 1)))
    x[2, 16:32] = 0.0
    for g in (2.0 ** -8, 0.37, 1.0):
        packed, sf = moe_ref.nvfp4_quantize_fp32(x, g)
        for r in range(x.shape[0]):
            for g0 in range(0, 64, 16):
                codes, sc = _quant16(list(x[r, g0:g0 + 16]), g)
                assert sf[r, g0 // 16] == sc
                got = [(int(packed[r, (g0 + i) // 2]) >> (4 * ((g0 + i) % 2))) & 15 for i in range(16)]
                # +-0 codes may differ in sign only
                assert [_e2m1(c) for c in got] == [_e2m1(c) for c in codes]


def test_fp32_quantizer_error_bound():
    x = codecs.round_bf16(np.random.default_rng(8).normal(size=(8, 128)) * 3.0)
    g = 2.0 ** -7
    packed, sf = moe_ref.nvfp4_quantize_fp32(x, g)
    deq = moe_ref.nvfp4_dequantize(packed, sf, g)
    d = np.repeat(codecs.e4m3_decode(sf), 16, 1) * g          # one unit of the group's scale
    a = np.abs(x) / d
    half_step = np.where(a < 2, 0.25, np.where(a < 4, 0.5, 1.0)) * d
    assert (np.abs(deq - x) <= half_step + np.maximum(np.abs(x) - 6 * d, 0) + 1e-12).all()


def test_prepare_nvfp4_weight_on_input_then_quantise():
    cfg = scaled(CONFIGS["llama1"], T=5, H=64, I=32, E=4, shared_I=0, quant="nvfp4")
    inp = make_inputs(cfg)
    w = torch.rand((5, 1), generator=torch.Generator().manual_seed(3))
    p, s = moe_ref.prepare_nvfp4(inp.a1, w, True, 2.0 ** -8)
    xb, _ = moe_ref.prepare(inp.a1, w, True, "bf16")          # the pinned bf16 weighting
    p2, s2 = moe_ref.nvfp4_quantize_fp32(xb.double().numpy(), 2.0 ** -8)
    assert np.array_equal(p.numpy(), p2) and np.array_equal(s.numpy(), s2)


def test_experts_nvfp4_matches_scalar_brute_force():
    cfg, inp, ids = _tiny()
    ga, gh = 2.0 ** -8, 2.0 ** -7
    a1q, a1sf = moe_ref.prepare_nvfp4(inp.a1, None, False, ga)
    al = moe_ref.align(ids, cfg.E, 128)
    y = moe_ref.experts_nvfp4(a1q, a1sf, ga, inp.w13, inp.w13_scale, inp.extra["w13_gscale"], inp.w2,
                              inp.w2_scale, inp.extra["w2_gscale"], gh, al, cfg.top_k)
    yb = _brute_experts(a1q.numpy(), a1sf.numpy(), ga, inp.w13.numpy(), inp.w13_scale.numpy(),
                        inp.extra["w13_gscale"].double().numpy(), inp.w2.numpy(), inp.w2_scale.numpy(),
                        inp.extra["w2_gscale"].double().numpy(), gh, ids.numpy())
    assert np.array_equal(y.numpy(), yb)


def test_experts_nvfp4_unit_scales_gemm1_is_plain_matmul():
    cfg, inp, ids = _tiny(seed=1, T=4, E=3, k=2, H=64, I=48)
    one = 0x38                                                  # E4M3 code of 1.0
    inp.w13_scale[:] = one
    a1q = torch.randint(0, 256, (4, 32), generator=torch.Generator().manual_seed(5), dtype=torch.int32).to(torch.uint8)
    a1sf = torch.full((4, 4), one, dtype=torch.uint8)
    al = moe_ref.align(ids, cfg.E, 128)
    ones = torch.ones(3)
    _, h = moe_ref.experts_nvfp4(a1q, a1sf, 1.0, inp.w13, inp.w13_scale, ones, inp.w2, inp.w2_scale,
                                 inp.extra["w2_gscale"], 2.0 ** -7, al, cfg.top_k, return_h=True)
    table = np.array([_e2m1(c) for c in range(16)])
    unpack = lambda b: np.stack([table[b & 15], table[b >> 4]], -1).reshape(b.shape[0], -1)
    X = unpack(a1q.numpy())
    offs, order = al.expert_offsets.numpy(), al.sorted_slot.numpy()
    for e in range(3):
        p0, p1 = int(offs[e]), int(offs[e + 1])
        gu = X[order[p0:p1] // 2] @ unpack(inp.w13[e].numpy()).T
        g, u = gu[:, :48], gu[:, 48:]
        assert np.allclose(h[p0:p1], g / (1 + np.exp(-g)) * u, rtol=1e-13, atol=1e-13)


def test_experts_nvfp4_scale_invariances():
    cfg, inp, ids = _tiny(seed=2, T=6, E=3, k=2, H=64, I=64)
    ga, gh = 2.0 ** -8, 2.0 ** -7
    a1q, a1sf = moe_ref.prepare_nvfp4(inp.a1, None, False, ga)
    al = moe_ref.align(ids, cfg.E, 128)
    g13, g2 = inp.extra["w13_gscale"], inp.extra["w2_gscale"]
    run = lambda gh_, g2_: moe_ref.experts_nvfp4(a1q, a1sf, ga, inp.w13, inp.w13_scale, g13, inp.w2,
                                                 inp.w2_scale, g2_, gh_, al, cfg.top_k)
    y = run(gh, g2)
    # the intermediate's global scale only moves its block scales by a power of two (as long
    # as they stay normal and below the E4M3 maximum: h of this case keeps amax/(6 g) in
    # [2^-5, 224] for both factors)
    _, h = moe_ref.experts_nvfp4(a1q, a1sf, ga, inp.w13, inp.w13_scale, g13, inp.w2, inp.w2_scale, g2, gh, al,
                                 cfg.top_k, return_h=True)
    am = np.abs(h).reshape(h.shape[0], -1, 16).max(axis=2) / (6 * gh)
    assert am.min() > 2.0 ** -5 and am.max() < 224
    assert torch.equal(run(gh * 2, g2), y) and torch.equal(run(gh / 2, g2), y)
    # expert 1's second-matrix global scale scales exactly its rows
    g2b = g2.clone()
    g2b[1] *= 2
    y2 = run(gh, g2b)
    rows1 = torch.from_numpy(al.sorted_slot.numpy()[int(al.expert_offsets[1]):int(al.expert_offsets[2])].astype(np.int64))
    mask = torch.zeros(y.shape[0], dtype=torch.bool)
    mask[rows1] = True
    assert torch.equal(y2[mask], 2 * y[mask]) and torch.equal(y2[~mask], y[~mask])
