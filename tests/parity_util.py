"""Tolerance checks shared by the GPU parity tests.

bf16 outputs: relative Frobenius error <= 5e-3 and, element by element,
|gpu - ref| <= 1e-2 * RMS(ref) + slack, against the fp64 oracle.  `slack` is
what the bf16 storage points of the method can cost on their own: half a bf16
ulp of the output, plus (for a whole layer) one bf16 ulp of every stored bf16
operand that enters the output linearly -- the expert rows y times their
weights and the shared-expert row -- scaled by the RMSNorm factor when there
is one.  Two correct implementations that accumulate in different orders can
round a stored y element to neighbouring bf16 values; the bound admits that
and nothing more.
fp8 paths: relative Frobenius error <= 3e-2 against an oracle that applies
the same quantisation steps; and, stage by stage, the GPU's quantised
intermediate against the oracle's quantisation of its own h (each element a
correct E4M3 code of h, rare flips at rounding boundaries), then the second GEMM
against the oracle's second GEMM applied to the GPU's own intermediate at the
bf16 bound.
"""
import numpy as np
import torch

from oracle import codecs, moe_ref

E4M3_VALUES = codecs.e4m3_decode(np.arange(256))


def to64(x):
    if isinstance(x, torch.Tensor):
        return x.detach().cpu().to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def half_ulp_bf16(r):
    a = np.abs(r)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.ldexp(1.0, (e - 8).astype(np.int64)), 0.0)


def stats(gpu, ref):
    g, r = to64(gpu), to64(ref)
    rms = float(np.sqrt(np.mean(r * r))) if r.size else 0.0
    nrm = float(np.linalg.norm(r))
    rel = float(np.linalg.norm(g - r) / nrm) if nrm > 0 else float(np.linalg.norm(g - r))
    maxabs = float(np.abs(g - r).max()) if r.size else 0.0
    return g, r, rms, rel, maxabs


def ulp_bf16(r):
    return 2.0 * half_ulp_bf16(r)


def check_bf16(gpu, ref, what="", slack=None):
    g, r, rms, rel, maxabs = stats(gpu, ref)
    bound = 1e-2 * rms + half_ulp_bf16(r) + (0.0 if slack is None else slack)
    bad = np.abs(g - r) > bound
    assert rel <= 5e-3, f"{what}: relative Frobenius {rel:.3e} > 5e-3"
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements beyond 1e-2*RMS + rounding slack "
                           f"(max |err| {maxabs:.3e}, RMS {rms:.3e}, max |err|/RMS {maxabs / max(rms, 1e-30):.3e})")
    return rel, maxabs / max(rms, 1e-30)


def check_fp8(gpu, ref, what="", tol=3e-2):
    g, r, rms, rel, maxabs = stats(gpu, ref)
    assert rel <= tol, f"{what}: relative Frobenius {rel:.3e} > {tol}"
    return rel, maxabs / max(rms, 1e-30)


def check_nvfp4(gpu, ref, what="", rel_tol=5e-3, frac_tol=1e-3):
    """NVFP4 experts: both sides apply the same quantisation steps, so the output
    matches like a bf16 path (relative Frobenius <= 5e-3; elements within
    1e-2*RMS + a bf16 ulp) except where the GPU's fp32 accumulation moved a stored
    bf16 h element to its neighbour and that neighbour rounds to another E2M1 code
    (or group scale) than the oracle's: such a flip moves whole output rows by one
    code step of one h element.  Those rows may exceed the element bound; they
    must be a rare fraction (<= 1e-3 of the elements)."""
    g, r, rms, rel, maxabs = stats(gpu, ref)
    bound = 1e-2 * rms + 2.0 * half_ulp_bf16(r)
    bad = np.abs(g - r) > bound
    frac = float(bad.mean()) if bad.size else 0.0
    assert rel <= rel_tol, f"{what}: relative Frobenius {rel:.3e} > {rel_tol}"
    assert frac <= frac_tol, (f"{what}: {int(bad.sum())} elements ({frac:.2e}) beyond 1e-2*RMS + rounding slack "
                              f"(max |err|/RMS {maxabs / max(rms, 1e-30):.3e})")
    return rel, maxabs / max(rms, 1e-30)


def e4m3_step(v):
    """Spacing of E4M3 values at magnitude |v| (normal range from 2^-6, subnormal below)."""
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a >= 2.0 ** -6, np.ldexp(1.0, (e - 3).astype(np.int64)), 2.0 ** -9)


def fp8_row_scales(hs, quant, rows, ngroups):
    """Per-element-group scales [len(rows), ngroups] of the GPU's intermediate from the
    workspace view (G(128): [I/128, S] transposed; "A"/"T": [S])."""
    hs = hs.detach().cpu().numpy().astype(np.float64)
    if quant == "fp8":
        return hs[:, rows].T
    return np.repeat(hs[rows][:, None], ngroups, axis=1)


def oracle_requant(h_ref, quant, h_all=None):
    """The oracle's quantisation of its own intermediate (fp64 h rows): G(128) from
    fp32 h, "A" per row from bf16 h, "T" one scale over `h_all` (every row of every
    expert, bf16).  Returns (codes [R, I], per-group scales [R, I/128])."""
    R, I = h_ref.shape
    if quant == "fp8":
        q, s = moe_ref.quantize_fp8_g128(codecs.round_fp32(h_ref))
        return q, s.astype(np.float64)
    if quant == "fp8_token":
        q, s = moe_ref.quantize_fp8_token(codecs.round_bf16(h_ref))
        return q, np.repeat(s.astype(np.float64)[:, None], I // 128, axis=1)
    _, s = moe_ref.quantize_fp8_tensor(codecs.round_bf16(h_all if h_all is not None else h_ref))
    q = codecs.e4m3_encode(codecs.round_fp32(codecs.round_bf16(h_ref) / float(s[0])))
    return q, np.full((R, I // 128), float(s[0]))


def check_fp8_intermediate(codes_gpu, scales_gpu, h_ref, quant, what, h_all=None, flip_frac=1e-2):
    """GPU intermediate (E4M3 codes [R, I] and per-group scales [R, I/128]) against the
    oracle's quantisation of its own h (fp64 [R, I]).  Both quantise h with the same
    rule; they see h through different fp32 summation orders, so a scale may differ in
    its last bits and an element on a rounding boundary may take the neighbouring code.
    Required: every scale within 2^-7 relative of the oracle's; every GPU element within
    half an E4M3 step (at the oracle's magnitude, plus 2^-10 relative for the h
    difference, 2^-8 for the bf16 h of "A"/"T") of the oracle's unquantised h; codes that differ from the oracle's are
    neighbours and at most `flip_frac` of the elements.  A mis-indexed scale or row moves
    h by far more and flips a large share of the codes.  Returns (flips, elements,
    largest scale difference)."""
    codes_gpu = np.asarray(codes_gpu).astype(np.uint8)
    R, I = codes_gpu.shape
    q_ref, s_ref = oracle_requant(h_ref, quant, h_all)
    s_gpu = np.asarray(scales_gpu, dtype=np.float64)
    sdiff = float(np.abs(s_gpu / s_ref - 1.0).max()) if R else 0.0
    assert sdiff <= 2.0 ** -7, f"{what}: intermediate scales differ by up to {sdiff:.3e} relative"
    sg = np.repeat(s_gpu, 128, axis=1)
    v_gpu = E4M3_VALUES[codes_gpu] * sg
    ratio = h_ref / np.repeat(s_ref, 128, axis=1)
    # the h difference: fp32 summation order (G(128)); plus a bf16 rounding of h ("A"/"T")
    rel = 2.0 ** -10 if quant == "fp8" else 2.0 ** -8
    bound = 0.5 * e4m3_step(np.minimum(np.abs(ratio), 448.0)) * sg * 1.001 + rel * np.abs(h_ref) + 1e-30
    over = np.abs(v_gpu - np.clip(h_ref, -448.0 * sg, 448.0 * sg)) > bound
    assert not over.any(), (f"{what}: {int(over.sum())} intermediate elements are not a rounding of h "
                            f"(worst |err|/bound {float((np.abs(v_gpu - h_ref) / bound).max()):.2f})")
    flips = E4M3_VALUES[codes_gpu] != E4M3_VALUES[q_ref]  # (+0 and -0 are one value)
    nflip = int(flips.sum())
    if nflip:
        vr = E4M3_VALUES[q_ref][flips]
        vg = E4M3_VALUES[codes_gpu][flips]
        assert np.all(np.abs(vg - vr) <= e4m3_step(np.maximum(np.abs(vr), np.abs(vg))) * 1.0001), \
            f"{what}: a flipped intermediate code is not a neighbour of the oracle's"
    assert nflip <= max(4, flip_frac * codes_gpu.size), f"{what}: {nflip} of {codes_gpu.size} intermediate codes flipped"
    print(f"{what}: intermediate {nflip} flips of {codes_gpu.size} codes, scales within {sdiff:.2e}")
    return nflip, codes_gpu.size, sdiff
