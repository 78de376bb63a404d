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
the same quantisation steps.
"""
import numpy as np
import torch


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
