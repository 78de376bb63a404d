"""Number-format codecs for the CPU oracle (test infrastructure, not product code).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this package.  Nothing here is shared with the CUDA library.

Formats, each written from its public definition:

* bf16: IEEE-754 binary32 with the low 16 fraction bits dropped (8 significant
  bits, 8 exponent bits, bias 127).  Rounding from a wider value is
  round-to-nearest, ties-to-even, straight from the fp64 value (one rounding).
* fp8 E4M3 ("e4m3fn"): OCP 8-bit Floating Point Specification (OFP8) v1.0,
  Table 1 -- 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits, no
  infinities, S.1111.111 is NaN, largest finite magnitude 448 (S.1111.110),
  smallest normal 2^-6, subnormals m/8 * 2^-6.  The encoder rounds to nearest,
  ties to even, and saturates out-of-range finite values to +-448 ("satfinite").
* fp4 E2M1: OCP Microscaling Formats (MX) v1.0, section 5.3.3 -- 1 sign bit,
  2 exponent bits with bias 1, 1 mantissa bit: magnitudes
  {0, 0.5, 1, 1.5, 2, 3, 4, 6}, code = sign<<3 | magnitude index.  Encoder:
  round to nearest, ties to even code, saturate to +-6.

The NVFP4 packing (two E2M1 codes per byte, 16-element groups sharing one E4M3
scale) is the output format named in the "[flashinfer] MoE Finalize + AllReduce
fusion" page, introduction (optional NVFP4 packed output quantisation).
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E2M1_MAX = 6.0
E2M1_VALUES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)


def _round_half_even(x: np.ndarray) -> np.ndarray:
    # numpy.rint rounds halves to the even integer (IEEE roundTiesToEven).
    return np.rint(x)


def _quantum(a: np.ndarray, mant_bits: int, min_exp: int) -> np.ndarray:
    """Spacing of a binary float grid with `mant_bits` stored fraction bits
    around magnitude `a`, with exponents clamped below at `min_exp`
    (the subnormal range keeps the spacing of the smallest binade)."""
    a = np.where(np.isfinite(a) & (a > 0), a, 1.0)
    e = np.floor(np.log2(a))
    # log2 of a double can be off by one ulp near powers of two: fix it exactly.
    e = np.where(np.ldexp(1.0, e.astype(np.int64)) > a, e - 1, e)
    e = np.where(np.ldexp(1.0, (e + 1).astype(np.int64)) <= a, e + 1, e)
    e = np.maximum(e, min_exp)
    return np.ldexp(1.0, (e - mant_bits).astype(np.int64))


# --------------------------------------------------------------------------- bf16
def round_bf16(x) -> np.ndarray:
    """Round fp64 values to the nearest bf16 value (ties to even), returned as fp64.

    Overflow beyond the largest finite bf16 goes to +-inf, as IEEE rounding does."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    q = _quantum(a, 7, -126)
    r = _round_half_even(a / q) * q
    bf16_max = (2.0 - 2.0 ** -7) * 2.0 ** 127
    # Values at or above the midpoint between bf16_max and 2^128 overflow.
    r = np.where(a >= (2.0 - 2.0 ** -8) * 2.0 ** 127, np.inf, np.minimum(r, bf16_max))
    r = np.where(np.isnan(x), np.nan, r)
    return np.copysign(r, x)


def round_fp32(x) -> np.ndarray:
    """Round fp64 to fp32 (IEEE round-to-nearest-even), returned as fp64."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


# --------------------------------------------------------------------------- e4m3
def e4m3_round(x) -> np.ndarray:
    """Value of the nearest E4M3 number to x (ties to even, saturating to +-448)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    q = _quantum(a, 3, -6)
    r = _round_half_even(a / q) * q
    r = np.minimum(r, E4M3_MAX)
    return np.copysign(r, x)


def e4m3_encode(x) -> np.ndarray:
    """fp64 -> E4M3 code (uint8): round to nearest even, saturate finite and
    infinite inputs to +-448, NaN -> 0x7F (sign kept).  Zero keeps its sign."""
    x = np.asarray(x, dtype=np.float64)
    v = e4m3_round(np.where(np.isnan(x), 0.0, x))
    a = np.abs(v)
    sign = np.signbit(x).astype(np.uint8) << 7
    sub = a < 2.0 ** -6
    # subnormal: value = m * 2^-9, m in 0..7, exponent field 0
    m_sub = np.rint(a / 2.0 ** -9)
    # normal: value = (1 + m/8) * 2^e, exponent field e + 7
    q = _quantum(np.where(sub, 1.0, a), 3, -6)  # = 2^(e-3)
    e = np.log2(q).astype(np.int64) + 3
    m_norm = np.rint(a / q) - 8
    code = np.where(sub, m_sub, ((e + 7) << 3) + m_norm).astype(np.uint8)
    code = code | sign
    return np.where(np.isnan(x), np.uint8(0x7F) | sign, code).astype(np.uint8)


def e4m3_decode(code) -> np.ndarray:
    c = np.asarray(code).astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    ef = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(ef == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, ef - 7))
    val = np.where((ef == 0xF) & (m == 0x7), np.nan, val)
    return s * val


# --------------------------------------------------------------------------- e2m1
def e2m1_round(x) -> np.ndarray:
    """Value of the nearest E2M1 number (ties to even code, saturating to +-6)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    q = _quantum(a, 1, 0)
    r = np.minimum(_round_half_even(a / q) * q, E2M1_MAX)
    return np.copysign(r, x)


def e2m1_encode(x) -> np.ndarray:
    """fp64 -> E2M1 code in the low 4 bits (sign in bit 3)."""
    x = np.asarray(x, dtype=np.float64)
    v = np.abs(e2m1_round(x))
    idx = np.searchsorted(E2M1_VALUES, v)  # v is exactly one of the table entries
    return (idx | (np.signbit(x).astype(np.int64) << 3)).astype(np.uint8)


def e2m1_decode(code) -> np.ndarray:
    c = np.asarray(code).astype(np.int64)
    return np.where(c & 0x8, -1.0, 1.0) * E2M1_VALUES[c & 0x7]
