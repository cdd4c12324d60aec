"""Number formats used by the latent-MoE tail, written from the OCP 8-bit floating point
and OCP microscaling (MX) format definitions.  Test infrastructure: only the tests, the
smoke check and the CPU timing leg of the benchmark use this package.

e4m3 (the "fn" variant): 1 sign, 4 exponent (bias 7), 3 mantissa bits; no infinities;
S.1111.111 is NaN; largest finite 448; smallest normal 2^-6; subnormal step 2^-9.
e2m1: 1 sign, 2 exponent (bias 1), 1 mantissa bit; values 0, 0.5, 1, 1.5, 2, 3, 4, 6.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def _e4m3_value(c: np.ndarray) -> np.ndarray:
    """Value of each code from its bit fields."""
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    sub = m * 2.0 ** -9
    nrm = (1.0 + m / 8.0) * np.exp2((e - 7).astype(np.float64))
    v = np.where(e == 0, sub, nrm) * sign
    return np.where((c & 0x7F) == 0x7F, np.nan, v)


_E4M3_TABLE = _e4m3_value(np.arange(256, dtype=np.int64))


def e4m3_decode(codes) -> np.ndarray:
    """uint8 codes -> float64 values (NaN for the two NaN codes); the 256 values come from
    the bit-field formula above and large arrays are decoded by table lookup."""
    return _E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


def e4m3_encode(v) -> np.ndarray:
    """float values -> e4m3 codes, round to nearest (ties to even code), saturating to
    +-448.  Input values are taken exactly (float32 inputs are exact in float64)."""
    x = np.asarray(v, dtype=np.float64)
    sign = np.signbit(x).astype(np.int64) << 7
    a = np.abs(x)
    # Normal range: a = f * 2^ex with f in [0.5, 1)  ->  a = (1 + frac) * 2^(ex-1).
    f, ex = np.frexp(a)
    e_unb = ex - 1                              # unbiased exponent of a
    mant = np.rint((2.0 * f - 1.0) * 8.0)       # nearest 1/8 step, half to even
    carry = mant >= 8
    e_unb = np.where(carry, e_unb + 1, e_unb)
    mant = np.where(carry, 0, mant)
    normal_code = ((e_unb + 7) << 3) + mant.astype(np.int64)
    # Subnormal range (a < 2^-6): nearest multiple of 2^-9, half to even; a result of 8
    # steps is the smallest normal, whose code (0x08) is the same integer.
    sub_code = np.rint(a * 2.0 ** 9).astype(np.int64)
    code = np.where(a < 2.0 ** -6, sub_code, normal_code)
    code = np.where(a >= E4M3_MAX, 0x7E, np.minimum(code, 0x7E))
    return (code | sign).astype(np.uint8)


def _e2m1_value(c: np.ndarray) -> np.ndarray:
    """Value of each 4-bit code from its bit fields."""
    sign = np.where(c & 0x8, -1.0, 1.0)
    e = (c >> 1) & 0x3
    m = (c & 0x1).astype(np.float64)
    v = np.where(e == 0, m * 0.5, (1.0 + m / 2.0) * np.exp2((e - 1).astype(np.float64)))
    return v * sign


_E2M1_TABLE = _e2m1_value(np.arange(16, dtype=np.int64))


def e2m1_decode(codes) -> np.ndarray:
    """4-bit e2m1 codes (one per array element, 0..15) -> float64, by table lookup of the
    16 values given by the bit-field formula above."""
    return _E2M1_TABLE[np.asarray(codes).astype(np.int64) & 0xF]


def unpack_e2m1(packed) -> np.ndarray:
    """[..., K/2] bytes -> [..., K] codes; element 2i is the low nibble of byte i."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def e2m1_encode(v) -> np.ndarray:
    """float values -> 4-bit e2m1 codes (one per array element): nearest of the eight
    magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6, a tie going to the code with an even mantissa
    bit, saturating at 6.  The sign bit is set only for a non-zero magnitude, so a value
    that rounds to zero has the single code 0.  Magnitudes are located by searching the
    sorted value table; a tie is detected as equal distance to the two neighbours."""
    x = np.asarray(v, dtype=np.float64)
    a = np.minimum(np.abs(x), 6.0)
    mags = _E2M1_TABLE[:8]                          # codes 0..7, increasing magnitudes
    hi = np.clip(np.searchsorted(mags, a, side="left"), 1, 7)
    lo = hi - 1
    d_lo = a - mags[lo]
    d_hi = mags[hi] - a
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(take_hi, hi, lo).astype(np.int64)
    sign = np.where((x < 0) & (code > 0), 8, 0)
    return (code | sign).astype(np.uint8)

