"""Number formats of the W4A4 layer, decoded from their bit definitions, and
round-to-nearest-even onto each grid.

Formats named by the pages: NVFP4 -- 4-bit e2m1 values with one scale per
16 elements ([dothoosh], "quantization_config" block: precision "nvfp4",
group_size 16) -- and the 16-bit low-rank branch kept in the compute dtype
bfloat16 ([dothoosh], same block: compute_dtype "bfloat16"; [hamidun-ar],
"What are Nunchaku and SVDQuant": "a small 16-bit low-rank branch").

Definitions used (the formats' own, not the pages'):
  e2m1  sign | 2 exponent bits (bias 1) | 1 mantissa bit.  Exponent field 0
        is subnormal (value m * 2^-1 ... i.e. 0 or 0.5); otherwise
        2^(e-1) * (1 + m/2).  No inf, no NaN.  Magnitudes, codes 0..7:
        0, 0.5, 1, 1.5, 2, 3, 4, 6.
  e4m3  (OCP 8-bit floating point, "FN" variant) sign | 4 exponent bits
        (bias 7) | 3 mantissa bits.  Exponent field 0 is subnormal
        (m/8 * 2^-6); S.1111.111 is NaN; there is no inf; max 448.
  bf16  the upper half of an IEEE binary32: 8 significant bits, same
        exponent range as binary32.

Rounding: to the nearest grid value; an exact tie goes to the code whose
mantissa LSB (bit 0) is 0; magnitudes above the largest finite value
saturate to it (satfinite).  This is the layer's fixed rule.
"""
from __future__ import annotations

import numpy as np

# --------------------------------------------------------------------------
# decode tables, built from the bit fields
# --------------------------------------------------------------------------


def e2m1_decode_code(code: int) -> float:
    """Value of a 4-bit e2m1 code, from sign/exponent/mantissa fields."""
    code = int(code) & 0xF
    sign = -1.0 if (code >> 3) & 1 else 1.0
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:
        mag = m * 0.5  # subnormal: m * 2^(1-bias) * 2^-1, bias 1
    else:
        mag = (2.0 ** (e - 1)) * (1.0 + m / 2.0)
    return sign * mag


def e4m3_decode_byte(b: int) -> float:
    """Value of an e4m3 (OCP FN) byte, from its fields; NaN for S.1111.111."""
    b = int(b) & 0xFF
    sign = -1.0 if (b >> 7) & 1 else 1.0
    e = (b >> 3) & 0xF
    m = b & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        mag = (m / 8.0) * 2.0 ** (1 - 7)
    else:
        mag = (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return sign * mag


E2M1_TABLE = np.array([e2m1_decode_code(c) for c in range(16)], dtype=np.float64)
E4M3_TABLE = np.array([e4m3_decode_byte(b) for b in range(256)], dtype=np.float64)

# non-negative finite magnitudes in code order (codes 0..7 / 0x00..0x7E)
_E2M1_MAGS = E2M1_TABLE[:8].copy()
_E4M3_MAGS = E4M3_TABLE[:0x7F].copy()
assert np.all(np.diff(_E2M1_MAGS) > 0) and np.all(np.diff(_E4M3_MAGS) > 0)


def _rne_to_magnitude_codes(a: np.ndarray, mags: np.ndarray) -> np.ndarray:
    """Index of the nearest entry of the increasing grid ``mags`` for each
    non-negative float64 ``a``; exact ties pick the even index (mantissa LSB
    0, which for these formats is bit 0 of the code); values beyond the last
    entry saturate to it.  Grid midpoints are dyadic with few bits, so they
    and the comparisons below are exact in float64."""
    a = np.asarray(a, dtype=np.float64)
    if np.any(np.isnan(a)) or np.any(a < 0):
        raise ValueError("magnitudes must be non-negative and not NaN")
    mids = (mags[:-1] + mags[1:]) * 0.5
    lt = np.searchsorted(mids, a, side="left")   # number of midpoints < a
    le = np.searchsorted(mids, a, side="right")  # number of midpoints <= a
    idx = lt.copy()
    tie = le != lt                               # a equals mids[lt]
    # tie between lt and lt+1: take the even code
    idx[tie] = np.where(lt[tie] % 2 == 0, lt[tie], lt[tie] + 1)
    return idx.astype(np.int64)


def rne_e2m1(x: np.ndarray) -> np.ndarray:
    """Round float64 values to e2m1 codes (uint8, 0..15): nearest, ties to
    even, saturating at +-6.  The sign bit of the code is the IEEE sign bit of
    the input, so a negative value that rounds to zero gives 0x8 (-0)."""
    x = np.asarray(x, dtype=np.float64)
    mag = _rne_to_magnitude_codes(np.abs(x), _E2M1_MAGS)
    sign = np.signbit(x).astype(np.int64) << 3
    return (mag | sign).astype(np.uint8)


def rne_e4m3(x: np.ndarray) -> np.ndarray:
    """Round non-negative float64 values to e4m3 bytes (0x00..0x7E): nearest,
    ties to even, saturating at 448 (never NaN)."""
    return _rne_to_magnitude_codes(np.asarray(x, dtype=np.float64), _E4M3_MAGS).astype(np.uint8)


def e2m1_decode(codes: np.ndarray) -> np.ndarray:
    return E2M1_TABLE[np.asarray(codes, dtype=np.int64) & 0xF]


def e4m3_decode(b: np.ndarray) -> np.ndarray:
    return E4M3_TABLE[np.asarray(b, dtype=np.int64) & 0xFF]


# --------------------------------------------------------------------------
# bfloat16 / float16 / float32
# --------------------------------------------------------------------------


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 value (ties to even),
    directly from float64 (no intermediate float32 rounding).  Returns the
    rounded values as float64.  Overflow rounds to +-inf, as IEEE RNE does."""
    x = np.asarray(x, dtype=np.float64)
    out = np.empty_like(x)
    finite = np.isfinite(x)
    out[~finite] = x[~finite]
    xf = x[finite]
    # bfloat16: 8 significant bits; smallest normal 2^-126; subnormal step 2^-133
    m, e = np.frexp(xf)                     # xf = m * 2^e, 0.5 <= |m| < 1
    normal = (e - 1) >= -126
    r = np.empty_like(xf)
    r[normal] = np.ldexp(np.rint(np.ldexp(m[normal], 8)), e[normal] - 8)
    r[~normal] = np.ldexp(np.rint(np.ldexp(xf[~normal], 133)), -133)
    max_bf16 = np.ldexp(255.0, 127 - 7)     # (2 - 2^-7) * 2^127
    r = np.where(np.abs(r) > max_bf16, np.copysign(np.inf, r), r)
    out[finite] = r
    return out


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """uint16 bit patterns of values that are exactly bfloat16."""
    x32 = np.asarray(x, dtype=np.float64).astype(np.float32)
    if not np.array_equal(x32.astype(np.float64), np.asarray(x, dtype=np.float64), equal_nan=True):
        raise ValueError("values are not exactly representable in float32")
    bits = x32.view(np.uint32)
    if np.any(bits & 0xFFFF):
        raise ValueError("values are not exactly representable in bfloat16")
    return (bits >> 16).astype(np.uint16)


def bf16_from_bits(bits: np.ndarray) -> np.ndarray:
    """float64 values of bfloat16 bit patterns."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def round_to_f16(x: np.ndarray) -> np.ndarray:
    """Nearest IEEE binary16 value (ties to even) of float64 values, as float64.
    NumPy's float64 -> float16 cast rounds correctly in one step."""
    return np.asarray(x, dtype=np.float64).astype(np.float16).astype(np.float64)


def f16_bits(x: np.ndarray) -> np.ndarray:
    x16 = np.asarray(x, dtype=np.float64).astype(np.float16)
    if not np.array_equal(x16.astype(np.float64), np.asarray(x, dtype=np.float64)):
        raise ValueError("values are not exactly representable in float16")
    return x16.view(np.uint16)


def f16_from_bits(bits: np.ndarray) -> np.ndarray:
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def round_to_f32(x: np.ndarray) -> np.ndarray:
    """Nearest binary32 value (ties to even) of float64 values, as float64."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)
