"""OCP 8-bit floating point E4M3 ("FN" variant) codec (oracle, test only).

The pages only fix that an FP8 cache stores one byte per element ("PagedAttention
Memory Management", "Calculating Physical Block Sizes": P_bytes is 1 for FP8).
The format is the OCP 8-bit floating point specification's E4M3: 1 sign bit,
4 exponent bits with bias 7, 3 mantissa bits; exponent field 0 holds the
subnormals m * 2^-9; there are no infinities; S.1111.111 is NaN; the largest
finite magnitude is 1.75 * 2^8 = 448.

Encoding rounds to the nearest representable value, ties to the even code,
and saturates finite magnitudes above 448 to 448 (the "satfinite" reading of
the fp8 cache; NaN stays NaN).  The encoder is the plain definition: it
compares the input with the table of all finite E4M3 values.
"""
from __future__ import annotations

import numpy as np

NAN_CODE = 0x7F
MAX_FINITE = 448.0


def decode_code(code: int) -> float:
    """Value of one E4M3 byte, computed from the bit fields."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return sign * m * 2.0 ** -9
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


# fp64 value of every byte, built from the bit fields above.
DECODE_TABLE = np.array([decode_code(c) for c in range(256)], dtype=np.float64)

# Non-negative finite codes 0x00..0x7E in increasing order of value.
_POS_CODES = np.arange(0x7F, dtype=np.int64)
_POS_VALUES = DECODE_TABLE[:0x7F]
assert np.all(np.diff(_POS_VALUES) > 0)


def decode(codes: np.ndarray) -> np.ndarray:
    """E4M3 bytes -> fp64 values."""
    return DECODE_TABLE[np.asarray(codes, dtype=np.uint8)]


def encode(x: np.ndarray) -> np.ndarray:
    """Values (any float array, compared exactly in fp64) -> E4M3 bytes, round
    to nearest with ties to the even code, saturating at +/-448."""
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(invalid="ignore"):
        return _encode(x)


def _encode(x: np.ndarray) -> np.ndarray:
    out = np.empty(x.shape, dtype=np.uint8)
    flat = x.reshape(-1)
    res = out.reshape(-1)
    mag = np.abs(flat)
    neg = np.signbit(flat)
    nan = np.isnan(flat)
    # index of the largest representable value <= |x|
    lo = np.searchsorted(_POS_VALUES, np.where(nan, 0.0, mag), side="right") - 1
    lo = np.clip(lo, 0, len(_POS_VALUES) - 1)
    hi = np.minimum(lo + 1, len(_POS_VALUES) - 1)
    d_lo = mag - _POS_VALUES[lo]
    d_hi = _POS_VALUES[hi] - mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (_POS_CODES[lo] % 2 == 1))
    code = np.where(pick_hi & (hi != lo), _POS_CODES[hi], _POS_CODES[lo])
    code = np.where(mag >= MAX_FINITE, 0x7E, code)  # saturate finite overflow
    code = code | np.where(neg, 0x80, 0)
    code = np.where(nan, NAN_CODE, code)
    res[:] = code.astype(np.uint8)
    return out


def quantize_fp32(x: np.ndarray, inv_scale) -> np.ndarray:
    """The slot write of an FP8 cache: the fp32 product x * inv_scale (one
    IEEE fp32 rounding), then the E4M3 encoding of that product.  inv_scale
    is a number or an array that broadcasts against x."""
    prod = np.asarray(x, dtype=np.float32) * np.asarray(inv_scale, dtype=np.float32)
    return encode(prod.astype(np.float64))
