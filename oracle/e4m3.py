"""Exact decoding of FP8 e4m3 codes (test infrastructure only).

Format (the "FN" variant used for DeepSeek-V3.2 FP8 activations and caches):
1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent field 0
encodes subnormals m * 2^-9; the codes 0x7F and 0xFF are NaN; there are no
infinities; the largest finite magnitude is 1.75 * 2^8 = 448.

Every finite value is an integer multiple of 2^-9 (the smallest subnormal), so
the decoder returns integers in units of 2^-9: |units| <= 448 * 512 = 229376.
"""
from __future__ import annotations

import numpy as np

UNIT_LOG2 = -9          # one unit = 2^-9
MAX_UNITS = 448 * 512   # 229376


def decode_units(code: int):
    """Decode one byte to an integer number of 2^-9 units; None for NaN."""
    code = int(code) & 0xFF
    sign = -1 if (code >> 7) & 1 else 1
    exp = (code >> 3) & 0xF
    man = code & 0x7
    if exp == 0xF and man == 0x7:
        return None  # NaN
    if exp == 0:
        # subnormal: (man / 8) * 2^(1 - 7) = man * 2^-9
        return sign * man
    # normal: (1 + man / 8) * 2^(exp - 7) = (8 + man) * 2^(exp - 10)
    #       = (8 + man) * 2^(exp - 1) units of 2^-9
    return sign * (8 + man) * (1 << (exp - 1))


def table_units() -> tuple[np.ndarray, np.ndarray]:
    """(int64[256] units, bool[256] is_nan); NaN entries hold 0 in units."""
    units = np.zeros(256, np.int64)
    nan = np.zeros(256, bool)
    for c in range(256):
        u = decode_units(c)
        if u is None:
            nan[c] = True
        else:
            units[c] = u
    return units, nan


def table_f64() -> np.ndarray:
    """float64[256] real values (NaN for the two NaN codes)."""
    units, nan = table_units()
    vals = units.astype(np.float64) * 2.0 ** UNIT_LOG2
    vals[nan] = np.nan
    return vals


_UNITS, _NAN = table_units()


def decode_array_units(codes: np.ndarray) -> np.ndarray:
    """Vectorised decode of a uint8 array to int64 units (NaN codes rejected)."""
    codes = np.asarray(codes, dtype=np.uint8)
    if _NAN[codes].any():
        raise ValueError("e4m3 NaN code in input; the indexer is undefined on NaN")
    return _UNITS[codes]
