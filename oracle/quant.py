"""Symmetric per-row quantisation and the E4M3 code book (test infrastructure).

Follows the low-precision GMM article (pwwt.cn), section 3.2: one scale per
row, ``scale = absmax(row) / 127``, ``q = clamp(round(x / scale), -127, 127)``
for INT8 (per output channel for weights, per token for activations). The
FP8-e4m3 variant (the article names FP8 beside INT8, section 3.1) uses
``scale = absmax / 448`` and rounds ``x / scale`` to the nearest E4M3 value,
ties to even, saturating at +-448.

Readings: the scale and the quotient are float32 operations (the article's
torch code runs in the weights' float32); ``round`` is round-half-to-even
(torch.round); an all-zero row gets scale 1 and codes 0.

The E4M3 code book is the OCP 8-bit floating point (OFP8) definition: sign
bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent field 0 encodes
subnormals m/8 * 2^-6; S.1111.111 is NaN; there are no infinities; the largest
finite magnitude is 448.
"""
from __future__ import annotations

import numpy as np

INT8_QMAX = 127.0
E4M3_MAX = 448.0


def e4m3_decode(code: int) -> float:
    """Value of one E4M3 byte from the OFP8 definition (NaN for the two NaN codes)."""
    code &= 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    exp = (code >> 3) & 0xF
    man = code & 0x7
    if exp == 0xF and man == 0x7:
        return float("nan")
    if exp == 0:
        return sign * (man / 8.0) * 2.0 ** -6
    return sign * (1.0 + man / 8.0) * 2.0 ** (exp - 7)


def _e4m3_table():
    vals = np.array([e4m3_decode(c) for c in range(256)])
    return vals


E4M3_VALUES = _e4m3_table()


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    """Round float values to E4M3 codes: nearest value, ties to the even code, saturate at +-448."""
    v = np.asarray(v, dtype=np.float64)
    pos_codes = np.arange(0, 0x7F)                 # 0x00..0x7E: all non-negative finite codes
    pos_vals = E4M3_VALUES[pos_codes]              # increasing
    a = np.minimum(np.abs(v), E4M3_MAX)
    hi = np.searchsorted(pos_vals, a, side="left")  # first value >= a
    hi = np.clip(hi, 0, len(pos_vals) - 1)
    lo = np.clip(hi - 1, 0, len(pos_vals) - 1)
    d_lo = a - pos_vals[lo]
    d_hi = pos_vals[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (pos_codes[hi] % 2 == 0))
    code = np.where(pick_hi, pos_codes[hi], pos_codes[lo])
    code = np.where(a == pos_vals[hi], pos_codes[hi], code)
    sign = (v < 0) | ((v == 0) & np.signbit(v))
    return (code | np.where(sign, 0x80, 0)).astype(np.uint8)


def quant_rows_int8(x: np.ndarray):
    """Per-row symmetric INT8: returns (q int8 [M, K], scale float32 [M])."""
    x32 = np.asarray(x, dtype=np.float32)
    amax = np.abs(x32).max(axis=1)
    scale = (amax / np.float32(INT8_QMAX)).astype(np.float32)
    scale = np.where(amax == 0, np.float32(1.0), scale).astype(np.float32)
    quot = (x32 / scale[:, None]).astype(np.float32)             # float32 division
    q = np.clip(np.rint(quot), -INT8_QMAX, INT8_QMAX).astype(np.int8)  # rint: half to even
    return q, scale


def quant_rows_e4m3(x: np.ndarray):
    """Per-row symmetric FP8-e4m3: returns (codes uint8 [M, K], scale float32 [M])."""
    x32 = np.asarray(x, dtype=np.float32)
    amax = np.abs(x32).max(axis=1)
    scale = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    scale = np.where(amax == 0, np.float32(1.0), scale).astype(np.float32)
    quot = (x32 / scale[:, None]).astype(np.float32)
    return e4m3_encode(quot), scale


def dequant(q: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 value of each code: int8 as an integer, e4m3 from the code book."""
    if dtype == "i8":
        return np.asarray(q, dtype=np.int8).astype(np.float64)
    if dtype == "e4m3":
        return E4M3_VALUES[np.asarray(q, dtype=np.uint8).astype(np.int64)]
    raise ValueError(dtype)
