"""FP8 (e4m3) quantisation of attention inputs, as its plain definition.

TEST INFRASTRUCTURE ONLY: imported by tests, never by the library.

"LLM Context Parallel in Production" lists BF16 / FP16 / FP8 among the
precisions a CP attention runs in; the format is OCP FP8 E4M3: 1 sign bit, 4
exponent bits (bias 7), 3 mantissa bits, no infinities, the all-ones code
(S.1111.111) NaN, largest finite value 448 = 1.75 * 2^8, subnormals down to
2^-9.

Readings taken for the Q K^T variant of the forward:
  * A tensor is quantised with one power-of-two scale s = 2^k, the largest
    with amax * s <= 448 (amax = max |x| over the tensor; k = 0 when amax is
    0): scaling by a power of two is exact, so dequantising (dividing by s) is
    exact too.
  * Rounding is to the nearest e4m3 value, ties to the even code, and values
    beyond 448 saturate to +-448 ("satfinite").
  * The scale is held as an fp32 number, so 2^k is kept to fp32's normal
    range, -126 <= k <= 127 (only an amax below 2^-119 reaches the bound).
"""
from __future__ import annotations

import math

import numpy as np

E4M3_MAX = 448.0


def e4m3_values() -> np.ndarray:
    """Value of every one of the 256 codes (NaN for the two NaN codes)."""
    v = np.empty(256)
    for c in range(256):
        s = -1.0 if c & 0x80 else 1.0
        e = (c >> 3) & 0xF
        m = c & 7
        if e == 0xF and m == 7:
            v[c] = np.nan
        elif e == 0:
            v[c] = s * m * 2.0 ** -9                      # subnormal: m/8 * 2^-6
        else:
            v[c] = s * (1 + m / 8.0) * 2.0 ** (e - 7)
    return v


_VALS = e4m3_values()
# Non-negative finite codes 0x00..0x7E in increasing value order.
_POS_CODES = np.arange(0x7F)
_POS_VALS = _VALS[_POS_CODES]


def quantize_codes(x) -> np.ndarray:
    """e4m3 code of every element of x (float64 array): nearest value, ties to
    the even code, saturating at +-448."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    hi = np.searchsorted(_POS_VALS, a, side="left")          # first value >= a
    hi = np.minimum(hi, len(_POS_VALS) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - _POS_VALS[lo]
    d_hi = _POS_VALS[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (_POS_CODES[hi] % 2 == 0))
    code = np.where(pick_hi, _POS_CODES[hi], _POS_CODES[lo])
    code = np.where(a == _POS_VALS[hi], _POS_CODES[hi], code)
    sign = np.signbit(x).astype(np.int64) << 7      # a zero result keeps its sign
    return (code | sign).astype(np.uint8)


def dequantize(codes) -> np.ndarray:
    return _VALS[np.asarray(codes, dtype=np.int64)]


def pow2_scale_exponent(amax: float) -> int:
    """k of the per-tensor scale 2^k: the largest with amax * 2^k <= 448."""
    if amax == 0.0:
        return 0
    m, e = math.frexp(amax)          # amax = m * 2^e, m in [0.5, 1)
    m, e = 2.0 * m, e - 1            # amax = m * 2^e, m in [1, 2)
    k = (8 if m <= 1.75 else 7) - e
    return max(-126, min(127, k))    # 2^k is an fp32 normal number


def quantize_tensor(x):
    """(codes, k): e4m3 codes of x * 2^k with the per-tensor scale of x."""
    x = np.asarray(x, dtype=np.float64)
    k = pow2_scale_exponent(float(np.max(np.abs(x))) if x.size else 0.0)
    return quantize_codes(x * 2.0 ** k), k


def dequantized_tensor(x) -> np.ndarray:
    """x as the Q K^T variant sees it: e4m3 codes of x * 2^k, divided back by 2^k."""
    codes, k = quantize_tensor(x)
    return dequantize(codes) * 2.0 ** -k
