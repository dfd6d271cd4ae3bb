"""The FP8 E4M3 ("fn") number format, written out from its bit definition.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Format facts used here (all pages agree on them):

* 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits
  ("news.rkmt.cn/news/5092" section 2.1; "lpnh.cn/news/2822121" section 2.1;
  "bhfrc.com/news/60211" section 2.1);
* the largest finite magnitude is 448 ("news.rkmt.cn/news/5092" section 5.2;
  "lpnh.cn/news/2822121" section 2.1; "bhfrc.com/news/60211" section 2.1).

The "fn" variant has no infinities: exponent 1111 with mantissa 111 is NaN,
and exponent 1111 with any other mantissa is an ordinary normal number (that
is how 448 = 1.75 * 2^8 fits).  Subnormals (exponent 0000) are m/8 * 2^-6.

Encoding from FP32 rounds to nearest with ties to even ("lpnh.cn/news/2822121"
section 6.3, second point: round to nearest, never toward zero) and saturates
magnitudes above 448 to 448.  The pages disagree on what overflow does (one
says NaN, one says infinity, which e4m3fn cannot hold); saturation is the
reading taken, because only FP32 rounding of x/s can push a quantised value
past 448.
"""

import numpy as np

E4M3_MAX = 448.0
E4M3_BIAS = 7
NAN_CODES = (0x7F, 0xFF)


def decode_code(code: int) -> float:
    """Value of one e4m3 byte, straight from the bit fields (float64)."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    exp = (code >> 3) & 0xF
    man = code & 0x7
    if exp == 0xF and man == 0x7:
        return float("nan")
    if exp == 0:  # subnormal: 0.mmm * 2^(1 - bias)
        return sign * (man / 8.0) * 2.0 ** (1 - E4M3_BIAS)
    return sign * (1.0 + man / 8.0) * 2.0 ** (exp - E4M3_BIAS)


def decode_table() -> np.ndarray:
    """All 256 codes decoded to float64 (index = byte value)."""
    return np.array([decode_code(c) for c in range(256)], dtype=np.float64)


_LUT = decode_table()
# Non-negative finite codes 0x00..0x7E are strictly increasing in value.
_POS_GRID = _LUT[:0x7F].copy()


def decode(q: np.ndarray) -> np.ndarray:
    """Decode an array of e4m3 bytes (uint8) to float64."""
    q = np.asarray(q, dtype=np.uint8)
    return _LUT[q]


def encode_rne_sat(x: np.ndarray) -> np.ndarray:
    """Encode FP32 values to e4m3 bytes: round to nearest, ties to even,
    saturate |x| > 448 to 448.  The sign of zero is kept (-0.0 -> 0x80).

    The nearest representable magnitude is found by comparing |x| with the
    exact midpoint between the two neighbouring grid values; a value exactly
    on the midpoint takes the neighbour whose code is even (even mantissa).
    NaN input gives 0x7F (NaN); the generators never produce one.
    """
    x = np.asarray(x, dtype=np.float32)
    mag = np.abs(x).astype(np.float64)
    sign = np.signbit(x)
    # index of first grid value >= mag (grid covers [0, 448])
    hi = np.searchsorted(_POS_GRID, mag, side="left")
    hi = np.minimum(hi, 0x7E)
    lo = np.maximum(hi - 1, 0)
    g_lo = _POS_GRID[lo]
    g_hi = _POS_GRID[hi]
    mid = (g_lo + g_hi) * 0.5  # exact: both have <= 4 significant bits
    take_hi = mag > mid
    tie = mag == mid
    take_hi = take_hi | (tie & (hi % 2 == 0))
    code = np.where(take_hi, hi, lo)
    # exact grid hits (including 0) land on hi == lo or on hi itself
    code = np.where(mag == g_hi, hi, code)
    code = np.where(mag > E4M3_MAX, 0x7E, code)  # saturate
    code = code.astype(np.uint8)
    code = np.where(sign, code | np.uint8(0x80), code).astype(np.uint8)
    code = np.where(np.isnan(x), np.uint8(0x7F), code).astype(np.uint8)
    return code
