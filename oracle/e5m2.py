"""The FP8 E5M2 number format, written out from its bit definition.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Format facts from the pages: FP8 is two formats; e5m2 has one more exponent
bit and one fewer mantissa bit than e4m3 -- 1 sign, 5 exponent, 2 mantissa
bits -- so it reaches much larger values with less precision; activations and
weights usually take e4m3 and gradients e5m2 ("news.rkmt.cn/news/5092"
section 2.1; "lpnh.cn/news/2822121" section 2.1, which also notes that mixing
an e4m3 A with an e5m2 B costs precision).  The pages' table of the two
formats did not survive extraction, so the rest follows the format's
definition: exponent bias 15; exponent 11111 is infinity (mantissa 00) or NaN
(mantissa != 00), as in IEEE binary formats; subnormals (exponent 00000) are
m/4 * 2^-14; the largest finite magnitude is 1.75 * 2^15 = 57344.

Encoding from FP32 rounds to nearest with ties to even (the pages' rounding
rule, "lpnh.cn/news/2822121" section 6.3) and saturates finite magnitudes
above 57344 to 57344, the same reading as for e4m3: only the FP32 rounding of
x/s can push a quantised value past the limit.
"""

import numpy as np

E5M2_MAX = 57344.0
E5M2_BIAS = 15


def decode_code(code: int) -> float:
    """Value of one e5m2 byte, straight from the bit fields (float64)."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    exp = (code >> 2) & 0x1F
    man = code & 0x3
    if exp == 0x1F:
        return sign * float("inf") if man == 0 else float("nan")
    if exp == 0:  # subnormal: 0.mm * 2^(1 - bias)
        return sign * (man / 4.0) * 2.0 ** (1 - E5M2_BIAS)
    return sign * (1.0 + man / 4.0) * 2.0 ** (exp - E5M2_BIAS)


def decode_table() -> np.ndarray:
    """All 256 codes decoded to float64 (index = byte value)."""
    return np.array([decode_code(c) for c in range(256)], dtype=np.float64)


_LUT = decode_table()
# Non-negative finite codes 0x00..0x7B are strictly increasing in value.
_POS_GRID = _LUT[:0x7C].copy()


def decode(q: np.ndarray) -> np.ndarray:
    """Decode an array of e5m2 bytes (uint8) to float64."""
    return _LUT[np.asarray(q, dtype=np.uint8)]


def encode_rne_sat(x: np.ndarray) -> np.ndarray:
    """Encode FP32 values to e5m2 bytes: round to nearest, ties to even,
    saturate finite |x| > 57344 to 57344.  The sign of zero is kept.

    The nearest representable magnitude is found by comparing |x| with the
    exact midpoint between its two neighbouring grid values; a value exactly
    on the midpoint takes the neighbour whose code is even (even mantissa).
    NaN input gives 0x7F; the generators never produce one.
    """
    x = np.asarray(x, dtype=np.float32)
    mag = np.abs(x).astype(np.float64)
    sign = np.signbit(x)
    hi = np.searchsorted(_POS_GRID, mag, side="left")  # first grid value >= mag
    hi = np.minimum(hi, 0x7B)
    lo = np.maximum(hi - 1, 0)
    g_lo = _POS_GRID[lo]
    g_hi = _POS_GRID[hi]
    mid = (g_lo + g_hi) * 0.5  # exact: both have <= 3 significant bits
    take_hi = (mag > mid) | ((mag == mid) & (hi % 2 == 0))
    code = np.where(take_hi, hi, lo)
    code = np.where(mag == g_hi, hi, code)
    code = np.where(mag > E5M2_MAX, 0x7B, code)  # saturate
    code = code.astype(np.uint8)
    code = np.where(sign, code | np.uint8(0x80), code).astype(np.uint8)
    return np.where(np.isnan(x), np.uint8(0x7F), code).astype(np.uint8)
