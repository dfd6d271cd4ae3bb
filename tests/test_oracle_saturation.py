"""Pins for the oracle's saturation count (the FP8 overflow counter of the
quantisers): each check rests on something other than the oracle itself --
exact rational arithmetic, closed forms, symmetries and special cases.

The count is the number of elements x of blocks with amax != 0 whose FP32
quotient x / s (s = amax / limit, both IEEE FP32 round-to-nearest) is not
within +-limit ("blog.hotdry.top: DeepGEMM FP8 GEMM fine-grained scaling
kernels", section on numerical-stability checks and monitoring: an FP8
overflow count among the metrics to watch)."""

from fractions import Fraction

import numpy as np

import oracle.quant as quant


def _fp32_rn(r: Fraction) -> Fraction:
    """IEEE binary32 round-to-nearest-even of a positive rational in the
    normal range, from the definition (24-bit significand)."""
    assert r > 0
    e = r.numerator.bit_length() - r.denominator.bit_length()
    while Fraction(2) ** e > r:
        e -= 1
    while Fraction(2) ** (e + 1) <= r:
        e += 1
    ulp = Fraction(2) ** (e - 23)
    m = r / ulp
    lo = m.numerator // m.denominator
    rem = m - lo
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1):
        lo += 1
    return lo * ulp


def _overshoots(amax: float, limit: int) -> bool:
    """Whether fl(amax / fl(amax / limit)) > limit, in exact arithmetic."""
    a = Fraction(float(np.float32(amax)))
    s = _fp32_rn(a / limit)
    return _fp32_rn(a / s) > limit


def test_amax_element_against_exact_rounding():
    # blocks whose other elements are far below amax: only the amax element
    # can pass the limit, and whether it does is decided exactly here
    g = np.random.default_rng(11)
    amaxes = np.abs(g.standard_normal(300)).astype(np.float32) + np.float32(1e-3)
    want = got = 0
    seen = set()
    for fmt, limit in (("e4m3", 448), ("e5m2", 57344)):
        for a in amaxes:
            blk = np.full(128, np.float32(a) / 4, dtype=np.float32)
            blk[37] = a
            over = _overshoots(a, limit)
            seen.add(over)
            want += int(over)
            got += quant._block_saturations(blk, fmt)
    assert got == want
    assert seen == {True, False}  # the sample has both kinds


def test_power_of_two_scales_never_saturate():
    # amax = limit * 2^k: s = 2^k exactly, every quotient exact and <= limit
    g = np.random.default_rng(3)
    for fmt, limit in (("e4m3", 448.0), ("e5m2", 57344.0)):
        for k in (-20, -3, 0, 5, 30):
            amax = np.float32(limit * 2.0 ** k)
            blk = (g.uniform(-1, 1, 128) * amax).astype(np.float32)
            blk[0] = -amax
            assert quant._block_saturations(blk, fmt) == 0
            q, s = quant._quant_block(blk, fmt)
            assert s == np.float32(2.0 ** k)


def test_quotient_equal_to_limit_is_not_counted():
    # x / s == 448 exactly (s a power of two) is representable: no clamp
    blk = np.zeros(128, np.float32)
    blk[5] = 448.0
    assert quant._block_saturations(blk) == 0
    assert quant.saturations_1x128(blk[None, :]) == 0


def test_zero_block_and_underflowing_scale():
    assert quant.saturations_1x128(np.zeros((3, 256), np.float32)) == 0
    # amax / 448 underflows to 0 in FP32: every quotient is +-inf or 0/0
    tiny = np.zeros(128, np.float32)
    tiny[::3] = np.float32(1e-44)
    assert np.float32(np.float32(1e-44) / np.float32(448)) == 0
    assert quant._block_saturations(tiny) == 128


def test_sign_and_power_of_two_invariance():
    g = np.random.default_rng(5)
    X = g.standard_normal((40, 384)).astype(np.float32)
    n = quant.saturations_1x128(X)
    assert n > 0
    assert quant.saturations_1x128(-X) == n
    for j in (-8, 8):
        assert quant.saturations_1x128((X * np.float32(2.0 ** j)).astype(np.float32)) == n


def test_ragged_block_counts_only_present_elements():
    g = np.random.default_rng(9)
    X = g.standard_normal((20, 144)).astype(np.float32)
    full = quant.saturations_1x128(X)
    assert full == (quant.saturations_1x128(X[:, :128])
                    + sum(quant._block_saturations(X[m, 128:]) for m in range(20)))


def test_tile_count_reduces_to_row_blocks_for_one_row():
    # a 128x128 tile with one nonzero row has that row's amax: same count
    g = np.random.default_rng(2)
    for _ in range(20):
        row = g.standard_normal(128).astype(np.float32)
        W = np.zeros((128, 128), np.float32)
        W[17] = row
        assert quant.saturations_128x128(W) == quant.saturations_1x128(row[None, :])
