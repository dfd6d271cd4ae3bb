"""Pins for the oracle's e4m3 codec (CPU only).

The decode table is pinned by the values the pages fix (448) plus the
format's bit definition (golden file), and by a library routine
(torch.float8_e4m3fn).  The encoder is pinned by the library cast, by a
brute-force nearest search with a different tie rule implementation, and by
round trips.
"""

import math
import os

import numpy as np
import pytest
import torch

from oracle import e4m3

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_codes():
    rows = []
    with open(os.path.join(GOLDEN, "e4m3_codes.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                c, v = line.split()
                rows.append((int(c, 16), float(v)))
    return rows


@pytest.mark.parametrize("code,value", _golden_codes())
def test_golden_codes(code, value):
    got = e4m3.decode_code(code)
    if math.isnan(value):
        assert math.isnan(got)
    else:
        assert got == value
        assert math.copysign(1.0, got) == math.copysign(1.0, value)


def test_decode_matches_library_cast():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    lib = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = e4m3.decode_table()
    nan = np.isnan(lib)
    assert np.array_equal(nan, np.isnan(ours))
    assert np.array_equal(lib[~nan], ours[~nan])
    assert np.array_equal(np.signbit(lib[~nan]), np.signbit(ours[~nan]))


def test_table_shape_facts():
    t = e4m3.decode_table()
    assert np.isnan(t).sum() == 2  # 0x7F, 0xFF only: no infinities
    fin = t[~np.isnan(t)]
    assert fin.max() == 448.0 and fin.min() == -448.0
    assert fin[fin > 0].min() == 2.0 ** -9  # smallest subnormal
    assert len(np.unique(fin)) == 253  # +0 and -0 coincide
    pos = t[:0x7F]
    assert np.all(np.diff(pos) > 0)  # codes 0x00..0x7E increase


def _bruteforce_encode(x):
    """Nearest finite e4m3 value by exhaustive distance search; on an exact
    tie pick the candidate whose code is even.  Saturates beyond 448."""
    t = e4m3.decode_table()
    codes = [c for c in range(256) if not math.isnan(t[c])]
    out = []
    for v in np.asarray(x, dtype=np.float32).astype(np.float64):
        if abs(v) > 448:
            out.append(0x7E | (0x80 if v < 0 else 0))
            continue
        best, bestd = None, None
        for c in codes:
            # same sign half only (so that -0/+0 follow the input's sign)
            if (c >= 0x80) != bool(np.signbit(v)):
                continue
            d = abs(t[c] - v)
            if bestd is None or d < bestd or (d == bestd and c % 2 == 0 and best % 2 == 1):
                best, bestd = c, d
        out.append(best)
    return np.array(out, dtype=np.uint8)


def _interesting_values(n, seed):
    g = np.random.default_rng(seed)
    mant = g.uniform(1.0, 2.0, n)
    exp = g.integers(-14, 9, n)
    v = mant * 2.0 ** exp
    v = np.where(g.random(n) < 0.5, -v, v)
    grid = e4m3.decode_table()[:0x7F]
    mids = (grid[:-1] + grid[1:]) / 2  # exact ties
    extra = np.concatenate([grid, -grid, mids, -mids, [0.0, -0.0, 448.0, -448.0]])
    return np.concatenate([v, extra]).astype(np.float32)


def test_encode_matches_library_cast():
    x = _interesting_values(20000, 1)
    x = x[np.abs(x) <= 448]
    lib = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(e4m3.encode_rne_sat(x), lib)


def test_encode_matches_bruteforce():
    x = _interesting_values(1500, 2)
    x = np.concatenate([x, np.array([449, 463.9, 464, 500, 1e6, -1e30], np.float32)])
    assert np.array_equal(e4m3.encode_rne_sat(x), _bruteforce_encode(x))


def test_encode_saturates():
    x = np.array([448.0, 448.5, 463.99, 464.0, 479.0, 480.0, 1e38], dtype=np.float32)
    assert np.all(e4m3.encode_rne_sat(x) == 0x7E)
    assert np.all(e4m3.encode_rne_sat(-x) == 0xFE)


def test_encode_ties_to_even_and_tiny():
    x = np.array([2.0 ** -10, 2.0 ** -10 * 1.0000001, 3 * 2.0 ** -10, 17.0, 19.0, -0.0],
                 dtype=np.float32)
    # 2^-10: tie 0 / 2^-9 -> 0; just above -> 0x01; 3*2^-10: tie 2^-9 / 2^-8 -> 0x02;
    # 17: tie 16 / 18 -> 16 (0x58); 19: tie 18 / 20 -> 20 (0x5A); -0 keeps sign
    assert list(e4m3.encode_rne_sat(x)) == [0x00, 0x01, 0x02, 0x58, 0x5A, 0x80]


def test_round_trip_every_finite_code():
    t = e4m3.decode_table()
    codes = np.array([c for c in range(256) if not math.isnan(t[c])], dtype=np.uint8)
    back = e4m3.encode_rne_sat(t[codes].astype(np.float32))
    assert np.array_equal(back, codes)
