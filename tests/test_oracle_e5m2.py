"""Pins for the oracle's e5m2 codec, its quantiser and its use in the GEMM
(CPU only).

Decode: the bit definition (golden file) and a library routine
(torch.float8_e5m2).  Encode: the library cast within the finite range, a
brute-force nearest search with its own tie rule, saturation and round
trips.  Quantiser: the block maximum lands on the format's limit and the
relative error bound of a 2-bit mantissa.  GEMM: brute force with mixed
formats and the dequantise-then-multiply identity.
"""

import math
import os

import numpy as np
import pytest
import torch

from oracle import e4m3, e5m2, gemm, quant

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_codes():
    rows = []
    with open(os.path.join(GOLDEN, "e5m2_codes.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                c, v = line.split()
                rows.append((int(c, 16), float(v)))
    return rows


@pytest.mark.parametrize("code,value", _golden_codes())
def test_golden_codes(code, value):
    got = e5m2.decode_code(code)
    if math.isnan(value):
        assert math.isnan(got)
    else:
        assert got == value
        assert math.copysign(1.0, got) == math.copysign(1.0, value)


def test_decode_matches_library_cast():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    lib = codes.view(torch.float8_e5m2).to(torch.float64).numpy()
    ours = e5m2.decode_table()
    nan = np.isnan(lib)
    assert np.array_equal(nan, np.isnan(ours))
    assert np.array_equal(lib[~nan], ours[~nan])
    assert np.array_equal(np.signbit(lib[~nan]), np.signbit(ours[~nan]))


def test_table_shape_facts():
    t = e5m2.decode_table()
    assert np.isnan(t).sum() == 6  # 0x7D-0x7F and 0xFD-0xFF
    assert np.isinf(t).sum() == 2
    fin = t[np.isfinite(t)]
    assert fin.max() == 57344.0 and fin.min() == -57344.0
    assert fin[fin > 0].min() == 2.0 ** -16
    assert len(np.unique(fin)) == 247  # 248 finite codes; +0 and -0 coincide
    assert np.all(np.diff(t[:0x7C]) > 0)


def _bruteforce_encode(x):
    """Nearest finite e5m2 value by exhaustive search; on an exact tie the
    candidate with the even code wins; finite values beyond 57344 saturate."""
    t = e5m2.decode_table()
    codes = [c for c in range(256) if np.isfinite(t[c])]
    out = []
    for v in np.asarray(x, dtype=np.float32).astype(np.float64):
        if abs(v) > 57344:
            out.append(0x7B | (0x80 if v < 0 else 0))
            continue
        best, bestd = None, None
        for c in codes:
            if (c >= 0x80) != bool(np.signbit(v)):
                continue
            d = abs(t[c] - v)
            if bestd is None or d < bestd or (d == bestd and c % 2 == 0 and best % 2 == 1):
                best, bestd = c, d
        out.append(best)
    return np.array(out, dtype=np.uint8)


def _interesting_values(n, seed):
    g = np.random.default_rng(seed)
    v = g.uniform(1.0, 2.0, n) * 2.0 ** g.integers(-18, 16, n)
    v = np.where(g.random(n) < 0.5, -v, v)
    grid = e5m2.decode_table()[:0x7C]
    mids = (grid[:-1] + grid[1:]) / 2  # exact ties
    extra = np.concatenate([grid, -grid, mids, -mids, [0.0, -0.0, 57344.0, -57344.0]])
    return np.concatenate([v, extra]).astype(np.float32)


def test_encode_matches_library_cast():
    x = _interesting_values(20000, 1)
    x = x[np.abs(x) <= 57344]
    lib = torch.from_numpy(x).to(torch.float8_e5m2).view(torch.uint8).numpy()
    assert np.array_equal(e5m2.encode_rne_sat(x), lib)


def test_encode_matches_bruteforce():
    x = _interesting_values(1200, 2)
    x = np.concatenate([x, np.array([57345, 61439, 61440, 1e6, -3e38], np.float32)])
    assert np.array_equal(e5m2.encode_rne_sat(x), _bruteforce_encode(x))


def test_encode_saturates_and_ties():
    x = np.array([57344.0, 60000.0, 61440.0, 1e38], dtype=np.float32)
    assert np.all(e5m2.encode_rne_sat(x) == 0x7B)
    assert np.all(e5m2.encode_rne_sat(-x) == 0xFB)
    # 2^-17: tie 0 / 2^-16 -> 0; 1.125: tie 1.0 / 1.25 -> 1.0 (0x3C); 1.375: tie
    # 1.25 / 1.5 -> 1.5 (0x3E); -0 keeps its sign
    y = np.array([2.0 ** -17, 1.125, 1.375, -0.0], dtype=np.float32)
    assert list(e5m2.encode_rne_sat(y)) == [0x00, 0x3C, 0x3E, 0x80]


def test_round_trip_every_finite_code():
    t = e5m2.decode_table()
    codes = np.array([c for c in range(256) if np.isfinite(t[c])], dtype=np.uint8)
    assert np.array_equal(e5m2.encode_rne_sat(t[codes].astype(np.float32)), codes)


def test_quantiser_limit_and_error_bound():
    g = np.random.default_rng(5)
    X = (g.standard_normal((64, 384)) * 10.0 ** g.integers(-6, 6, (64, 1))).astype(np.float32)
    Q, S = quant.quant_1x128(X, fmt="e5m2")
    assert np.array_equal(S, (np.abs(X).reshape(64, 3, 128).max(axis=2) / np.float32(57344))
                          .astype(np.float32))
    # the element holding amax lands on +-57344 (codes 0x7B / 0xFB)
    blocks = np.abs(X).reshape(64, 3, 128)
    at = blocks.argmax(axis=2)
    q_at = Q.reshape(64, 3, 128)[np.arange(64)[:, None], np.arange(3)[None, :], at]
    assert np.all((q_at & 0x7F) == 0x7B)
    D = quant.dequant_1x128(Q, S, fmt="e5m2")
    normal = np.abs(X) >= np.repeat(S, 128, axis=1) * 2.0 ** -14
    err = np.abs(D - X.astype(np.float64))
    assert np.all(err[normal] <= 2.0 ** -3 * np.abs(X[normal]))
    assert np.array_equal(quant.quant_1x128_fast(X, fmt="e5m2")[0], Q)


def test_weight_quantiser_fast_form_agrees():
    g = np.random.default_rng(6)
    W = (g.standard_normal((300, 256)) * 0.02).astype(np.float32)
    Q1, S1 = quant.quant_128x128(W, fmt="e5m2")
    Q2, S2 = quant.quant_128x128_fast(W, fmt="e5m2")
    assert np.array_equal(Q1, Q2) and np.array_equal(S1.view(np.uint32), S2.view(np.uint32))


@pytest.mark.parametrize("a_fmt,b_fmt", [("e5m2", "e5m2"), ("e4m3", "e5m2"), ("e5m2", "e4m3")])
def test_gemm_bruteforce_mixed_formats(a_fmt, b_fmt):
    g = np.random.default_rng(7)
    M, N, K = 3, 5, 256
    A = g.integers(0, 0x7B, (M, K), dtype=np.int64).astype(np.uint8)  # finite codes of both
    B = g.integers(0, 0x7B, (N, K), dtype=np.int64).astype(np.uint8)
    sA = g.uniform(0.5, 2.0, (M, 2)).astype(np.float32)
    sB = g.uniform(0.5, 2.0, (1, 2)).astype(np.float32)
    dec = {"e4m3": e4m3.decode_code, "e5m2": e5m2.decode_code}
    ref = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            tot = 0.0
            for kb in range(2):
                part = 0.0
                for k in range(kb * 128, kb * 128 + 128):
                    part += dec[a_fmt](A[m, k]) * dec[b_fmt](B[n, k])
                tot += float(sA[m, kb]) * float(sB[0, kb]) * part
            ref[m, n] = tot
    got = gemm.gemm_dense(A, sA, B, sB, a_fmt=a_fmt, b_fmt=b_fmt)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_gemm_dequantise_then_matmul_mixed():
    g = np.random.default_rng(8)
    X = g.standard_normal((20, 384)).astype(np.float32)
    W = (g.standard_normal((260, 384)) * 0.02).astype(np.float32)
    A, sA = quant.quant_1x128(X, fmt="e5m2")
    B, sB = quant.quant_128x128(W, fmt="e4m3")
    Ad = quant.dequant_1x128(A, sA, fmt="e5m2")
    Bd = e4m3.decode(B) * np.repeat(np.repeat(sB.astype(np.float64), 128, 0), 128, 1)[:260, :384]
    ref = Ad @ Bd.T
    got = gemm.gemm_dense(A, sA, B, sB, a_fmt="e5m2", b_fmt="e4m3")
    assert np.allclose(got, ref, rtol=1e-10, atol=1e-12)
