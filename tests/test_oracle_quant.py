"""Pins for the oracle's 1x128 and 128x128 quantisers (CPU only)."""

import os

import numpy as np
import pytest
import torch

from oracle import e4m3, quant
from fp8_fine_grained_e4m3_gb300 import synthetic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_blocks():
    rows = []
    with open(os.path.join(GOLDEN, "quant_worked_example.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            lhs, rhs = line.split("->")
            lhs = lhs.split()
            blk, scale, xs = int(lhs[0]), float(lhs[1]), [float(v) for v in lhs[2:]]
            qs = [int(v, 16) for v in rhs.split()]
            rows.append((blk, scale, xs, qs))
    return rows


@pytest.mark.parametrize("blk,scale,xs,qs", _golden_blocks())
def test_golden_worked_blocks(blk, scale, xs, qs):
    X = np.zeros((1, 128), dtype=np.float32)
    X[0, :len(xs)] = xs
    Q, S = quant.quant_1x128(X)
    assert S[0, 0] == np.float32(scale)
    assert list(Q[0, :len(qs)]) == qs
    assert np.all(Q[0, len(qs):] == 0)


def _library_quant_1x128(X):
    """The same rule through torch: FP32 amax, FP32 divisions, library e4m3 cast
    (which rounds to nearest-even and is exact on |x/s| <= 448 -- and x/s can
    only exceed 448 by FP32 rounding, which the clamp below settles)."""
    t = torch.from_numpy(X).view(X.shape[0], -1, 128)
    amax = t.abs().amax(dim=2)
    s = amax / torch.tensor(448.0, dtype=torch.float32)
    y = t / torch.where(amax > 0, s, torch.ones_like(s))[:, :, None]
    y = y.clamp(-448.0, 448.0)
    q = y.to(torch.float8_e4m3fn).view(torch.uint8)
    q[amax == 0] = 0
    return q.reshape(X.shape).numpy(), s.numpy()


@pytest.mark.parametrize("kind", ["normal", "prefill"])
def test_quant_1x128_matches_library(kind):
    X, _ = synthetic.dense_operands(64, 8, 1024, kind=kind, seed=3)
    X[5, 128:256] = 0.0  # one all-zero block
    Q, S = quant.quant_1x128(X)
    Ql, Sl = _library_quant_1x128(X)
    assert np.array_equal(S, Sl)
    assert np.array_equal(Q, Ql)


def test_fast_equals_loop():
    X, _ = synthetic.dense_operands(33, 8, 640, kind="prefill", seed=4)
    X[3, :128] = 0.0
    X[4, 5] = -0.0
    Q1, S1 = quant.quant_1x128(X)
    Q2, S2 = quant.quant_1x128_fast(X)
    assert np.array_equal(Q1, Q2) and np.array_equal(S1, S2)


def test_amax_element_hits_448():
    X = synthetic.masked_operands(2, 16, 8, 512, seed=5)[0].reshape(-1, 512)
    Q, S = quant.quant_1x128(X)
    for m in range(X.shape[0]):
        for kb in range(4):
            blk = X[m, kb * 128:(kb + 1) * 128]
            i = int(np.argmax(np.abs(blk)))
            assert Q[m, kb * 128 + i] in (0x7E, 0xFE)
            assert S[m, kb] == np.float32(np.float32(np.abs(blk).max()) / np.float32(448))


def test_dequant_error_bound():
    X, _ = synthetic.dense_operands(16, 8, 1024, kind="prefill", seed=6)
    Q, S = quant.quant_1x128(X)
    D = quant.dequant_1x128(Q, S)
    s = np.repeat(S.astype(np.float64), 128, axis=1)
    x = X.astype(np.float64)
    normal = np.abs(x) >= 2.0 ** -6 * s
    err = np.abs(D - x)
    # 3 mantissa bits: half an ulp is 2^-4 of the leading bit; the FP32 x/s
    # rounding adds at most a relative 2^-24
    assert np.all(err[normal] <= 2.0 ** -4 * np.abs(x[normal]) * (1 + 2.0 ** -20))
    assert np.all(err[~normal] <= 2.0 ** -10 * s[~normal] * (1 + 2.0 ** -20))


def test_zero_block_rule():
    X = np.zeros((2, 256), dtype=np.float32)
    X[1, 128:] = 1.0
    X[0, 3] = -0.0
    Q, S = quant.quant_1x128(X)
    assert np.all(S[0] == 0) and S[1, 0] == 0 and S[1, 1] == np.float32(1.0 / 448.0)
    assert np.all(Q[0] == 0) and np.all(Q[1, :128] == 0)
    assert np.all(Q[1, 128:] == 0x7E)


def test_ragged_k_block():
    X = np.zeros((1, 200), dtype=np.float32)
    X[0, 150] = 7.0
    Q, S = quant.quant_1x128(X)
    assert S.shape == (1, 2) and S[0, 1] == np.float32(7.0 / 448.0) and Q[0, 150] == 0x7E


def test_quant_128x128_scale_is_max_of_row_scales():
    _, W = synthetic.dense_operands(8, 300, 384, kind="decode", seed=7)
    Qw, Sw = quant.quant_128x128(W)
    _, Srow = quant.quant_1x128(W)
    Nb = Sw.shape[0]
    assert Sw.shape == (3, 3)
    for nb in range(Nb):
        # division by 448 is monotone, so max of the row scales equals the tile scale
        assert np.array_equal(Sw[nb], Srow[nb * 128:(nb + 1) * 128].max(axis=0))


def test_quant_128x128_matches_library():
    _, W = synthetic.dense_operands(8, 256, 256, kind="decode", seed=8)
    Qw, Sw = quant.quant_128x128(W)
    t = torch.from_numpy(W)
    for nb in range(2):
        for kb in range(2):
            tile = t[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128]
            s = tile.abs().max() / torch.tensor(448.0)
            q = (tile / s).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            assert Sw[nb, kb] == s.item()
            assert np.array_equal(Qw[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128], q)


def test_grouped_weight_quant_is_per_expert():
    _, W, _ = synthetic.masked_operands(3, 8, 128, 256, seed=9)
    Q, S = quant.quant_128x128_grouped(W)
    for e in range(3):
        q, s = quant.quant_128x128(W[e])
        assert np.array_equal(Q[e], q) and np.array_equal(S[e], s)


def test_quant_128x128_fast_equals_loop():
    _, W = synthetic.dense_operands(8, 300, 512, kind="decode", seed=10)
    W[128:256, 128:256] = 0.0  # an all-zero tile
    Q1, S1 = quant.quant_128x128(W)
    Q2, S2 = quant.quant_128x128_fast(W)
    assert np.array_equal(Q1, Q2) and np.array_equal(S1, S2)
