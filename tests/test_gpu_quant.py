"""GPU quantisers vs the oracle: bit-exact bytes and scales."""

import numpy as np
import pytest

from fp8_fine_grained_e4m3_gb300 import synthetic
from tests.gpu_helpers import dev, host, oquant, quant_weights

pytestmark = pytest.mark.gpu


def _binding():
    from fp8_fine_grained_e4m3_gb300 import binding
    return binding


@pytest.mark.parametrize("M,K,kind", [(128, 512, "normal"), (257, 4096, "prefill"),
                                      (64, 7168, "decode"), (1, 128, "normal"),
                                      (33, 144, "normal"), (5, 16, "normal"),    # partial K block
                                      (3000, 400, "prefill")])                   # many CTAs, partial
def test_quant_1x128_bit_exact(M, K, kind):
    X, _ = synthetic.dense_operands(M, 8, K, kind=kind, seed=M + K)
    Q, S = _binding().fp8_quant_1x128(dev(X))
    Qo, So = oquant.quant_1x128_fast(X)
    assert np.array_equal(host(Q), Qo)
    assert np.array_equal(host(S).view(np.uint32), So.view(np.uint32))


def test_quant_1x128_student_t_masked_shape():
    X, _, _ = synthetic.masked_operands(16, 256, 8, 7168, seed=1)
    X2 = X.reshape(-1, 7168)
    Q, S = _binding().fp8_quant_1x128(dev(X2))
    Qo, So = oquant.quant_1x128_fast(X2)
    assert np.array_equal(host(Q), Qo)
    assert np.array_equal(host(S).view(np.uint32), So.view(np.uint32))


def test_quant_1x128_edge_values():
    """Zero blocks, signed zeros, exact ties, subnormal results, the golden
    worked blocks, and values one ulp around e4m3 midpoints."""
    from tests.test_oracle_quant import _golden_blocks
    rows = []
    for _, _, xs, _ in _golden_blocks():
        r = np.zeros(128, np.float32)
        r[:len(xs)] = xs
        rows.append(r)
    g = np.random.default_rng(5)
    grid = np.array(sorted({abs(v) for v in __import__("oracle").e4m3.decode_table()[:0x7F]}))
    mids = ((grid[:-1] + grid[1:]) / 2).astype(np.float32)
    for _ in range(8):
        r = np.zeros(128, np.float32)
        r[0] = 448.0  # s = 1: x / s is x itself
        sel = g.choice(mids, 127)
        nudge = g.integers(-1, 2, 127)
        r[1:] = np.array([np.nextafter(v, np.float32(np.inf * n)) if n else v
                          for v, n in zip(sel, nudge)], np.float32)
        r[1:] *= np.where(g.random(127) < 0.5, -1, 1).astype(np.float32)
        rows.append(r)
    r = np.full(128, -0.0, np.float32)
    rows.append(r)
    r = np.zeros(128, np.float32)
    r[7] = 1e-30  # amax tiny: x/s lands at 448 exactly
    r[8] = 1e-33
    rows.append(r)
    X = np.stack(rows)
    Q, S = _binding().fp8_quant_1x128(dev(X))
    Qo, So = oquant.quant_1x128(X)
    assert np.array_equal(host(Q), Qo)
    assert np.array_equal(host(S).view(np.uint32), So.view(np.uint32))


@pytest.mark.parametrize("E,N,K", [(1, 256, 512), (1, 300, 384), (3, 520, 256), (1, 7168, 2048),
                                   (2, 300, 400), (1, 130, 16)])  # partial last K tile
def test_quant_128x128_bit_exact(E, N, K):
    _, W, _ = synthetic.masked_operands(E, 1, N, K, seed=E * N + K)
    Q, S = _binding().fp8_quant_128x128(dev(W))
    for e in range(E):
        Qo, So = quant_weights(W[e])
        assert np.array_equal(host(Q)[e], Qo)
        assert np.array_equal(host(S)[e].view(np.uint32), So.view(np.uint32))


def test_quant_zero_rows_is_noop():
    import torch
    X = torch.zeros((0, 256), dtype=torch.float32, device="cuda")
    Q, S = _binding().fp8_quant_1x128(X)
    assert Q.shape == (0, 256) and S.shape == (0, 2)


@pytest.mark.parametrize("M,K,fmt,kind", [(300, 1024, "e4m3", "normal"), (257, 4096, "e4m3", "prefill"),
                                          (130, 400, "e4m3", "normal"),   # ragged last K block
                                          (200, 768, "e5m2", "normal"), (3000, 400, "e4m3", "prefill"),
                                          (16, 7168, "e4m3", "decode")])  # one wave: the PDL launch
def test_quant_1x128_saturation_count(M, K, fmt, kind):
    """fp8_quant_1x128_ex: the count equals the oracle's, the bytes and scales
    are those of the call without a counter, and the counter accumulates."""
    import torch
    b = _binding()
    X, _ = synthetic.dense_operands(M, 8, K, kind=kind, seed=M * 3 + K)
    X[min(7, M - 1), :128] = np.float32(1e-44) * (np.arange(128) % 2)  # amax / limit underflows
    want = oquant.saturations_1x128(X, fmt)
    assert want > 0
    cnt = torch.zeros(1, dtype=torch.int64, device="cuda")
    Q, S = b.fp8_quant_1x128_fmt(dev(X), fmt, sat_count=cnt)
    Q0, S0 = b.fp8_quant_1x128_fmt(dev(X), fmt)
    assert int(cnt.item()) == want
    assert np.array_equal(host(Q), host(Q0))
    assert np.array_equal(host(S).view(np.uint32), host(S0).view(np.uint32))
    b.fp8_quant_1x128_fmt(dev(X), fmt, sat_count=cnt)
    assert int(cnt.item()) == 2 * want


@pytest.mark.parametrize("E,N,K,fmt", [(1, 300, 640, "e4m3"), (3, 256, 400, "e4m3"),
                                       (2, 200, 256, "e5m2")])
def test_quant_128x128_saturation_count(E, N, K, fmt):
    import torch
    b = _binding()
    g = np.random.default_rng(E * 100 + N)
    W = g.standard_normal((E, N, K)).astype(np.float32)
    W[0, :128, :128] = 0
    W[0, 5, 3] = np.float32(1e-44)  # one tile whose scale underflows
    want = oquant.saturations_128x128(W, fmt)
    assert want > 0
    cnt = torch.zeros(1, dtype=torch.int64, device="cuda")
    Q, S = b.fp8_quant_128x128_fmt(dev(W), fmt, sat_count=cnt)
    Q0, S0 = b.fp8_quant_128x128_fmt(dev(W), fmt)
    assert int(cnt.item()) == want
    assert np.array_equal(host(Q), host(Q0))
    assert np.array_equal(host(S).view(np.uint32), host(S0).view(np.uint32))


@pytest.mark.parametrize("E,N,K,fmt", [(1, 256, 512, "e4m3"), (2, 300, 400, "e4m3"),
                                       (1, 256, 256, "e5m2")])
def test_quant_128x128_quotients_near_rounding_points(E, N, K, fmt):
    """Weights whose quotients x / s sit within 8 ulps of every FP8 value and
    midpoint, per 128 x 128 tile (e4m3 and e5m2, two experts, a ragged N and
    a partial K tile): bytes, scales and the saturation count equal the
    oracle's, and the plain and counting instances agree."""
    import torch
    from oracle import e4m3, e5m2
    b = _binding()
    mod, limit = (e4m3, 448.0) if fmt == "e4m3" else (e5m2, 57344.0)
    lut = mod.decode_table()
    vals = np.unique(np.abs(lut[np.isfinite(lut)]))
    vals = vals[vals <= limit]
    points = np.concatenate([vals, (vals[1:] + vals[:-1]) / 2.0])
    points = points[points < limit]
    g = np.random.default_rng(E * 1000 + N + K)
    W = np.zeros((E, N, K), np.float32)
    for e in range(E):
        for n0 in range(0, N, 128):
            for k0 in range(0, K, 128):
                rows, cols = min(128, N - n0), min(128, K - k0)
                amax = np.float32(g.uniform(0.25, 4.0))
                s = np.float32(amax / np.float32(limit))
                q = g.choice(points, (rows, cols)) * g.choice([-1.0, 1.0], (rows, cols))
                q = q * (1.0 + g.integers(-8, 9, (rows, cols)) * 2.0 ** -23)
                t = np.clip((q * np.float64(s)).astype(np.float32), -amax, amax)
                t[0, 0] = amax
                W[e, n0:n0 + rows, k0:k0 + cols] = t
    Q, S = b.fp8_quant_128x128_fmt(dev(W), fmt)
    cnt = torch.zeros(1, dtype=torch.int64, device="cuda")
    Qc, Sc = b.fp8_quant_128x128_fmt(dev(W), fmt, sat_count=cnt)
    for e in range(E):
        Qo, So = oquant.quant_128x128(W[e], fmt=fmt)
        assert np.array_equal(host(Q)[e], Qo)
        assert np.array_equal(host(S)[e].view(np.uint32), So.view(np.uint32))
    assert np.array_equal(host(Q), host(Qc))
    assert np.array_equal(host(S).view(np.uint32), host(Sc).view(np.uint32))
    assert int(cnt.item()) == oquant.saturations_128x128(W, fmt)
