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
