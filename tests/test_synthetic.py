"""The seeded workload generators: shapes, determinism, grouping structure."""

import numpy as np

from fp8_fine_grained_e4m3_gb300 import synthetic


def test_dense_deterministic_and_shaped():
    X1, W1 = synthetic.dense_operands(4, 6, 256, kind="prefill", seed=1)
    X2, W2 = synthetic.dense_operands(4, 6, 256, kind="prefill", seed=1)
    assert X1.shape == (4, 256) and W1.shape == (6, 256)
    assert X1.dtype == np.float32 and np.array_equal(X1, X2) and np.array_equal(W1, W2)


def test_prefill_outlier_columns():
    K = 4096
    cols = synthetic.outlier_columns(K, 0)
    assert len(cols) == 41 and len(np.unique(cols)) == 41
    X, W = synthetic.dense_operands(256, 64, K, kind="prefill", seed=0)
    col_std = X.std(axis=0)
    assert np.all(col_std[cols] > 20) and np.median(col_std) < 1.5
    assert 0.015 < W.std() < 0.025
    assert len(synthetic.outlier_columns(16384, 0)) == 164


def test_zipf_counts():
    c = synthetic.zipf_counts(32, 8192, seed=0)
    assert c.sum() == 8192 and len(c) == 32
    assert c[0] > c[8] > c[31]
    assert 0.2 < c[0] / 8192 < 0.35


def test_contiguous_layout():
    lay = synthetic.contiguous_layout(np.array([3, 0, 128, 130]))
    assert list(lay.padded) == [128, 0, 128, 256]
    assert list(lay.offsets) == [0, 128, 128, 256]
    assert lay.M_pad == 512
    mi = lay.m_indices
    assert list(mi[:4]) == [0, 0, 0, -1] and np.all(mi[3:128] == -1)
    assert np.all(mi[128:256] == 2) and np.all(mi[256:386] == 3) and np.all(mi[386:] == -1)


def test_contiguous_padding_rows_zero():
    X, W, lay = synthetic.contiguous_operands(4, 100, 128, 128, seed=2)
    assert X.shape[0] == lay.M_pad and W.shape == (4, 128, 128)
    assert np.all(X[lay.m_indices < 0] == 0)


def test_masked_counts_range():
    mm = synthetic.masked_counts(16, 256, seed=0)
    assert mm.dtype == np.int32 and mm.min() >= 0 and mm.max() <= 256
    X, W, mm2 = synthetic.masked_operands(2, 8, 16, 128, seed=3)
    assert X.shape == (2, 8, 128) and W.shape == (2, 16, 128)
    big = synthetic.masked_operands(1, 64, 8, 1024, seed=4)[0]
    # Student-t(3): heavy tails
    assert np.abs(big).max() > 10
