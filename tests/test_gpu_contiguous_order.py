"""The contiguous MoE form at a wave or more of whole tiles takes its tiles in
expert-segment order (built on the device by a one-CTA ordering kernel from
m_indices: segments largest and smallest alternating, each in the dense
form's rasterisation) and claims them dynamically.  Against the oracle with
empty experts, padding blocks between segments, an expert split over two runs
and e5m2 operands; a bad expert index sets the status word and leaves every
other tile right; launches back to back, right after the quantiser with no
host synchronisation, and replayed from a CUDA graph."""

import numpy as np
import pytest

from fp8_fine_grained_e4m3_gb300 import synthetic
from tests.gpu_helpers import assert_close, dev, host, ogemm, oquant, quant_weights

pytestmark = pytest.mark.gpu


def _b():
    from fp8_fine_grained_e4m3_gb300 import binding
    return binding


def _weights(E, N, K, seed, fmt="e4m3"):
    W = synthetic.dense_operands(8, N, K, kind="normal", seed=seed)[1]
    Ws = [np.roll(W, 37 * e, axis=1) * np.float32(1 + 0.1 * e) for e in range(E)]
    if fmt == "e4m3":
        Bq = [quant_weights(w) for w in Ws]
    else:
        Bq = [oquant.quant_128x128(w, fmt=fmt) for w in Ws]
    return np.stack([q for q, _ in Bq]), np.stack([s for _, s in Bq])


def _rows(m_indices, K, seed, fmt="e4m3"):
    X = synthetic.dense_operands(len(m_indices), 8, K, kind="prefill", seed=seed)[0]
    X[m_indices < 0] = 0
    if fmt == "e4m3":
        return oquant.quant_1x128_fast(X)
    return oquant.quant_1x128(X, fmt=fmt)


def _layout(counts):
    return synthetic.contiguous_layout(np.asarray(counts)).m_indices


@pytest.mark.parametrize("counts,N,K", [
    (synthetic.zipf_counts(12, 3000, seed=4), 4096, 512),      # 480 tiles, Zipf sizes
    (synthetic.zipf_counts(20, 4000, seed=5), 2048, 256),      # 8 column tiles, 20 experts
    ([1500, 0, 3, 700, 0, 129, 1, 256], 2304, 384),            # empty experts, 1- and 3-row ones
])
def test_ordered_contiguous_matches_oracle(counts, N, K):
    b = _b()
    mi = _layout(counts)
    E = len(counts)
    A, sA = _rows(mi, K, seed=len(mi))
    B, sB = _weights(E, N, K, seed=E)
    l0 = b.num_kernel_launches()
    got = host(b.fp8gemm_grouped_contiguous(dev(A), dev(sA), dev(B), dev(sB), dev(mi)))
    assert b.num_kernel_launches() - l0 == 2  # the ordering kernel, then the GEMM
    assert_close(got, ogemm.gemm_contiguous(A, sA, B, sB, mi), f"ordered contiguous {counts}")
    assert b.fp8gemm_get_device_status() == b.OK


def test_ordered_contiguous_padding_blocks_and_split_expert():
    """Whole padding blocks between segments (first index -1: no tile) and one
    expert whose rows come in two separate runs (two segments of the same
    expert): every real row against the oracle."""
    b = _b()
    N, K, E = 4096, 256, 5
    parts = [_layout([300, 0, 0, 0, 0]), np.full(256, -1, np.int32), _layout([0, 700, 0, 0, 0]),
             np.full(128, -1, np.int32), _layout([0, 0, 129, 0, 40]), _layout([260, 0, 0, 0, 0]),
             _layout([0, 0, 0, 1, 0])]
    mi = np.concatenate(parts).astype(np.int32)
    A, sA = _rows(mi, K, seed=9)
    B, sB = _weights(E, N, K, seed=10)
    got = host(b.fp8gemm_grouped_contiguous(dev(A), dev(sA), dev(B), dev(sB), dev(mi)))
    assert_close(got, ogemm.gemm_contiguous(A, sA, B, sB, mi), "padding blocks, split expert")
    assert b.fp8gemm_get_device_status() == b.OK


def test_ordered_contiguous_bad_expert_index():
    """A block whose expert index is >= E: the ordering kernel sets
    FP8GEMM_ERR_DEVICE_STATUS and gives it no tile; every other row is right."""
    b = _b()
    N, K, E = 4096, 512, 6
    mi = _layout([900, 300, 0, 500, 130, 77])
    A, sA = _rows(mi, K, seed=11)
    B, sB = _weights(E, N, K, seed=12)
    bad = mi.copy()
    bad[1024:1152] = E + 3  # one whole block of the first expert
    got = host(b.fp8gemm_grouped_contiguous(dev(A), dev(sA), dev(B), dev(sB), dev(bad)))
    assert b.fp8gemm_get_device_status() == b.ERR_DEVICE_STATUS
    keep = bad.copy()
    keep[1024:1152] = -1  # the oracle's "not an output" rows
    assert_close(got, ogemm.gemm_contiguous(A, sA, B, sB, keep), "bad expert block")
    assert b.fp8gemm_get_device_status() == b.OK


@pytest.mark.parametrize("a_fmt,b_fmt", [("e5m2", "e4m3"), ("e4m3", "e5m2")])
def test_ordered_contiguous_e5m2(a_fmt, b_fmt):
    b = _b()
    N, K, E = 2048, 384, 9
    counts = synthetic.zipf_counts(E, 2600, seed=13)
    mi = _layout(counts)
    A, sA = _rows(mi, K, seed=14, fmt=a_fmt)
    B, sB = _weights(E, N, K, seed=15, fmt=b_fmt)
    got = host(b.fp8gemm_grouped_contiguous_fmt(dev(A), dev(sA), a_fmt, dev(B), dev(sB), b_fmt,
                                                dev(mi)))
    assert_close(got, ogemm.gemm_contiguous(A, sA, B, sB, mi, a_fmt, b_fmt),
                 f"ordered contiguous {a_fmt} x {b_fmt}")
    assert b.fp8gemm_get_device_status() == b.OK


def test_ordered_contiguous_chains_and_graph_replay():
    """Quantise on the device and run the contiguous GEMM right after, two
    layouts back to back with no host synchronisation (the ordering kernel
    waits for the quantiser, the GEMM for the ordering); then the call
    captured in a CUDA graph and replayed into NaN-filled output: every replay
    takes every tile (the counters go back to zero)."""
    import torch
    b = _b()
    N, K, E = 4096, 1024, 10
    B, sB = _weights(E, N, K, seed=16)
    tB, tsB = dev(B), dev(sB)
    runs = []
    for seed in (17, 18):
        mi = _layout(synthetic.zipf_counts(E, 2500, seed=seed))
        X = synthetic.dense_operands(len(mi), 8, K, kind="prefill", seed=seed)[0]
        X[mi < 0] = 0
        A8, sA8 = b.fp8_quant_1x128(dev(X))
        runs.append((X, mi, b.fp8gemm_grouped_contiguous(A8, sA8, tB, tsB, dev(mi))))
    for X, mi, D in runs:
        A, sA = oquant.quant_1x128_fast(X)
        assert_close(host(D), ogemm.gemm_contiguous(A, sA, B, sB, mi), "after the quantiser")
    X, mi, D = runs[-1]
    A8, sA8 = b.fp8_quant_1x128(dev(X))
    tmi = dev(mi)
    ref = host(D)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        b.fp8gemm_grouped_contiguous(A8, sA8, tB, tsB, tmi, D=D)  # the stream's workspace
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        b.fp8gemm_grouped_contiguous(A8, sA8, tB, tsB, tmi, D=D)
    real = mi >= 0
    for rep in range(3):
        D.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(host(D)[real], ref[real]), f"graph replay {rep}"
    assert b.fp8gemm_get_device_status() == b.OK


def test_ordered_contiguous_many_segments_keep_block_order():
    """More than 256 expert segments: the ordering kernel keeps them in block
    order (no ranking) and the result is still every row against the oracle
    (300 experts of 1-9 tokens, one 128-row block each)."""
    b = _b()
    E, N, K = 300, 512, 256
    counts = 1 + np.random.default_rng(21).integers(0, 9, E)
    mi = _layout(counts)
    A, sA = _rows(mi, K, seed=22)
    W = synthetic.dense_operands(8, N, K, kind="normal", seed=23)[1]
    Bq = [quant_weights(np.roll(W, e, axis=1)) for e in range(E)]
    B = np.stack([q for q, _ in Bq])
    sB = np.stack([s for _, s in Bq])
    l0 = b.num_kernel_launches()
    got = host(b.fp8gemm_grouped_contiguous(dev(A), dev(sA), dev(B), dev(sB), dev(mi)))
    assert b.num_kernel_launches() - l0 == 2
    assert_close(got, ogemm.gemm_contiguous(A, sA, B, sB, mi), "300 segments")
    assert b.fp8gemm_get_device_status() == b.OK
