"""Dense GEMM on the GPU vs the FP64 oracle (per-element acceptance test)."""

import numpy as np
import pytest

from tests.gpu_helpers import (assert_close, dev, host, ogemm, oquant, quant_weights,
                               quantised_dense, sample_rows_cols)

pytestmark = pytest.mark.gpu


def _b():
    from fp8_fine_grained_e4m3_gb300 import binding
    return binding


def _run(A, sA, B, sB):
    return host(_b().fp8gemm_dense(dev(A), dev(sA), dev(B), dev(sB)))


@pytest.mark.parametrize("M,N,K,kind", [
    (128, 256, 512, "normal"),      # the correctness configuration, whole
    (300, 520, 1024, "normal"),     # ragged M and N, several tiles (128-wide N tiles)
    (256, 512, 640, "prefill"),     # 256-wide N tiles, outlier columns
    (65, 256, 256, "normal"),       # smallest M on the large-M path
    (520, 2304, 384, "prefill"),    # many tiles, 256-wide N tiles, ragged M
    (257, 768, 1024, "prefill"),    # one row into a third M tile
    (777, 2176, 512, "normal"),     # N >= 2048 not a multiple of 256: half-empty last N tile
    (1, 7168, 2048, "decode"),      # decode shapes, whole
    (16, 7168, 2048, "decode"),
    (64, 7168, 2048, "decode"),
    (1, 2048, 7168, "decode"),
    (16, 2048, 7168, "decode"),
    (64, 2048, 7168, "decode"),
    (5, 264, 384, "normal"),        # small M, ragged N tile
    (33, 1000, 1280, "normal"),
    (17, 128, 16384, "decode"),     # split-K over one N tile
    (3, 3840, 1280, "decode"),      # K split over an 8-CTA cluster, fewer rows than CTAs
    (33, 2816, 768, "decode"),      # 6-CTA cluster, uneven row shares
    (20, 1536, 7168, "decode"),     # 12-CTA cluster (above the portable size)
    (2, 24576, 1536, "decode"),     # one whole tile per CTA, no split
    (130, 256, 400, "normal"),      # partial last K block (16 of 128 columns), 256-wide tiles
    (300, 520, 144, "prefill"),     # K = 144: two K blocks, the second 16 wide
    (70, 1001, 208, "normal"),      # N odd: element-store epilogue; partial K block
    (100, 2056, 1040, "prefill"),   # N >= 2048 with a partial 256-wide tile, K % 128 = 16
    (5, 777, 400, "decode"),        # small M: partial K block, N odd
    (48, 3000, 2064, "decode"),     # small M, clusters, partial last K block
    # a wave or more of whole tiles (CTAs loop over several tiles)
    (517, 7936, 1024, "prefill"),   # 5 M blocks, the last one 5 rows: TMA and direct stores
    (1300, 4000, 640, "normal"),    # 11 M blocks, partial last N tile
    (1300, 1800, 272, "normal"),    # 128-wide N tiles, partial last K block
    (2100, 2060, 384, "prefill"),   # N % 8 != 0: direct stores only, 17 M blocks
    # deeper K with a partial last round of tiles
    (2100, 2060, 2048, "prefill"),  # 153 tiles: one CTA takes a second tile
    (1700, 4096, 2560, "normal"),   # 224 tiles: 72 CTAs take a second tile
])
def test_dense_matches_oracle(M, N, K, kind):
    A, sA, B, sB = quantised_dense(M, N, K, kind, seed=M * 7 + N)
    got = _run(A, sA, B, sB)
    ref = ogemm.gemm_dense(A, sA, B, sB)
    assert_close(got, ref, f"dense {M}x{N}x{K}")


@pytest.mark.parametrize("M", [1, 16, 64])
def test_small_m_is_deterministic(M):
    A, sA, B, sB = quantised_dense(M, 7168, 2048, "decode", seed=3)
    b = _b()
    tA, tsA, tB, tsB = dev(A), dev(sA), dev(B), dev(sB)
    d1 = host(b.fp8gemm_dense(tA, tsA, tB, tsB))
    d2 = host(b.fp8gemm_dense(tA, tsA, tB, tsB))
    assert np.array_equal(d1, d2)


def test_extreme_scales():
    """Large and tiny block scales whose products stay finite in FP32; errors
    must not concentrate in any K block."""
    M, N, K = 130, 256, 1024
    A, sA, B, sB = quantised_dense(M, N, K, "normal", seed=11)
    g = np.random.default_rng(12)
    sA = (sA * (2.0 ** g.integers(-60, 60, sA.shape))).astype(np.float32)
    sB = (sB * (2.0 ** g.integers(-40, 40, sB.shape))).astype(np.float32)
    got = _run(A, sA, B, sB)
    ref = ogemm.gemm_dense(A, sA, B, sB)
    assert_close(got, ref, "extreme scales")


@pytest.mark.slow
@pytest.mark.parametrize("M,N,K", [(4096, 4096, 4096), (4096, 7168, 16384)])
def test_prefill_full_size_sampled(M, N, K):
    """Full prefill size, launched exactly as the benchmark does; the oracle
    computes a sample of rows x columns (including the last tile's edges)."""
    A, sA, B, sB = quantised_dense(M, N, K, "prefill", seed=0)
    got = _run(A, sA, B, sB)
    rows, cols = sample_rows_cols(M, N, 48, 96, seed=1)
    rows = np.unique(np.concatenate([rows, [127, 128, M - 128]]))
    cols = np.unique(np.concatenate([cols, [255, 256, N - 256]]))
    ref = ogemm.gemm_dense_at(A, sA, B, sB, rows, cols)
    assert_close(got[rows][:, cols], ref, f"prefill {M}x{N}x{K}")
    assert np.isfinite(got).all()


@pytest.mark.parametrize("M,N,K", [(4, 2048, 1024), (64, 7168, 2048), (16, 2048, 7168)])
def test_decode_chain_without_host_sync(M, N, K):
    """The decode GEMM is launched as a programmatic dependent of the previous
    kernel.  Run it right after the kernels that produce its A and B, and
    three GEMMs back to back sharing the stream's split-K workspace, with no
    host synchronisation in between."""
    from fp8_fine_grained_e4m3_gb300 import synthetic
    b = _b()
    outs, refs = [], []
    for seed in (21, 22, 23):
        X, W = synthetic.dense_operands(M, N, K, kind="decode", seed=seed)
        A8, sA = b.fp8_quant_1x128(dev(X))
        B8, sB = b.fp8_quant_128x128(dev(W))
        outs.append(b.fp8gemm_dense(A8, sA, B8, sB))
        Ao, sAo = oquant.quant_1x128_fast(X)
        Bo, sBo = oquant.quant_128x128_fast(W)
        refs.append(ogemm.gemm_dense(Ao, sAo, Bo, sBo))
    for got, ref in zip(outs, refs):
        assert_close(host(got), ref, f"chained decode {M}x{N}x{K}")
    assert b.fp8gemm_get_device_status() == b.OK


@pytest.mark.parametrize("M,N,K", [
    (2560, 4096, 2048),  # whole tiles after a multi-wave (plain-launch) quantiser
    (1280, 4096, 1024),  # 160 whole tiles after a one-wave quantiser
    (256, 4096, 4096),   # 32 tiles split along K over clusters
    (96, 2048, 4096),    # one-wave quantiser (a programmatic dependent itself), split tiles
])
def test_large_m_chain_without_host_sync(M, N, K):
    """The tensor-core GEMM is launched as a programmatic dependent of the
    previous kernel and lets the next one launch early.  Quantise the FP32
    activations and run the GEMM right after, three such pairs back to back,
    with no host synchronisation in between: each GEMM must read what its
    quantiser wrote."""
    from fp8_fine_grained_e4m3_gb300 import synthetic
    b = _b()
    _, W = synthetic.dense_operands(M, N, K, kind="prefill", seed=5)
    Bo, sBo = quant_weights(W)
    B8, sB = dev(Bo), dev(sBo)
    outs, xs = [], []
    for seed in (31, 32, 33):
        X, _ = synthetic.dense_operands(M, 8, K, kind="prefill", seed=seed)
        A8, sA = b.fp8_quant_1x128(dev(X))
        outs.append(b.fp8gemm_dense(A8, sA, B8, sB))
        xs.append(X)
    for X, got in zip(xs, outs):
        Ao, sAo = oquant.quant_1x128_fast(X)
        assert_close(host(got), ogemm.gemm_dense(Ao, sAo, Bo, sBo), f"chained {M}x{N}x{K}")
    assert b.fp8gemm_get_device_status() == b.OK


def test_two_streams_with_library_workspaces():
    """Calls that use the library's per-stream workspaces (split-K partials
    and counters of the decode path; the quantised A of the FP32-activation
    call) issued on two streams with no ordering between them: each stream
    has its own workspace, so the results are those of running them alone."""
    import torch
    b = _b()
    cases = []
    for seed, (M, N, K) in enumerate([(17, 128, 16384), (33, 1000, 1280), (5, 128, 131072)]):
        A, sA, B, sB = quantised_dense(M, N, K, "decode", seed=60 + seed)
        cases.append(((dev(A), dev(sA), dev(B), dev(sB)), ogemm.gemm_dense(A, sA, B, sB)))
    X = synthetic_ops(200, 2304, 1024)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    torch.cuda.synchronize()
    for rep in range(3):
        for i, ((tA, tsA, tB, tsB), _) in enumerate(cases):
            s = s1 if (i + rep) % 2 == 0 else s2
            with torch.cuda.stream(s):
                outs.append((i, b.fp8gemm_dense(tA, tsA, tB, tsB)))
        with torch.cuda.stream(s2 if rep % 2 == 0 else s1):
            outs.append((-1, b.fp8gemm_dense_quant_a(X[0], X[1], X[2])))
    torch.cuda.synchronize()
    for i, D in outs:
        ref = cases[i][1] if i >= 0 else X[3]
        assert_close(host(D), ref, f"two streams, case {i}")
    assert b.fp8gemm_get_device_status() == b.OK


def synthetic_ops(M, N, K):
    """FP32 activations, oracle-quantised weights and the reference result of
    fp8gemm_dense_quant_a for them."""
    from fp8_fine_grained_e4m3_gb300 import synthetic
    Xf, Wf = synthetic.dense_operands(M, N, K, kind="decode", seed=70)
    Ao, sAo = oquant.quant_1x128_fast(Xf)
    Bo, sBo = oquant.quant_128x128_fast(Wf)
    return dev(Xf), dev(Bo), dev(sBo), ogemm.gemm_dense(Ao, sAo, Bo, sBo)


@pytest.mark.parametrize("M,N,K", [
    (1, 7168, 2048),     # 5-CTA clusters
    (64, 2048, 7168),    # 8-CTA clusters
    (20, 1536, 7168),    # 12-CTA clusters
    (17, 128, 16384),    # stream-K: the split-K workspace
    (33, 1000, 1280),    # stream-K, ragged N tile
])
def test_read_only_weights_flag_in_a_chain(M, N, K):
    """FP8GEMM_FLAG_B_READ_ONLY: the decode kernel stages its first weight
    tiles before waiting for the kernel ahead of it.  Each GEMM's activations
    are quantised by the kernel launched just before it (no host sync), so the
    activation side must still wait; the weights are constant."""
    from fp8_fine_grained_e4m3_gb300 import synthetic
    b = _b()
    _, W = synthetic.dense_operands(1, N, K, kind="decode", seed=N + K)
    Bo, sBo = oquant.quant_128x128_fast(W) if K % 128 == 0 else oquant.quant_128x128(W)
    tB, tsB = dev(Bo), dev(sBo)
    outs, refs = [], []
    for seed in (51, 52, 53):
        X, _ = synthetic.dense_operands(M, 8, K, kind="decode", seed=seed)
        tX = dev(X * np.float32(0.5)) * 2.0  # written by a kernel just before
        A8, sA = b.fp8_quant_1x128(tX)
        outs.append(b.fp8gemm_dense_ex(A8, sA, "e4m3", tB, tsB, "e4m3",
                                       flags=b.FLAG_B_READ_ONLY))
        Ao, sAo = oquant.quant_1x128_fast(X)
        refs.append(ogemm.gemm_dense(Ao, sAo, Bo, sBo))
    for got, ref in zip(outs, refs):
        assert_close(host(got), ref, f"read-only weights {M}x{N}x{K}")
    assert b.fp8gemm_get_device_status() == b.OK
