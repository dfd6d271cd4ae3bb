"""fp8gemm_dense_quant_a: the dense GEMM on FP32 activations, quantised 1x128
on the way in (the quantiser, then the GEMM as its programmatic dependent).
The quantised bytes and scales must equal the oracle's bit for bit, D must
meet the GEMM tolerance against the oracle, and D must equal the separate
calls (fp8_quant_1x128, then fp8gemm_dense) bit for bit."""

import numpy as np
import pytest

from fp8_fine_grained_e4m3_gb300 import synthetic
from tests.gpu_helpers import assert_close, dev, host, ogemm, oquant, quant_weights

pytestmark = pytest.mark.gpu


def _b():
    from fp8_fine_grained_e4m3_gb300 import binding
    return binding


def _weights(N, K, seed):
    _, W = synthetic.dense_operands(1, N, K, kind="decode", seed=seed)
    return quant_weights(W)


@pytest.mark.parametrize("M,N,K", [
    (1, 7168, 2048),     # decode: 5-CTA clusters
    (16, 2048, 7168),    # decode: 8-CTA clusters
    (20, 1536, 7168),    # decode: 12-CTA clusters
    (64, 7168, 2048),
    (33, 1000, 1280),    # stream-K, ragged N tile
    (5, 264, 384),
    (17, 128, 16384),    # one N tile, split-K reduction
    (5, 128, 131072),    # stream-K across tile boundaries
    (200, 2304, 1024),   # large-M GEMM
    (3, 1000, 400),      # partial last K block
    (150, 333, 272),     # large M, N odd, partial K block
    (16, 7168, 2064),    # partial last K block (17 blocks over 5-CTA clusters)
    (48, 3000, 2064),    # 48 of 64 rows, 8-CTA clusters, partial K block
    # quantised inside the decode GEMM (a few rows, K range within the stages)
    (3, 7168, 2064),     # 3 of 16 rows, partial last K block, 5-CTA clusters
    (4, 3000, 2048),     # 8-CTA clusters, 2 K blocks each
    (2, 1536, 7168),     # 12-CTA clusters (above the portable size)
    (1, 2048, 7168),     # 7 K blocks per CTA, more than the stages: quantiser, then the GEMM
    (2, 2048, 7168),
])
def test_quant_a_matches_oracle_and_two_call_path(M, N, K):
    b = _b()
    X, _ = synthetic.dense_operands(M, 8, K, kind="decode", seed=M + K)
    if M > 1:
        X[M // 2] = 0.0  # a zero row: s = 0, bytes 0
    Bq, sB = _weights(N, K, seed=N)
    tX, tB, tsB = dev(X), dev(Bq), dev(sB)
    import torch
    Q = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    sA = torch.empty((M, -(-K // 128)), dtype=torch.float32, device="cuda")
    D = b.fp8gemm_dense_quant_a(tX, tB, tsB, Q=Q, sA=sA)
    Qo, sAo = oquant.quant_1x128_fast(X)
    assert np.array_equal(host(Q), Qo)
    assert np.array_equal(host(sA).view(np.uint32), sAo.view(np.uint32))
    assert_close(host(D), ogemm.gemm_dense(Qo, sAo, Bq, sB), f"quant-on-load {M}x{N}x{K}")
    Q2, sA2 = b.fp8_quant_1x128(tX)
    D2 = b.fp8gemm_dense(Q2, sA2, tB, tsB)
    assert np.array_equal(host(D), host(D2))
    D3 = b.fp8gemm_dense_quant_a(tX, tB, tsB)  # without the optional outputs
    assert np.array_equal(host(D3), host(D))
    assert b.fp8gemm_get_device_status() == b.OK


def test_quant_a_chain_without_host_sync():
    """Activations produced by the previous kernel in the stream (the
    quantiser, launched as a programmatic dependent, waits for it before
    loading them), three calls back to back."""
    import torch
    b = _b()
    M, N, K = 16, 7168, 2048
    Bq, sB = _weights(N, K, seed=3)
    tB, tsB = dev(Bq), dev(sB)
    outs, xs = [], []
    for seed in (31, 32, 33):
        X, _ = synthetic.dense_operands(M, 8, K, kind="decode", seed=seed)
        base = dev(X * np.float32(0.5))
        tX = base * 2.0  # written by a kernel just before the GEMM
        outs.append(b.fp8gemm_dense_quant_a(tX, tB, tsB))
        xs.append(X)
    for X, D in zip(xs, outs):
        Qo, sAo = oquant.quant_1x128_fast(X)
        assert_close(host(D), ogemm.gemm_dense(Qo, sAo, Bq, sB), "chained quant-on-load")
    assert b.fp8gemm_get_device_status() == b.OK


def test_quant_a_rejects_half_given_outputs():
    import torch
    b = _b()
    X = torch.zeros((4, 256), dtype=torch.float32, device="cuda")
    B = torch.zeros((256, 256), dtype=torch.uint8, device="cuda")
    sB = torch.ones((2, 2), dtype=torch.float32, device="cuda")
    Q = torch.empty((4, 256), dtype=torch.uint8, device="cuda")
    with pytest.raises(ValueError):
        b.fp8gemm_dense_quant_a(X, B, sB, Q=Q)


@pytest.mark.parametrize("M,N,K", [(1, 7168, 2048), (16, 2048, 7168), (33, 1000, 1280),
                                   (1, 2048, 7168)])
def test_quant_a_read_only_weights_chain(M, N, K):
    """fp8gemm_dense_quant_a_ex with FLAG_B_READ_ONLY: the GEMM stages its
    weights while the quantiser (its predecessor in the stream) runs; the
    activations come from the kernel just before; three calls back to back."""
    b = _b()
    Bq, sB = _weights(N, K, seed=N + 1)
    tB, tsB = dev(Bq), dev(sB)
    outs, xs = [], []
    for seed in (61, 62, 63):
        X, _ = synthetic.dense_operands(M, 8, K, kind="decode", seed=seed)
        tX = dev(X * np.float32(0.5)) * 2.0  # written by a kernel just before
        outs.append(b.fp8gemm_dense_quant_a(tX, tB, tsB, flags=b.FLAG_B_READ_ONLY))
        xs.append(X)
    for X, D in zip(xs, outs):
        Qo, sAo = oquant.quant_1x128_fast(X)
        assert_close(host(D), ogemm.gemm_dense(Qo, sAo, Bq, sB), "read-only quant-on-load")
    assert b.fp8gemm_get_device_status() == b.OK
