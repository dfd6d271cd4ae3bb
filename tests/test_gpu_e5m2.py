"""e5m2 operands: the quantisers with fmt = e5m2 bit for bit against the
oracle, and the dense GEMM with every mix of e4m3 / e5m2 operands against the
oracle within the GEMM tolerance, on the large-M, decode-cluster and stream-K
paths."""

import numpy as np
import pytest

from fp8_fine_grained_e4m3_gb300 import synthetic
from oracle import quant as oq
from tests.gpu_helpers import assert_close, dev, host, ogemm

pytestmark = pytest.mark.gpu


def _b():
    from fp8_fine_grained_e4m3_gb300 import binding
    return binding


def _q128(W, fmt):
    return oq.quant_128x128_fast(W, fmt=fmt) if W.shape[-1] % 128 == 0 else oq.quant_128x128(W, fmt=fmt)


@pytest.mark.parametrize("M,K", [(64, 7168), (300, 400), (3000, 1024)])
def test_quant_1x128_e5m2_bit_exact(M, K):
    X, _ = synthetic.dense_operands(M, 8, K, kind="prefill", seed=M + K)
    X[1] *= np.float32(1e6)   # a row far above e4m3's range: e5m2 keeps its relative precision
    X[2] = 0.0
    Q, S = _b().fp8_quant_1x128_fmt(dev(X), "e5m2")
    Qo, So = oq.quant_1x128_fast(X, fmt="e5m2")
    assert np.array_equal(host(Q), Qo)
    assert np.array_equal(host(S).view(np.uint32), So.view(np.uint32))


@pytest.mark.parametrize("E,N,K", [(1, 300, 512), (2, 256, 400)])
def test_quant_128x128_e5m2_bit_exact(E, N, K):
    _, W, _ = synthetic.masked_operands(E, 1, N, K, seed=N + K)
    Q, S = _b().fp8_quant_128x128_fmt(dev(W), "e5m2")
    for e in range(E):
        Qo, So = _q128(W[e], "e5m2")
        assert np.array_equal(host(Q)[e], Qo)
        assert np.array_equal(host(S)[e].view(np.uint32), So.view(np.uint32))


@pytest.mark.parametrize("a_fmt,b_fmt", [("e5m2", "e5m2"), ("e5m2", "e4m3"), ("e4m3", "e5m2")])
@pytest.mark.parametrize("M,N,K", [
    (256, 512, 640),     # large M, 256-wide tiles
    (300, 520, 384),     # large M, 128-wide tiles
    (16, 2048, 7168),    # decode, 8-CTA clusters
    (33, 1000, 1280),    # decode, stream-K
    (5, 777, 400),       # decode, partial K block, N odd
])
def test_dense_mixed_formats(M, N, K, a_fmt, b_fmt):
    b = _b()
    X, W = synthetic.dense_operands(M, N, K, kind="prefill", seed=M * 3 + N)
    A, sA = oq.quant_1x128_fast(X, fmt=a_fmt)
    B, sB = _q128(W, b_fmt)
    got = host(b.fp8gemm_dense_fmt(dev(A), dev(sA), a_fmt, dev(B), dev(sB), b_fmt))
    ref = ogemm.gemm_dense(A, sA, B, sB, a_fmt=a_fmt, b_fmt=b_fmt)
    assert_close(got, ref, f"{a_fmt} x {b_fmt} {M}x{N}x{K}")
    assert b.fp8gemm_get_device_status() == b.OK


def test_e4m3_through_fmt_call_is_the_plain_call():
    b = _b()
    X, W = synthetic.dense_operands(130, 512, 1024, kind="normal", seed=4)
    A, sA = oq.quant_1x128_fast(X)
    B, sB = oq.quant_128x128_fast(W)
    tA, tsA, tB, tsB = dev(A), dev(sA), dev(B), dev(sB)
    d1 = host(b.fp8gemm_dense(tA, tsA, tB, tsB))
    d2 = host(b.fp8gemm_dense_fmt(tA, tsA, "e4m3", tB, tsB, "e4m3"))
    assert np.array_equal(d1, d2)


@pytest.mark.parametrize("a_fmt,b_fmt", [("e5m2", "e4m3"), ("e4m3", "e5m2")])
def test_grouped_mixed_formats(a_fmt, b_fmt):
    """Contiguous and masked grouped forms with e5m2 operands."""
    import torch
    b = _b()
    E, N, K = 3, 384, 512
    X, W, lay = synthetic.contiguous_operands(E, 300, N, K, seed=9)
    A, sA = oq.quant_1x128_fast(X, fmt=a_fmt)
    Bq = [_q128(W[e], b_fmt) for e in range(E)]
    B = np.stack([q for q, _ in Bq])
    sB = np.stack([s_ for _, s_ in Bq])
    got = host(b.fp8gemm_grouped_contiguous_fmt(dev(A), dev(sA), a_fmt, dev(B), dev(sB), b_fmt,
                                                dev(lay.m_indices.astype(np.int32))))
    ref = ogemm.gemm_contiguous(A, sA, B, sB, lay.m_indices, a_fmt, b_fmt)
    assert_close(got, ref, f"contiguous {a_fmt} x {b_fmt}")

    Xm, Wm, mm = synthetic.masked_operands(E, 160, N, K, seed=10,
                                           masked_m=np.array([160, 0, 37], np.int32))
    Am, sAm = oq.quant_1x128_fast(Xm.reshape(-1, K), fmt=a_fmt)
    Am, sAm = Am.reshape(E, 160, K), sAm.reshape(E, 160, -1)
    Bq = [_q128(Wm[e], b_fmt) for e in range(E)]
    Bm = np.stack([q for q, _ in Bq])
    sBm = np.stack([s_ for _, s_ in Bq])
    D = torch.zeros((E, 160, N), dtype=torch.bfloat16, device="cuda")
    b.fp8gemm_grouped_masked_fmt(dev(Am), dev(sAm), a_fmt, dev(Bm), dev(sBm), b_fmt,
                                 dev(mm), D=D)
    ref = ogemm.gemm_masked(Am, sAm, Bm, sBm, mm, a_fmt, b_fmt)
    assert_close(host(D), ref, f"masked {a_fmt} x {b_fmt}")
    assert b.fp8gemm_get_device_status() == b.OK
