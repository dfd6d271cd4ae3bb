"""Failure detection without a GPU fault: every pipeline wait in the GEMM
kernels is bounded.  With the limit set to 1 ns (fp8gemm_set_wait_limit_ns)
a genuine wait -- for a tile's copies to land, or for the tensor cores --
runs out on a whole-tile dense case (no cluster barriers involved): the CTA
gives up, lets its copies and MMAs in flight finish, frees TMEM and exits;
the status word reads FP8GEMM_ERR_TIMEOUT, and the next call, at the default
limit, is correct against the oracle on the same context."""

import pytest

from tests.gpu_helpers import assert_close, dev, host, ogemm, quantised_dense

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_the_context_stays_usable():
    from fp8_fine_grained_e4m3_gb300 import binding as b
    # 16 x 10 = 160 tiles >= the SMs: the persistent whole-tile instance
    M, N, K = 2048, 2560, 1024
    A, sA, B, sB = quantised_dense(M, N, K, "normal", seed=41)
    ops = (dev(A), dev(sA), dev(B), dev(sB))
    ref = ogemm.gemm_dense(A, sA, B, sB)
    # a decode call that keeps a split-K workspace on this stream
    Ad, sAd, Bd, sBd = quantised_dense(17, 128, 16384, "decode", seed=42)
    dops = (dev(Ad), dev(sAd), dev(Bd), dev(sBd))
    dref = ogemm.gemm_dense(Ad, sAd, Bd, sBd)
    assert_close(host(b.fp8gemm_dense(*dops)), dref, "decode before")
    assert b.fp8gemm_get_device_status() == b.OK
    try:
        b.set_wait_limit_ns(1)
        b.fp8gemm_dense(*ops)
        status = b.fp8gemm_get_device_status()
    finally:
        b.set_wait_limit_ns(0)
    assert status == b.ERR_TIMEOUT, b.strerror(status)
    assert b.workspace_bytes() == 0  # dropped after the timeout
    assert_close(host(b.fp8gemm_dense(*ops)), ref, "dense after the timeout")
    assert_close(host(b.fp8gemm_dense(*dops)), dref, "decode after the timeout")
    assert b.fp8gemm_get_device_status() == b.OK


def test_batched_launch_timeout_leaves_the_next_launch_correct():
    """The batched launch's extra waits (its tile ring) are bounded too: at a
    1 ns limit the launch gives up with FP8GEMM_ERR_TIMEOUT, every CTA still
    exits, and the next batched launches (on fresh counters: the timeout read
    drops the workspaces) match the oracle."""
    from fp8_fine_grained_e4m3_gb300 import binding as b
    shapes = [(2048, 2560, 1024), (640, 768, 512)]
    probs = [quantised_dense(M, N, K, "normal", seed=50 + i) for i, (M, N, K) in enumerate(shapes)]
    ops = [tuple(dev(x) for x in p) for p in probs]
    refs = [ogemm.gemm_dense(*p) for p in probs]
    for D, r in zip(b.fp8gemm_dense_batch(ops), refs):  # the stream's counters exist
        assert_close(host(D), r, "batch before")
    assert b.fp8gemm_get_device_status() == b.OK
    try:
        b.set_wait_limit_ns(1)
        b.fp8gemm_dense_batch(ops)
        status = b.fp8gemm_get_device_status()
    finally:
        b.set_wait_limit_ns(0)
    assert status == b.ERR_TIMEOUT, b.strerror(status)
    assert b.workspace_bytes() == 0
    for _ in range(2):
        for D, r in zip(b.fp8gemm_dense_batch(ops), refs):
            assert_close(host(D), r, "batch after the timeout")
    assert b.fp8gemm_get_device_status() == b.OK
