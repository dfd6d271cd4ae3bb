"""Tiles split along K (problems whose tiles all fit in one wave of CTAs) on
the GPU vs the oracle: each tile gets a cluster of CTAs whose FP32 partials
are summed in rank order through distributed shared memory, so results are
also checked for run-to-run identity, across launches of different cluster
sizes."""

import numpy as np
import pytest

from tests.gpu_helpers import assert_close, dev, host, ogemm, quantised_dense
from tests.test_gpu_grouped import SENTINEL, _masked_case, _run_masked

pytestmark = pytest.mark.gpu


def _b():
    from fp8_fine_grained_e4m3_gb300 import binding
    return binding


@pytest.mark.parametrize("M,N,K,kind", [
    (128, 4096, 7168, "prefill"),   # 16 tiles, clusters of 8 parts of 7 K blocks
    (256, 7168, 4096, "decode"),    # 56 tiles, clusters of 2
    (200, 1000, 4112, "normal"),    # 128-wide tiles, 8 parts over 33 K blocks (last 16 wide)
    (96, 300, 4096, "normal"),      # 3 tiles, ragged rows, N % 8 != 0
])
def test_split_dense_matches_oracle_and_repeats(M, N, K, kind):
    A, sA, B, sB = quantised_dense(M, N, K, kind, seed=M + N + K)
    b = _b()
    tA, tsA, tB, tsB = dev(A), dev(sA), dev(B), dev(sB)
    d1 = host(b.fp8gemm_dense(tA, tsA, tB, tsB))
    assert_close(d1, ogemm.gemm_dense(A, sA, B, sB), f"split dense {M}x{N}x{K}")
    d2 = host(b.fp8gemm_dense(tA, tsA, tB, tsB))
    assert np.array_equal(d1, d2), "split reduction not deterministic"


def test_split_repeats_across_cluster_sizes():
    """Launches with different cluster sizes back to back, repeated: each
    result matches the oracle and its own first run bit for bit."""
    b = _b()
    cases = []
    for (M, N, K) in ((128, 4096, 4096), (256, 7168, 4096), (384, 2048, 4096)):
        A, sA, B, sB = quantised_dense(M, N, K, "normal", seed=M * 3 + K)
        t = (dev(A), dev(sA), dev(B), dev(sB))
        ref = host(b.fp8gemm_dense(*t))
        assert_close(ref, ogemm.gemm_dense(A, sA, B, sB), f"{M}x{N}x{K}")
        cases.append((t, ref))
    for _ in range(3):
        for t, ref in cases:
            assert np.array_equal(host(b.fp8gemm_dense(*t)), ref)
    assert b.fp8gemm_get_device_status() == b.OK


def test_split_masked_idle_clusters():
    """Masked form with few possible tiles: one cluster per possible tile,
    and the clusters past the valid tiles (empty experts) find no work."""
    E, M_max, N, K = 20, 128, 262, 4096  # 128-wide tiles, N % 4 != 0: element stores
    g = np.random.default_rng(5)
    mm = g.integers(1, M_max + 1, E).astype(np.int32)
    mm[g.choice(E, 6, replace=False)] = 0
    A, sA, B, sB, mm = _masked_case(E, M_max, N, K, mm, seed=9)
    got, bits = _run_masked(A, sA, B, sB, mm)
    assert_close(got, ogemm.gemm_masked(A, sA, B, sB, mm), "masked, idle clusters")
    for e in range(E):
        assert np.all(bits[e, mm[e]:] == SENTINEL)
        assert not np.any(bits[e, :mm[e]] == SENTINEL)


def test_split_masked_all_empty():
    E, M_max, N, K = 4, 64, 256, 256
    mm = np.zeros(E, np.int32)
    A, sA, B, sB, mm = _masked_case(E, M_max, N, K, mm, seed=2)
    _, bits = _run_masked(A, sA, B, sB, mm)
    assert np.all(bits == SENTINEL)
    assert _b().fp8gemm_get_device_status() == _b().OK
