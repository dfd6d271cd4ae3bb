"""MoE grouped GEMMs (contiguous and masked) on the GPU vs the oracle."""

import numpy as np
import pytest

from fp8_fine_grained_e4m3_gb300 import synthetic
from tests.gpu_helpers import (assert_close, dev, host, ogemm, oquant, quant_weights,
                               rotated_experts, sample_rows_cols)

pytestmark = pytest.mark.gpu

SENTINEL = 0xFFFF  # a bf16 NaN bit pattern that no result can take


def _b():
    from fp8_fine_grained_e4m3_gb300 import binding
    return binding


def _contig_case(E, T, N, K, seed, counts=None):
    X, W, lay = synthetic.contiguous_operands(E, T, N, K, seed=seed, counts=counts)
    A, sA = oquant.quant_1x128_fast(X)
    Bq = [quant_weights(W[e]) for e in range(E)]
    B = np.stack([q for q, _ in Bq])
    sB = np.stack([s for _, s in Bq])
    return A, sA, B, sB, lay


def _run_contig(A, sA, B, sB, m_indices):
    return host(_b().fp8gemm_grouped_contiguous(dev(A), dev(sA), dev(B), dev(sB),
                                                dev(m_indices.astype(np.int32))))


def test_contiguous_two_experts_eight_tokens():
    A, sA, B, sB, lay = _contig_case(2, 16, 256, 256, seed=1, counts=np.array([8, 8]))
    got = _run_contig(A, sA, B, sB, lay.m_indices)
    assert_close(got, ogemm.gemm_contiguous(A, sA, B, sB, lay.m_indices), "2x8")


@pytest.mark.parametrize("E,T,N,K", [(5, 300, 384, 512), (8, 1000, 512, 1024), (3, 200, 2048, 256),
                                     (4, 300, 300, 400),  # partial last K block, N % 8 != 0
                                     (6, 2500, 4096, 2048)])  # 368 tiles: a partial last round
def test_contiguous_matches_oracle(E, T, N, K):
    A, sA, B, sB, lay = _contig_case(E, T, N, K, seed=E + T)
    got = _run_contig(A, sA, B, sB, lay.m_indices)
    assert_close(got, ogemm.gemm_contiguous(A, sA, B, sB, lay.m_indices), f"contig E={E}")


def test_contiguous_empty_expert_and_padding_block():
    counts = np.array([130, 0, 0, 5])
    A, sA, B, sB, lay = _contig_case(4, 135, 256, 384, seed=3, counts=counts)
    # append one whole padding block (first index -1): it must be skipped
    A = np.concatenate([A, np.zeros((128, 384), np.uint8)])
    sA = np.concatenate([sA, np.zeros((128, 3), np.float32)])
    mi = np.concatenate([lay.m_indices, np.full(128, -1, np.int32)])
    got = _run_contig(A, sA, B, sB, mi)
    assert_close(got, ogemm.gemm_contiguous(A, sA, B, sB, mi), "empty expert")


@pytest.mark.slow
def test_contiguous_full_size_sampled():
    """32 experts, 8192 Zipf(1.1) tokens, N=4096, K=7168, as the benchmark
    launches it.  Experts' weights are the 128-row-tile rotations of one
    quantised matrix (distinct per expert)."""
    E, T, N, K = 32, 8192, 4096, 7168
    counts = synthetic.zipf_counts(E, T, seed=0)
    lay = synthetic.contiguous_layout(counts)
    X, W = synthetic.dense_operands(lay.M_pad, N, K, kind="decode", seed=0)
    X[lay.m_indices < 0] = 0
    A, sA = oquant.quant_1x128_fast(X)
    B0, sB0 = oquant.quant_128x128_fast(W)
    B, sB = rotated_experts(B0, sB0, E)
    got = _run_contig(A, sA, B, sB, lay.m_indices)
    real = np.nonzero(lay.m_indices >= 0)[0]
    g = np.random.default_rng(2)
    rows = np.unique(np.concatenate([g.choice(real, 64), lay.offsets[counts > 0]]))
    _, cols = sample_rows_cols(1, N, 1, 96, seed=3)
    ref = np.full((len(rows), len(cols)), np.nan)
    for e in range(E):
        sel = np.nonzero(lay.m_indices[rows] == e)[0]
        if sel.size:
            ref[sel] = ogemm.gemm_dense_at(A, sA, B[e], sB[e], rows[sel], cols)
    assert_close(got[rows][:, cols], ref, "contiguous full size")


def _masked_case(E, M_max, N, K, masked_m, seed):
    X, W, mm = synthetic.masked_operands(E, M_max, N, K, seed=seed, masked_m=masked_m)
    A, sA = oquant.quant_1x128_fast(X.reshape(-1, K))
    A, sA = A.reshape(E, M_max, K), sA.reshape(E, M_max, -(-K // 128))
    Bq = [quant_weights(W[e]) for e in range(E)]
    B = np.stack([q for q, _ in Bq])
    sB = np.stack([s for _, s in Bq])
    return A, sA, B, sB, mm


def _run_masked(A, sA, B, sB, mm):
    import torch
    E, M_max, _ = A.shape
    N = B.shape[1]
    D = torch.full((E, M_max, N), 0, dtype=torch.int16, device="cuda")
    D.fill_(np.int16(np.uint16(SENTINEL).view(np.int16)))
    D = D.view(torch.bfloat16)
    _b().fp8gemm_grouped_masked(dev(A), dev(sA), dev(B), dev(sB), dev(mm.astype(np.int32)), D=D)
    bits = D.view(torch.int16).cpu().numpy().view(np.uint16)
    return host(D), bits


@pytest.mark.parametrize("E,M_max,N,K,mm", [
    (4, 160, 256, 256, [0, 160, 5, 129]),
    (3, 256, 512, 512, [256, 1, 128]),
    (6, 64, 2048, 384, [64, 0, 0, 63, 1, 17]),
    (3, 200, 250, 272, [200, 7, 0]),  # partial last K block, N % 8 != 0
    # 160 tiles over the SMs: 8 CTAs take a second tile
    (10, 128, 4096, 4096, [128, 1, 77, 128, 5, 100, 128, 64, 3, 128]),
])
def test_masked_matches_oracle_and_leaves_rows(E, M_max, N, K, mm):
    mm = np.array(mm, np.int32)
    A, sA, B, sB, mm = _masked_case(E, M_max, N, K, mm, seed=E + N)
    got, bits = _run_masked(A, sA, B, sB, mm)
    ref = ogemm.gemm_masked(A, sA, B, sB, mm)
    assert_close(got, ref, "masked")
    for e in range(E):
        assert np.all(bits[e, mm[e]:] == SENTINEL), f"expert {e} rows >= masked_m written"
        assert not np.any(bits[e, :mm[e]] == SENTINEL)


@pytest.mark.slow
def test_masked_full_size_sampled():
    E, M_max, N, K = 16, 256, 4096, 7168
    mm = synthetic.masked_counts(E, M_max, seed=0)
    X, _, _ = synthetic.masked_operands(E, M_max, 8, K, seed=0, masked_m=mm)
    A, sA = oquant.quant_1x128_fast(X.reshape(-1, K))
    A, sA = A.reshape(E, M_max, K), sA.reshape(E, M_max, -(-K // 128))
    _, W = synthetic.dense_operands(1, N, K, kind="decode", seed=1)
    B0, sB0 = oquant.quant_128x128_fast(W)
    B, sB = rotated_experts(B0, sB0, E)
    got, bits = _run_masked(A, sA, B, sB, mm)
    _, cols = sample_rows_cols(1, N, 1, 64, seed=4)
    for e in range(E):
        assert np.all(bits[e, mm[e]:] == SENTINEL)
        if mm[e] == 0:
            continue
        rows = np.unique(np.array([0, mm[e] - 1, mm[e] // 2, min(127, mm[e] - 1)]))
        ref = ogemm.gemm_dense_at(A[e], sA[e], B[e], sB[e], rows, cols)
        assert_close(got[e][rows][:, cols], ref, f"masked expert {e}")


@pytest.mark.parametrize("form", ["masked", "contiguous"])
def test_grouped_after_quantiser_without_host_sync(form):
    """The grouped GEMMs are launched as programmatic dependents of the
    previous kernel: quantise each batch's FP32 activations on the device and
    run the GEMM right after, two batches back to back, no host sync."""
    b = _b()
    E, N, K = 6, 2048, 4096
    outs, refs = [], []
    for seed in (41, 42):
        if form == "masked":
            mm = np.array([256, 1, 130, 0, 64, 200], np.int32)
            X, W, mm = synthetic.masked_operands(E, 256, N, K, seed=seed, masked_m=mm)
            Xf = X.reshape(-1, K)
        else:
            X, W, lay = synthetic.contiguous_operands(E, 900, N, K, seed=seed)
            Xf = X
        Bq = [quant_weights(W[e]) for e in range(E)]
        B = np.stack([q for q, _ in Bq])
        sB = np.stack([s for _, s in Bq])
        A8, sA = b.fp8_quant_1x128(dev(Xf))
        Ao, sAo = oquant.quant_1x128_fast(Xf)
        if form == "masked":
            A8, sA = A8.view(E, 256, K), sA.view(E, 256, K // 128)
            outs.append((b.fp8gemm_grouped_masked(A8, sA, dev(B), dev(sB), dev(mm)), mm))
            refs.append(ogemm.gemm_masked(Ao.reshape(E, 256, K), sAo.reshape(E, 256, -1), B, sB, mm))
        else:
            mi = lay.m_indices.astype(np.int32)
            outs.append((b.fp8gemm_grouped_contiguous(A8, sA, dev(B), dev(sB), dev(mi)), None))
            refs.append(ogemm.gemm_contiguous(Ao, sAo, B, sB, mi))
    for (got, mm), ref in zip(outs, refs):
        got = host(got)
        if mm is not None:  # rows past masked_m are not outputs
            for e in range(E):
                assert_close(got[e, :mm[e]], ref[e, :mm[e]], f"{form} expert {e}")
        else:
            assert_close(got, ref, form)
    assert b.fp8gemm_get_device_status() == b.OK
