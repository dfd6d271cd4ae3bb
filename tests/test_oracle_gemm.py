"""Pins for the oracle's block-scaled GEMM (CPU only).

Each test fixes the oracle against something other than itself: brute-force
loops, a mathematically identical dequantise-then-matmul form, closed forms
(constant scale, identity, all-ones), linearity in one block's scale, and the
grouped forms against per-expert dense calls.  Shapes are non-square with
N > 128 so that a transposed operand or a wrong scale index fails.
"""

import math

import numpy as np
import pytest
import torch

from oracle import e4m3, gemm, quant
from fp8_fine_grained_e4m3_gb300 import synthetic


def _random_fp8(shape, seed):
    """Random finite e4m3 bytes (NaN codes excluded)."""
    g = np.random.default_rng(seed)
    q = g.integers(0, 256, size=shape, dtype=np.int64).astype(np.uint8)
    return np.where((q & 0x7F) == 0x7F, np.uint8(0x38), q).astype(np.uint8)


def _random_scales(shape, seed):
    g = np.random.default_rng(seed)
    return (2.0 ** g.uniform(-12, 4, size=shape)).astype(np.float32)


def _case(M, N, K, seed):
    A = _random_fp8((M, K), seed)
    B = _random_fp8((N, K), seed + 1)
    sA = _random_scales((M, -(-K // 128)), seed + 2)
    sB = _random_scales((-(-N // 128), -(-K // 128)), seed + 3)
    return A, sA, B, sB


def _bruteforce(A, sA, B, sB):
    """Triple loop in Python floats over the pages' formula, term by term."""
    M, K = A.shape
    N = B.shape[0]
    D = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            terms = []
            for k in range(K):
                kb = k // 128
                terms.append(e4m3.decode_code(A[m, k]) * e4m3.decode_code(B[n, k])
                             * float(sA[m, kb]) * float(sB[n // 128, kb]))
            D[m, n] = math.fsum(terms)
    return D


def _close(a, b, rtol=1e-12):
    scale = np.max(np.abs(b)) + 1e-300
    return np.max(np.abs(a - b)) <= rtol * scale


@pytest.mark.parametrize("M,N,K", [(3, 260, 256), (2, 5, 384)])
def test_bruteforce(M, N, K):
    A, sA, B, sB = _case(M, N, K, seed=M * 100 + N)
    if N > 128:  # keep the brute force quick: only some columns
        cols = np.array([0, 1, 127, 128, 200, 255, 256, N - 1])
        # one column at a time, handing the brute force that column's scale row
        ref = np.stack([_bruteforce(A, sA, B[c:c + 1], sB[c // 128:c // 128 + 1])[:, 0]
                        for c in cols], axis=1)
        got = gemm.gemm_dense(A, sA, B, sB)[:, cols]
    else:
        ref = _bruteforce(A, sA, B, sB)
        got = gemm.gemm_dense(A, sA, B, sB)
    assert _close(got, ref)


def test_dequantise_then_matmul():
    A, sA, B, sB = _case(37, 300, 640, seed=11)
    sA_full = np.repeat(sA.astype(np.float64), 128, axis=1)
    sB_full = np.repeat(np.repeat(sB.astype(np.float64), 128, axis=1), 128, axis=0)[:300]
    ref = (e4m3.decode(A) * sA_full) @ (e4m3.decode(B) * sB_full).T
    assert _close(gemm.gemm_dense(A, sA, B, sB), ref, 1e-13)


def test_constant_scale_closed_form():
    A, _, B, _ = _case(9, 130, 384, seed=12)
    a, b = np.float32(0.37), np.float32(5.5)
    sA = np.full((9, 3), a, np.float32)
    sB = np.full((2, 3), b, np.float32)
    ref = float(a) * float(b) * (e4m3.decode(A) @ e4m3.decode(B).T)
    assert _close(gemm.gemm_dense(A, sA, B, sB), ref, 1e-14)


def test_identity_closed_form():
    K = N = 256
    A, sA, _, _ = _case(5, N, K, seed=13)
    B = np.zeros((N, K), np.uint8)
    B[np.arange(N), np.arange(N)] = 0x38  # 1.0
    sB = np.ones((2, 2), np.float32)
    D = gemm.gemm_dense(A, sA, B, sB)
    expect = e4m3.decode(A) * np.repeat(sA.astype(np.float64), 128, axis=1)
    assert np.array_equal(D, expect)


def test_all_ones_is_k():
    A = np.full((4, 512), 0x38, np.uint8)
    B = np.full((256, 512), 0x38, np.uint8)
    D = gemm.gemm_dense(A, np.ones((4, 4), np.float32), B, np.ones((2, 4), np.float32))
    assert np.all(D == 512.0)
    assert np.all(gemm.bf16_rne(D) == 512.0)


def test_block_linearity():
    A, sA, B, sB = _case(6, 256, 512, seed=14)
    D0 = gemm.gemm_dense(A, sA, B, sB)
    sA2 = sA.copy()
    sA2[2, 1] *= 2
    D1 = gemm.gemm_dense(A, sA2, B, sB)
    blk = slice(128, 256)
    contrib = (float(sA[2, 1]) * np.repeat(sB[:, 1].astype(np.float64), 128)
               * (e4m3.decode(A[2, blk]) @ e4m3.decode(B[:, blk]).T))
    diff = D1 - D0
    assert _close(diff[2], contrib, 1e-12)
    assert np.all(diff[np.arange(6) != 2] == 0)


def test_scale_row_follows_n_block():
    # B's scale changes at n = 128: only columns >= 128 move with sB[1, :]
    A, sA, B, sB = _case(3, 256, 256, seed=15)
    D0 = gemm.gemm_dense(A, sA, B, sB)
    sB2 = sB.copy()
    sB2[1, :] *= 4
    D1 = gemm.gemm_dense(A, sA, B, sB2)
    assert np.array_equal(D0[:, :128], D1[:, :128])
    assert _close(D1[:, 128:], 4 * D0[:, 128:], 1e-15)


def test_dense_at_equals_full():
    A, sA, B, sB = _case(20, 384, 256, seed=16)
    rows = np.array([0, 7, 19])
    cols = np.array([3, 130, 131, 383, 0])
    full = gemm.gemm_dense(A, sA, B, sB)
    assert np.array_equal(gemm.gemm_dense_at(A, sA, B, sB, rows, cols), full[rows][:, cols])


def test_contiguous_two_experts_eight_tokens():
    # simplest fixed grouping first: 2 experts x 8 tokens each
    X, W, lay = synthetic.contiguous_operands(2, 16, 256, 256, seed=17,
                                              counts=np.array([8, 8]))
    assert lay.M_pad == 256 and list(lay.m_indices[:9]) == [0] * 8 + [-1]
    A, sA = quant.quant_1x128(X)
    B, sB = quant.quant_128x128_grouped(W)
    D = gemm.gemm_contiguous(A, sA, B, sB, lay.m_indices)
    assert np.array_equal(D[0:8], gemm.gemm_dense(A[0:8], sA[0:8], B[0], sB[0]))
    assert np.array_equal(D[128:136], gemm.gemm_dense(A[128:136], sA[128:136], B[1], sB[1]))
    assert np.all(np.isnan(D[8:128])) and np.all(np.isnan(D[136:]))


def test_contiguous_equals_per_expert_dense():
    X, W, lay = synthetic.contiguous_operands(5, 300, 256, 384, seed=18)
    A, sA = quant.quant_1x128(X)
    B, sB = quant.quant_128x128_grouped(W)
    D = gemm.gemm_contiguous(A, sA, B, sB, lay.m_indices)
    for e in range(5):
        o, c = lay.offsets[e], lay.counts[e]
        if c:
            assert np.array_equal(D[o:o + c], gemm.gemm_dense(A[o:o + c], sA[o:o + c], B[e], sB[e]))


def test_masked_equals_per_expert_dense():
    X, W, mm = synthetic.masked_operands(4, 32, 256, 256, seed=19,
                                         masked_m=np.array([0, 32, 5, 17]))
    A, sA = quant.quant_1x128(X.reshape(-1, 256))
    A, sA = A.reshape(4, 32, 256), sA.reshape(4, 32, 2)
    B, sB = quant.quant_128x128_grouped(W)
    D = gemm.gemm_masked(A, sA, B, sB, mm)
    assert np.all(np.isnan(D[0]))
    for e in range(1, 4):
        m = mm[e]
        assert np.array_equal(D[e, :m], gemm.gemm_dense(A[e, :m], sA[e, :m], B[e], sB[e]))
        assert np.all(np.isnan(D[e, m:]))


def test_bf16_matches_library_on_f32_values():
    g = np.random.default_rng(20)
    x = (g.standard_normal(50000) * np.exp(g.uniform(-80, 80, 50000))).astype(np.float32)
    ties = (np.arange(1, 2000, dtype=np.float32) * np.float32(2.0 ** -8) + np.float32(2.0 ** -9)
            + np.float32(1.0))
    x = np.concatenate([x, ties, -ties, np.float32([3e38, -3.4e38, 1e-40, 0.0])])
    lib = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(gemm.bf16_rne(x.astype(np.float64)), lib)
