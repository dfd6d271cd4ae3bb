"""Shared pieces of the GPU parity tests: device copies, oracle-prepared
inputs and the acceptance check.

Acceptance for the GEMM (the tolerance fixed for this path): per element
|gpu - ref| <= 1e-2 |ref| + 1e-3 rms(ref), with ref the FP64 oracle and rms
over the compared elements.  The quantisers must match bit for bit.
"""

import numpy as np

from oracle import gemm as ogemm
from oracle import quant as oquant

RTOL = 1e-2
RMS_TOL = 1e-3


def dev(a, dtype=None):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def host(t):
    import torch
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy().astype(np.float64)
    return t.cpu().numpy()


def assert_close(got, ref, what=""):
    """The per-element acceptance test; ignores NaN (don't-care) reference
    entries.  Returns (max abs err / (rms), max rel err) for reporting."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    mask = ~np.isnan(ref)
    g, r = got[mask], ref[mask]
    if r.size == 0:
        return 0.0, 0.0
    rms = float(np.sqrt(np.mean(r * r)))
    bound = RTOL * np.abs(r) + RMS_TOL * rms
    err = np.abs(g - r)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argsort(-(err - bound) * bad)[:8]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {r.size} elements out of tolerance; worst "
            f"got={g[idx]} ref={r[idx]} rms={rms}")
    return float(err.max() / (rms + 1e-300)), float(np.max(err / (np.abs(r) + 1e-300)))


def quantised_dense(M, N, K, kind, seed):
    """Oracle-quantised (A, sA, B, sB) for a dense workload."""
    from fp8_fine_grained_e4m3_gb300 import synthetic
    X, W = synthetic.dense_operands(M, N, K, kind=kind, seed=seed)
    A, sA = oquant.quant_1x128_fast(X)
    B, sB = quant_weights(W) if N >= 1 else (np.zeros((0, K), np.uint8), None)
    return A, sA, B, sB


def quant_weights(W):
    """The oracle's 128x128 quantiser: the vectorised form for whole K blocks,
    the tile loop for a partial last K block."""
    if W.shape[-1] % 128 == 0:
        return oquant.quant_128x128_fast(W)
    return oquant.quant_128x128(W)


def rotated_experts(B, sB, E):
    """E distinct quantised weight matrices from one: expert e is B with its
    128-row tiles rotated by e tiles (a permutation of whole scale tiles, so
    each is itself a valid 128x128-quantised matrix)."""
    Nb = sB.shape[0]
    Bs = np.stack([np.roll(B, -128 * (e % Nb), axis=0) for e in range(E)])
    sBs = np.stack([np.roll(sB, -(e % Nb), axis=0) for e in range(E)])
    return Bs, sBs


def sample_rows_cols(M, N, n_rows, n_cols, seed):
    g = np.random.default_rng(seed)
    rows = np.unique(np.concatenate([[0, M - 1], g.integers(0, M, n_rows)]))
    cols = np.unique(np.concatenate([[0, N - 1], g.integers(0, N, n_cols)]))
    return rows, cols


__all__ = ["dev", "host", "assert_close", "quantised_dense", "rotated_experts",
           "sample_rows_cols", "ogemm", "oquant"]
