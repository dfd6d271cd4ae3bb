"""Seeded synthetic workloads for the FP8 block-scaled GEMM.

This module draws raw FP32 operands and the grouping structure (expert token
counts, row layout, valid-row counts).  It holds none of the method's
arithmetic -- no quantisation, no scaling, no GEMM -- so both the CUDA path
and the CPU oracle can take their inputs from it.

Workloads (sizes as the benchmark configurations state them):

* ``normal``   -- A, B ~ N(0, 1)                         (correctness case)
* ``prefill``  -- A ~ N(0, 1) with 1 % of the K columns scaled x50 as outlier
                  channels; B ~ N(0, 0.02)
* ``decode``   -- A ~ N(0, 1), B ~ N(0, 0.02)
* contiguous MoE -- expert token counts ~ Multinomial(T, p), p_e proportional
                  to (e + 1)^-1.1 (Zipf, s = 1.1); each expert's rows padded
                  to a multiple of 128; ``m_indices`` = expert per row, -1 on
                  padding rows (padding rows of A are zero)
* masked MoE   -- masked_m[e] ~ U{0, ..., M_max}; A ~ Student-t(nu = 3)

N(0, 0.02) is read as standard deviation 0.02 (the usual weight-init
convention).  Host arrays come from NumPy ``Generator(PCG64(seed))``; the
device variants (``*_device``) draw on the GPU with ``torch.Generator`` so
that full-size benchmark inputs never cross the host; their values differ
from the host variants but follow the same recipe.
"""

from dataclasses import dataclass
from typing import Optional

import numpy as np

BLOCK = 128


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def outlier_columns(K: int, seed: int) -> np.ndarray:
    """The seeded 1 % of K columns (round(0.01 K), at least 1) that carry x50."""
    n = max(1, int(round(0.01 * K)))
    return np.sort(rng(seed + 7919).permutation(K)[:n])


def dense_operands(M: int, N: int, K: int, kind: str = "normal", seed: int = 0):
    """Return (X f32 [M, K], W f32 [N, K]) for a dense workload."""
    g = rng(seed)
    if kind == "normal":
        X = g.standard_normal((M, K), dtype=np.float32)
        W = g.standard_normal((N, K), dtype=np.float32)
    elif kind in ("prefill", "decode"):
        X = g.standard_normal((M, K), dtype=np.float32)
        W = (g.standard_normal((N, K), dtype=np.float32) * np.float32(0.02)).astype(np.float32)
        if kind == "prefill":
            X[:, outlier_columns(K, seed)] *= np.float32(50.0)
    else:
        raise ValueError(f"unknown dense workload kind {kind!r}")
    return X, W


def zipf_counts(E: int, T: int, s: float = 1.1, seed: int = 0) -> np.ndarray:
    """Tokens per expert: Multinomial(T, p) with p_e proportional to (e+1)^-s."""
    p = (np.arange(1, E + 1, dtype=np.float64)) ** (-s)
    p /= p.sum()
    return rng(seed + 104729).multinomial(T, p).astype(np.int64)


@dataclass
class ContiguousLayout:
    counts: np.ndarray      # [E] real tokens per expert
    padded: np.ndarray      # [E] rows per expert after padding to 128
    offsets: np.ndarray     # [E] first row of each expert segment
    m_indices: np.ndarray   # [M_pad] int32, expert per row or -1
    M_pad: int


def contiguous_layout(counts: np.ndarray, align: int = BLOCK) -> ContiguousLayout:
    counts = np.asarray(counts, dtype=np.int64)
    padded = -(-counts // align) * align
    offsets = np.concatenate([[0], np.cumsum(padded)[:-1]]).astype(np.int64)
    M_pad = int(padded.sum())
    m_indices = np.full(M_pad, -1, dtype=np.int32)
    for e, (o, c) in enumerate(zip(offsets, counts)):
        m_indices[o:o + c] = e
    return ContiguousLayout(counts, padded, offsets, m_indices, M_pad)


def contiguous_operands(E: int, T: int, N: int, K: int, seed: int = 0,
                        counts: Optional[np.ndarray] = None):
    """Return (X f32 [M_pad, K], W f32 [E, N, K], layout)."""
    if counts is None:
        counts = zipf_counts(E, T, seed=seed)
    lay = contiguous_layout(counts)
    g = rng(seed)
    X = np.zeros((lay.M_pad, K), dtype=np.float32)
    real = lay.m_indices >= 0
    X[real] = g.standard_normal((int(real.sum()), K), dtype=np.float32)
    W = (g.standard_normal((E, N, K), dtype=np.float32) * np.float32(0.02)).astype(np.float32)
    return X, W, lay


def masked_counts(E: int, M_max: int, seed: int = 0) -> np.ndarray:
    """masked_m[e] ~ U{0, ..., M_max} (inclusive)."""
    return rng(seed + 15485863).integers(0, M_max + 1, size=E).astype(np.int32)


def masked_operands(E: int, M_max: int, N: int, K: int, seed: int = 0,
                    masked_m: Optional[np.ndarray] = None):
    """Return (X f32 [E, M_max, K] ~ Student-t(3), W f32 [E, N, K], masked_m)."""
    if masked_m is None:
        masked_m = masked_counts(E, M_max, seed)
    g = rng(seed)
    X = g.standard_t(3.0, size=(E, M_max, K)).astype(np.float32)
    W = (g.standard_normal((E, N, K), dtype=np.float32) * np.float32(0.02)).astype(np.float32)
    return X, W, np.asarray(masked_m, dtype=np.int32)


# ---------------------------------------------------------------- device side
def _tgen(seed: int, device):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def dense_operands_device(M, N, K, kind="normal", seed=0, device="cuda"):
    """Device-drawn (X, W) f32 torch tensors following :func:`dense_operands`."""
    import torch
    g = _tgen(seed, device)
    X = torch.randn((M, K), generator=g, device=device, dtype=torch.float32)
    W = torch.randn((N, K), generator=g, device=device, dtype=torch.float32)
    if kind in ("prefill", "decode"):
        W.mul_(0.02)
    if kind == "prefill":
        cols = torch.from_numpy(outlier_columns(K, seed)).to(device)
        X[:, cols] *= 50.0
    return X, W


def expert_weights_device(E, N, K, seed=0, device="cuda"):
    import torch
    g = _tgen(seed + 1, device)
    W = torch.randn((E, N, K), generator=g, device=device, dtype=torch.float32)
    return W.mul_(0.02)


def contiguous_activations_device(lay: ContiguousLayout, K, seed=0, device="cuda"):
    import torch
    g = _tgen(seed, device)
    X = torch.randn((lay.M_pad, K), generator=g, device=device, dtype=torch.float32)
    pad = torch.from_numpy(lay.m_indices < 0).to(device)
    X[pad] = 0.0
    return X


def masked_activations_device(E, M_max, K, seed=0, device="cuda"):
    """Student-t(3) draws on the device: Z / sqrt(V / 3), V ~ chi^2(3)."""
    import torch
    g = _tgen(seed, device)
    Z = torch.randn((E, M_max, K), generator=g, device=device, dtype=torch.float32)
    V = torch.randn((3, E, M_max, K), generator=g, device=device, dtype=torch.float32)
    V = V.square_().sum(0)
    return Z / torch.sqrt(V / 3.0)
