"""Block-scaled FP8 GEMM, written out as its definition, in FP64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Definition ("lpnh.cn/news/2822121" section 2.3): with per-block scales
sA[m, kBlock] and sB[n, kBlock], the output is the sum over K blocks of each
block's own product multiplied by that block's sA x sB -- the scale product
changes with the K block, so it cannot be applied once at the end:

    D[m, n] = sum_kb  sA[m, kb] * sB[n // 128, kb]
                      * sum_{k in block kb} dec(A[m, k]) * dec(B[n, k])

B's scale is per 128x128 tile, so its row index is n // 128 ("blog.hotdry.top:
DeepGEMM FP8 GEMM fine-grained scaling kernels", section "fine-grained scaling
core design").  A is [M, K] and B is [N, K], both K-contiguous (D = A B^T), as
in the call sketch of "bhfrc.com/news/60211" section 6.  The accumulation is in
a wide format (FP32 on the GPU, "news.rkmt.cn/news/5092" section 2.3; FP64
here), and the result is rounded to the output type only when written
(BF16 here).

Grouped forms ("news.rkmt.cn/news/5092" section 5.3: experts' tokens are
contiguous, with group ids per row; "bhfrc.com/news/60211" sections 4.2-4.3:
shape data lives in device memory):

* contiguous: A rows are grouped by expert, each expert segment padded to a
  multiple of 128 rows; m_indices[r] is the expert of row r, -1 for padding.
  Row r uses B[m_indices[r]].  Padding rows are "don't care" (NaN here).
* masked: A is [E, M_max, K]; only the first masked_m[e] rows of expert e are
  computed; the other rows are not written (NaN here).

Steps: decode bytes through the format's table; for each K block form the
block product with a float64 matmul (library primitive); multiply by the
float64 scale product; accumulate in float64.

Operand formats: A and B are e4m3 by default; either may be e5m2
(``a_fmt`` / ``b_fmt``), e.g. an e5m2 gradient against e4m3 weights
("news.rkmt.cn/news/5092" section 2.1; "lpnh.cn/news/2822121" section 2.1:
mixing the two formats is allowed and costs precision).  Only the decoding of
the bytes changes.
"""

import numpy as np

from . import e4m3, e5m2


def _decoder(fmt):
    return {"e4m3": e4m3.decode, "e5m2": e5m2.decode}[fmt]

BLOCK = 128


def _block_scaled(Ad, sA, Bd, sB_rows) -> np.ndarray:
    """The definition with B's scale given per row: Ad f64 [M, K] and Bd f64
    [N, K] decoded operands, sA [M, Kb], sB_rows [N, Kb] (row n holds the
    scales of its 128x128 tile)."""
    M, K = Ad.shape
    N = Bd.shape[0]
    Kb = sA.shape[1]
    D = np.zeros((M, N), dtype=np.float64)
    for kb in range(Kb):
        ks = slice(kb * BLOCK, min(K, (kb + 1) * BLOCK))
        P = Ad[:, ks] @ Bd[:, ks].T  # this K block's product, FP64
        D += (sA[:, kb][:, None] * sB_rows[:, kb][None, :]) * P
    return D


def gemm_dense(A, sA, B, sB, a_fmt="e4m3", b_fmt="e4m3") -> np.ndarray:
    """A u8 [M, K], sA f32 [M, Kb], B u8 [N, K], sB f32 [Nb, Kb] -> f64 [M, N]."""
    A = np.asarray(A, dtype=np.uint8)
    B = np.asarray(B, dtype=np.uint8)
    M, K = A.shape
    N, K2 = B.shape
    assert K == K2
    Kb = -(-K // BLOCK)
    sA = np.asarray(sA, dtype=np.float32).astype(np.float64)
    sB = np.asarray(sB, dtype=np.float32).astype(np.float64)
    assert sA.shape == (M, Kb) and sB.shape == (-(-N // BLOCK), Kb)
    sB_rows = sB[np.arange(N) // BLOCK]  # scale row of B row n is n // 128
    return _block_scaled(_decoder(a_fmt)(A), sA, _decoder(b_fmt)(B), sB_rows)


def gemm_dense_at(A, sA, B, sB, rows, cols, a_fmt="e4m3", b_fmt="e4m3") -> np.ndarray:
    """D[rows][:, cols] of :func:`gemm_dense`, without forming the rest:
    D[m, n] depends only on A[m], sA[m], B[n] and sB[n // 128]."""
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.asarray(cols, dtype=np.int64)
    sA = np.asarray(sA, dtype=np.float32).astype(np.float64)[rows]
    sB = np.asarray(sB, dtype=np.float32).astype(np.float64)
    return _block_scaled(_decoder(a_fmt)(np.asarray(A)[rows]), sA,
                         _decoder(b_fmt)(np.asarray(B)[cols]), sB[cols // BLOCK])


def gemm_contiguous(A, sA, B, sB, m_indices, a_fmt="e4m3", b_fmt="e4m3") -> np.ndarray:
    """A u8 [M_pad, K], sA [M_pad, Kb], B u8 [E, N, K], sB [E, Nb, Kb],
    m_indices i32 [M_pad] -> f64 [M_pad, N]; padding rows (index -1) are NaN."""
    A = np.asarray(A, dtype=np.uint8)
    m_indices = np.asarray(m_indices, dtype=np.int64)
    E, N, K = B.shape
    D = np.full((A.shape[0], N), np.nan, dtype=np.float64)
    for e in range(E):
        r = np.nonzero(m_indices == e)[0]
        if r.size:
            D[r] = gemm_dense(A[r], np.asarray(sA)[r], B[e], sB[e], a_fmt, b_fmt)
    return D


def gemm_masked(A, sA, B, sB, masked_m, a_fmt="e4m3", b_fmt="e4m3") -> np.ndarray:
    """A u8 [E, M_max, K], sA [E, M_max, Kb], B u8 [E, N, K], sB [E, Nb, Kb],
    masked_m i32 [E] -> f64 [E, M_max, N]; rows >= masked_m[e] are NaN."""
    E, M_max, K = A.shape
    N = B.shape[1]
    D = np.full((E, M_max, N), np.nan, dtype=np.float64)
    for e in range(E):
        m = int(masked_m[e])
        if m > 0:
            D[e, :m] = gemm_dense(A[e, :m], sA[e, :m], B[e], sB[e], a_fmt, b_fmt)
    return D


def bf16_rne(x: np.ndarray) -> np.ndarray:
    """Round float64 values to bfloat16 (8 significant bits; nearest, ties to
    even; +-inf past the largest finite bf16).  Returned as float64 holding the
    bf16 value.  Rounding happens once, directly from float64."""
    x = np.asarray(x, dtype=np.float64)
    fin = np.isfinite(x) & (x != 0)
    xs = np.where(fin, x, 1.0)
    _, e = np.frexp(xs)  # |x| = m * 2^e with 0.5 <= m < 1
    qexp = np.where(e - 1 < -126, -133, e - 8)  # quantum: 2^-133 below the normals
    q = np.ldexp(1.0, qexp)
    y = np.round(xs / q) * q  # x / q is exact; np.round ties to even
    y = np.where(np.abs(y) > 3.3895313892515355e38, np.copysign(np.inf, xs), y)
    return np.where(fin, y, x)
