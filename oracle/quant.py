"""Fine-grained FP8 quantisers (FP32 semantics), written out step by step.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Granularity ("blog.hotdry.top: DeepGEMM FP8 GEMM fine-grained scaling
kernels", section "fine-grained scaling core design"): the left operand A
(activations) gets one scale per 1x128 tile -- one row, 128 consecutive K
elements -- and the right operand B (weights) one scale per 128x128 tile.
Scales are FP32 tensors kept beside the FP8 bytes.

Scale rule ("news.rkmt.cn/news/5092" section 5.2): take the largest absolute
value of the block and divide it by the e4m3 limit 448; every block gets its
own scale.  The stored scale is the DEquantisation factor s = amax / 448, so a
byte q stands for dec(q) * s and q is the e4m3 rounding of x / s.  (The same
paragraph also words it as "limit divided by the max"; the formula it prints,
max_val / 448, is the one taken.)

Rounding ("lpnh.cn/news/2822121" section 6.3, second point): round to
nearest (ties to even), never toward zero.

Arithmetic, in this order, all in IEEE FP32 with round-to-nearest:

1. amax = max |x| over the block (exact);
2. s = amax / 448;
3. q = e4m3_rne_sat(x / s) for every x of the block.

A block whose amax is 0 stores s = 0 and all-zero bytes (0x00), so that no
0/0 is formed.  K (and N for the weight quantiser) may end in a ragged block:
its amax runs over the elements that exist.

Every function takes ``fmt`` = "e4m3" (the default, limit 448) or "e5m2"
(limit 57344, the largest finite e5m2 value): the same rule with that
format's limit and encoder (gradients and other wide-range tensors,
"news.rkmt.cn/news/5092" section 2.1).
"""

import numpy as np

from . import e4m3, e5m2

BLOCK = 128

_FORMATS = {"e4m3": (e4m3.E4M3_MAX, e4m3.encode_rne_sat),
            "e5m2": (e5m2.E5M2_MAX, e5m2.encode_rne_sat)}


def _quant_block(x: np.ndarray, fmt: str = "e4m3"):
    """Quantise one block (any shape) of FP32 values -> (bytes, scale)."""
    limit, encode = _FORMATS[fmt]
    x = np.asarray(x, dtype=np.float32)
    amax = np.float32(np.max(np.abs(x))) if x.size else np.float32(0.0)
    s = np.float32(amax / np.float32(limit))
    if amax == 0:
        return np.zeros(x.shape, dtype=np.uint8), s
    y = (x / s).astype(np.float32)  # IEEE FP32 division, round to nearest
    return encode(y), s


def quant_1x128(X: np.ndarray, fmt: str = "e4m3"):
    """Activations: X f32 [M, K] -> (Q u8 [M, K], sX f32 [M, ceil(K/128)]).

    One scale per row and 128-wide K block.  Loops over (row, K block) so each
    step is the three-line rule above; :func:`quant_1x128_fast` is the same
    rule over whole columns of blocks at once.
    """
    X = np.ascontiguousarray(X, dtype=np.float32)
    M, K = X.shape
    Kb = -(-K // BLOCK)
    Q = np.zeros((M, K), dtype=np.uint8)
    S = np.zeros((M, Kb), dtype=np.float32)
    for m in range(M):
        for kb in range(Kb):
            sl = slice(kb * BLOCK, min(K, (kb + 1) * BLOCK))
            Q[m, sl], S[m, kb] = _quant_block(X[m, sl], fmt)
    return Q, S


def quant_1x128_fast(X: np.ndarray, fmt: str = "e4m3"):
    """Same result as :func:`quant_1x128`, one K block at a time over all rows
    (NumPy broadcasting instead of a row loop), for the large test sizes."""
    limit, encode = _FORMATS[fmt]
    X = np.ascontiguousarray(X, dtype=np.float32)
    M, K = X.shape
    Kb = -(-K // BLOCK)
    Q = np.zeros((M, K), dtype=np.uint8)
    S = np.zeros((M, Kb), dtype=np.float32)
    for kb in range(Kb):
        sl = slice(kb * BLOCK, min(K, (kb + 1) * BLOCK))
        blk = X[:, sl]
        amax = np.max(np.abs(blk), axis=1).astype(np.float32)
        s = (amax / np.float32(limit)).astype(np.float32)
        S[:, kb] = s
        nz = amax != 0
        safe = np.where(nz, s, np.float32(1.0)).astype(np.float32)
        y = (blk / safe[:, None]).astype(np.float32)
        q = encode(y)
        q[~nz, :] = 0
        Q[:, sl] = q
    return Q, S


def quant_128x128(W: np.ndarray, fmt: str = "e4m3"):
    """Weights: W f32 [N, K] -> (Q u8 [N, K], sW f32 [ceil(N/128), ceil(K/128)]).

    One scale per 128x128 tile (ragged tiles at the N and K ends allowed).
    """
    W = np.ascontiguousarray(W, dtype=np.float32)
    N, K = W.shape
    Nb, Kb = -(-N // BLOCK), -(-K // BLOCK)
    Q = np.zeros((N, K), dtype=np.uint8)
    S = np.zeros((Nb, Kb), dtype=np.float32)
    for nb in range(Nb):
        rs = slice(nb * BLOCK, min(N, (nb + 1) * BLOCK))
        for kb in range(Kb):
            cs = slice(kb * BLOCK, min(K, (kb + 1) * BLOCK))
            Q[rs, cs], S[nb, kb] = _quant_block(W[rs, cs], fmt)
    return Q, S


def quant_128x128_fast(W: np.ndarray, fmt: str = "e4m3"):
    """Same result as :func:`quant_128x128`, one 128-row band at a time with
    every K tile of the band handled together (for the large test sizes)."""
    limit, encode = _FORMATS[fmt]
    W = np.ascontiguousarray(W, dtype=np.float32)
    N, K = W.shape
    assert K % BLOCK == 0, "vectorised form wants whole K blocks"
    Nb, Kb = -(-N // BLOCK), K // BLOCK
    Q = np.zeros((N, K), dtype=np.uint8)
    S = np.zeros((Nb, Kb), dtype=np.float32)
    for nb in range(Nb):
        band = W[nb * BLOCK:min(N, (nb + 1) * BLOCK)]          # [rows, K]
        tiles = band.reshape(band.shape[0], Kb, BLOCK)          # [rows, Kb, 128]
        amax = np.abs(tiles).max(axis=(0, 2)).astype(np.float32)  # [Kb]
        s = (amax / np.float32(limit)).astype(np.float32)
        S[nb] = s
        nz = amax != 0
        safe = np.where(nz, s, np.float32(1.0)).astype(np.float32)
        q = encode((tiles / safe[None, :, None]).astype(np.float32))
        q[:, ~nz, :] = 0
        Q[nb * BLOCK:nb * BLOCK + band.shape[0]] = q.reshape(band.shape[0], K)
    return Q, S


def quant_128x128_grouped(W: np.ndarray):
    """Per-expert weights: W f32 [E, N, K] -> (Q [E, N, K], sW [E, Nb, Kb])."""
    W = np.asarray(W, dtype=np.float32)
    qs, ss = zip(*(quant_128x128(W[e]) for e in range(W.shape[0])))
    return np.stack(qs), np.stack(ss)


def _block_saturations(x: np.ndarray, fmt: str = "e4m3") -> int:
    """Saturations of one block: the steps of :func:`_quant_block` up to the
    quotient, then the number of elements whose FP32 quotient x / s is not
    within +-limit (a NaN quotient included) -- the values the saturating
    encoding clamps.  A block with amax = 0 forms no quotient and counts 0.

    Monitoring an FP8 overflow count: "blog.hotdry.top: DeepGEMM FP8 GEMM
    fine-grained scaling kernels", section on numerical-stability checks and
    monitoring."""
    limit, _ = _FORMATS[fmt]
    x = np.asarray(x, dtype=np.float32)
    amax = np.float32(np.max(np.abs(x))) if x.size else np.float32(0.0)
    if amax == 0:
        return 0
    s = np.float32(amax / np.float32(limit))
    with np.errstate(divide="ignore", invalid="ignore"):
        y = (x / s).astype(np.float32)  # IEEE FP32 division, round to nearest
    return int(np.count_nonzero(~(np.abs(y) <= np.float32(limit))))


def saturations_1x128(X: np.ndarray, fmt: str = "e4m3") -> int:
    """Total saturations of :func:`quant_1x128` on X f32 [M, K]: the sum of
    :func:`_block_saturations` over its (row, K block) blocks."""
    X = np.ascontiguousarray(X, dtype=np.float32)
    M, K = X.shape
    n = 0
    for m in range(M):
        for kb in range(-(-K // BLOCK)):
            n += _block_saturations(X[m, kb * BLOCK:min(K, (kb + 1) * BLOCK)], fmt)
    return n


def saturations_128x128(W: np.ndarray, fmt: str = "e4m3") -> int:
    """Total saturations of :func:`quant_128x128` on W f32 [N, K] (or a batch
    [E, N, K]): the sum over its 128x128 tiles."""
    W = np.asarray(W, dtype=np.float32)
    if W.ndim == 3:
        return sum(saturations_128x128(w, fmt) for w in W)
    N, K = W.shape
    n = 0
    for nb in range(-(-N // BLOCK)):
        for kb in range(-(-K // BLOCK)):
            n += _block_saturations(W[nb * BLOCK:min(N, (nb + 1) * BLOCK),
                                      kb * BLOCK:min(K, (kb + 1) * BLOCK)], fmt)
    return n


def dequant_1x128(Q: np.ndarray, S: np.ndarray, fmt: str = "e4m3") -> np.ndarray:
    """dec(q) * s per element (float64), for error-bound checks."""
    decode = e4m3.decode if fmt == "e4m3" else e5m2.decode
    M, K = Q.shape
    s_full = np.repeat(S.astype(np.float64), BLOCK, axis=1)[:, :K]
    return decode(Q) * s_full
