"""fp8gemm_dense_batch: independent dense problems in one launch of the
tensor-core GEMM, against the FP64 oracle per problem (ragged sizes, empty
entries, mixed formats, several rounds of tiles); bit-identical to the
single-problem whole-tile path; the tile counters across launches issued back
to back and across replays of a captured CUDA graph; the full prefill pair."""

import numpy as np
import pytest

from fp8_fine_grained_e4m3_gb300 import synthetic
from tests.gpu_helpers import (assert_close, dev, host, ogemm, oquant, quant_weights,
                               quantised_dense, sample_rows_cols)

pytestmark = pytest.mark.gpu


def _b():
    from fp8_fine_grained_e4m3_gb300 import binding
    return binding


def _operands(M, N, K, seed, kind="normal", a_fmt="e4m3", b_fmt="e4m3"):
    """Oracle-quantised (A, sA, B, sB); empty when M or N is 0."""
    Kb = -(-K // 128)
    if M == 0 or N == 0:
        A = np.zeros((M, K), np.uint8)
        sA = np.zeros((M, Kb), np.float32)
        B = np.zeros((N, K), np.uint8)
        sB = np.zeros((-(-N // 128), Kb), np.float32)
        return A, sA, B, sB
    if a_fmt == "e4m3" and b_fmt == "e4m3":
        return quantised_dense(M, N, K, kind, seed=seed)
    X, W = synthetic.dense_operands(M, N, K, kind=kind, seed=seed)
    A, sA = oquant.quant_1x128(X, fmt=a_fmt) if a_fmt != "e4m3" else oquant.quant_1x128_fast(X)
    B, sB = oquant.quant_128x128(W, fmt=b_fmt) if b_fmt != "e4m3" else quant_weights(W)
    return A, sA, B, sB


def _check(probs, outs, what, fmts=None, sample=False):
    for i, ((A, sA, B, sB), D) in enumerate(zip(probs, outs)):
        M, N = A.shape[0], B.shape[0]
        assert tuple(D.shape) == (M, N)
        if M == 0 or N == 0:
            continue
        a_fmt, b_fmt = fmts[i] if fmts else ("e4m3", "e4m3")
        got = host(D)
        if sample:
            rows, cols = sample_rows_cols(M, N, 40, 80, seed=i)
            ref = ogemm.gemm_dense_at(A, sA, B, sB, rows, cols, a_fmt=a_fmt, b_fmt=b_fmt)
            assert_close(got[rows][:, cols], ref, f"{what}: problem {i} {M}x{N}")
        else:
            ref = ogemm.gemm_dense(A, sA, B, sB, a_fmt=a_fmt, b_fmt=b_fmt)
            assert_close(got, ref, f"{what}: problem {i} {M}x{N}")


@pytest.mark.parametrize("shapes", [
    [(300, 520, 1024), (200, 256, 512)],                     # two; reordered by K on the host
    [(200, 256, 512), (300, 520, 1024)],                     # same pair, already in K order
    [(129, 300, 272), (640, 768, 2048), (65, 256, 144), (1, 17, 160)],  # ragged M/N/K, one row, N odd
    [(0, 256, 256), (257, 2304, 640), (128, 0, 128)],        # empty entries are skipped
    [(2100, 2060, 384), (517, 7936, 1024)],                  # several rounds; N % 8 != 0; 5-row M block
    [(130, 256, 400)],                                       # one problem
    [(1300, 4000, 640), (1300, 1800, 272), (96, 520, 1024), (777, 2176, 512)],  # four, all kinds
])
def test_batch_matches_oracle(shapes):
    b = _b()
    probs = [_operands(M, N, K, seed=11 * i + M + N) for i, (M, N, K) in enumerate(shapes)]
    outs = b.fp8gemm_dense_batch([tuple(dev(x) for x in p) for p in probs])
    _check(probs, outs, f"batch {shapes}")
    assert b.fp8gemm_get_device_status() == b.OK


def test_batch_mixed_formats():
    """Each entry carries its own operand formats."""
    b = _b()
    spec = [((300, 512, 640), ("e5m2", "e4m3")), ((256, 520, 384), ("e4m3", "e5m2")),
            ((140, 256, 1024), ("e5m2", "e5m2")), ((129, 768, 256), ("e4m3", "e4m3"))]
    probs = [_operands(M, N, K, seed=70 + i, kind="prefill", a_fmt=f[0], b_fmt=f[1])
             for i, ((M, N, K), f) in enumerate(spec)]
    entries = [tuple(dev(x) for x in p) + f for p, (_, f) in zip(probs, spec)]
    outs = b.fp8gemm_dense_batch(entries)
    _check(probs, outs, "mixed formats", fmts=[f for _, f in spec])
    assert b.fp8gemm_get_device_status() == b.OK


def test_batch_bit_identical_to_single_calls():
    """Problems with at least a wave of 256-column tiles take the whole-tile
    path alone too: the batched launch gives the same bits; a third problem
    (fewer tiles than SMs, split along K when alone) is checked against the
    oracle on a sample."""
    b = _b()
    shapes = [(2048, 4096, 512), (2560, 4096, 256), (1280, 2560, 1024)]
    probs = [_operands(M, N, K, seed=90 + i, kind="prefill") for i, (M, N, K) in enumerate(shapes)]
    tens = [tuple(dev(x) for x in p) for p in probs]
    outs = b.fp8gemm_dense_batch(tens)
    for t, D in list(zip(tens, outs))[:2]:
        assert np.array_equal(host(b.fp8gemm_dense(*t)), host(D))
    _check(probs, outs, "batch vs single calls", sample=True)
    assert b.fp8gemm_get_device_status() == b.OK


def test_batch_counters_back_to_back_and_graph_replay():
    """Four launches back to back with no host synchronisation, each into
    buffers filled with NaN: every launch must take every tile (a counter
    left past zero by the launch before would leave tiles unwritten).  Then
    the call captured in a CUDA graph on another stream and replayed three
    times, each into NaN-filled buffers."""
    import torch
    b = _b()
    shapes = [(1300, 4000, 640), (520, 2304, 384), (300, 520, 1024)]
    probs = [_operands(M, N, K, seed=120 + i, kind="prefill") for i, (M, N, K) in enumerate(shapes)]
    tens = [tuple(dev(x) for x in p) for p in probs]
    ref = [host(D) for D in b.fp8gemm_dense_batch(tens)]
    _check(probs, [dev(r, torch.bfloat16) for r in ref], "first launch", sample=True)

    def nan_outs():
        return [torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
                for (M, N, _) in shapes]

    runs = []
    for _ in range(4):
        Ds = nan_outs()
        b.fp8gemm_dense_batch([t + (D,) for t, D in zip(tens, Ds)])
        runs.append(Ds)
    torch.cuda.synchronize()
    for k, Ds in enumerate(runs):
        for D, r in zip(Ds, ref):
            assert np.array_equal(host(D), r), f"launch {k} of a back-to-back run"

    Ds = nan_outs()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        b.fp8gemm_dense_batch([t + (D,) for t, D in zip(tens, Ds)])  # the stream's workspace
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        b.fp8gemm_dense_batch([t + (D,) for t, D in zip(tens, Ds)])
    for rep in range(3):
        for D in Ds:
            D.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        for D, r in zip(Ds, ref):
            assert np.array_equal(host(D), r), f"graph replay {rep}"
    assert b.fp8gemm_get_device_status() == b.OK


def test_batch_after_quantiser_without_host_sync():
    """The batched launch is a programmatic dependent of the kernel before
    it: quantise both problems' activations and launch the batch right
    after, twice, with no host synchronisation."""
    b = _b()
    shapes = [(1280, 4096, 2048), (2560, 2048, 1024)]
    Ws = [synthetic.dense_operands(M, N, K, kind="prefill", seed=140 + i)[1]
          for i, (M, N, K) in enumerate(shapes)]
    Bq = [quant_weights(W) for W in Ws]
    Bd = [(dev(B), dev(sB)) for B, sB in Bq]
    runs = []
    for seed in (150, 151):
        Xs = [synthetic.dense_operands(M, 8, K, kind="prefill", seed=seed + i)[0]
              for i, (M, N, K) in enumerate(shapes)]
        qa = [b.fp8_quant_1x128(dev(X)) for X in Xs]
        outs = b.fp8gemm_dense_batch([(A8, sA, B8, sB) for (A8, sA), (B8, sB) in zip(qa, Bd)])
        runs.append((Xs, outs))
    for Xs, outs in runs:
        probs = [oquant.quant_1x128_fast(X) + Bq[i] for i, X in enumerate(Xs)]
        _check(probs, outs, "batch after its quantisers", sample=True)
    assert b.fp8gemm_get_device_status() == b.OK


@pytest.mark.slow
def test_batch_prefill_pair_full_size():
    """The two prefill shapes in one launch, as the benchmark runs them:
    bit-identical to the single calls (both take the whole-tile path), and a
    sample against the oracle."""
    b = _b()
    shapes = [(4096, 4096, 4096), (4096, 7168, 16384)]
    probs = [_operands(M, N, K, seed=i, kind="prefill") for i, (M, N, K) in enumerate(shapes)]
    tens = [tuple(dev(x) for x in p) for p in probs]
    outs = b.fp8gemm_dense_batch(tens)
    for t, D in zip(tens, outs):
        assert np.array_equal(host(b.fp8gemm_dense(*t)), host(D))
    _check(probs, outs, "prefill pair", sample=True)
    assert b.fp8gemm_get_device_status() == b.OK


def test_batch_moe_experts_match_the_contiguous_form():
    """A MoE layer whose token counts the host knows, each expert's unpadded
    rows as one entry (24 experts, one of them empty: the 32-slot instance):
    on the real rows bit-identical to fp8gemm_grouped_contiguous over the
    padded layout (same tile arithmetic), and a sample of every expert
    against the oracle."""
    b = _b()
    E, T, N, K = 24, 2048, 4096, 1024
    counts = synthetic.zipf_counts(E, T, seed=7)
    counts[5] = 0
    X, W, lay = synthetic.contiguous_operands(E, T, N, K, seed=7, counts=counts)
    A, sA = oquant.quant_1x128_fast(X)
    Bq = [quant_weights(W[e]) for e in range(E)]
    B = np.stack([q for q, _ in Bq])
    sB = np.stack([s for _, s in Bq])
    tA, tsA, tB, tsB = dev(A), dev(sA), dev(B), dev(sB)
    Dc = host(b.fp8gemm_grouped_contiguous(tA, tsA, tB, tsB, dev(lay.m_indices)))
    live = [e for e in range(E) if counts[e] > 0]
    ents = []
    for e in live:
        o, c = int(lay.offsets[e]), int(counts[e])
        ents.append((tA[o:o + c], tsA[o:o + c], tB[e], tsB[e]))
    outs = b.fp8gemm_dense_batch(ents)
    for e, D in zip(live, outs):
        o, c = int(lay.offsets[e]), int(counts[e])
        got = host(D)
        assert np.array_equal(got, Dc[o:o + c]), f"expert {e}"
        rows, cols = sample_rows_cols(c, N, 6, 40, seed=e)
        ref = ogemm.gemm_dense_at(A[o:o + c], sA[o:o + c], B[e], sB[e], rows, cols)
        assert_close(got[rows][:, cols], ref, f"expert {e} ({c} rows)")
    assert b.fp8gemm_get_device_status() == b.OK


def test_batch_many_problems_mixed_k_and_formats():
    """Nine problems (the 32-slot instance) of three depths of K, ragged sizes
    and mixed formats: ordered by K, then largest and smallest alternating;
    each against the oracle."""
    b = _b()
    spec = [((300, 512, 1024), ("e4m3", "e4m3")), ((129, 256, 256), ("e5m2", "e4m3")),
            ((640, 768, 512), ("e4m3", "e4m3")), ((64, 520, 1024), ("e4m3", "e5m2")),
            ((1100, 1024, 256), ("e4m3", "e4m3")), ((200, 300, 512), ("e5m2", "e5m2")),
            ((17, 2304, 1024), ("e4m3", "e4m3")), ((400, 256, 256), ("e4m3", "e4m3")),
            ((257, 1000, 512), ("e4m3", "e4m3"))]
    probs = [_operands(M, N, K, seed=200 + i, kind="prefill", a_fmt=f[0], b_fmt=f[1])
             for i, ((M, N, K), f) in enumerate(spec)]
    entries = [tuple(dev(x) for x in p) + f for p, (_, f) in zip(probs, spec)]
    outs = b.fp8gemm_dense_batch(entries)
    _check(probs, outs, "nine problems", fmts=[f for _, f in spec])
    assert b.fp8gemm_get_device_status() == b.OK


def test_batch_full_32_problems():
    """Exactly FP8GEMM_MAX_DENSE_BATCH problems (every parameter slot of the
    32-slot instance in use): random sizes, two depths of K, against the
    oracle; one more entry is refused on the host."""
    b = _b()
    g = np.random.default_rng(33)
    shapes = [(int(g.integers(1, 300)), int(g.choice([256, 512, 520])), int(g.choice([128, 256])))
              for _ in range(b.MAX_DENSE_BATCH)]
    probs = [_operands(M, N, K, seed=300 + i) for i, (M, N, K) in enumerate(shapes)]
    tens = [tuple(dev(x) for x in p) for p in probs]
    outs = b.fp8gemm_dense_batch(tens)
    _check(probs, outs, "32 problems")
    with pytest.raises(ValueError, match="at most"):
        b.fp8gemm_dense_batch(tens + tens[:1])
    assert b.fp8gemm_get_device_status() == b.OK
