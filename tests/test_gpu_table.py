"""fp8gemm_grouped_table: many problems from a device-resident table, against
the oracle -- decode-sized ones, entries of a few hundred rows (taken 64 rows
at a time), e5m2 and mixed-format entries; a captured CUDA graph replayed
after the table was rewritten with other shapes and pointers; entries that
are empty or break the contract."""

import numpy as np
import pytest

from fp8_fine_grained_e4m3_gb300 import synthetic
from tests.gpu_helpers import assert_close, dev, host, ogemm, oquant, quant_weights

pytestmark = pytest.mark.gpu


def _b():
    from fp8_fine_grained_e4m3_gb300 import binding
    return binding


def _problem(M, N, K, seed, a_fmt="e4m3", b_fmt="e4m3"):
    import torch
    X, W = synthetic.dense_operands(M, N, K, kind="decode", seed=seed)
    A, sA = oquant.quant_1x128(X, fmt=a_fmt) if a_fmt != "e4m3" else oquant.quant_1x128_fast(X)
    B, sB = oquant.quant_128x128(W, fmt=b_fmt) if b_fmt != "e4m3" else quant_weights(W)
    ref = ogemm.gemm_dense(A, sA, B, sB, a_fmt=a_fmt, b_fmt=b_fmt)
    D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    return (dev(A), dev(sA), dev(B), dev(sB), D, a_fmt, b_fmt), ref


SHAPES = [(1, 2048, 7168), (5, 300, 400), (16, 7168, 2048), (33, 777, 1024), (64, 128, 256),
          (7, 1000, 272), (64, 2048, 2048), (2, 129, 4096)]


@pytest.mark.parametrize("max_M,shapes", [
    (64, SHAPES),                                            # 64-wide kernel, mixed shapes
    (16, [(1, 2048, 7168), (5, 300, 400), (16, 640, 1024)]),  # 16-wide kernel
    (32, [(20, 1536, 7168), (32, 256, 144)]),                 # 32-wide kernel, partial K block
])
def test_table_matches_oracle(max_M, shapes):
    b = _b()
    probs, refs = zip(*[_problem(M, N, K, seed=i + M) for i, (M, N, K) in enumerate(shapes)])
    table = b.problem_table(probs)
    b.fp8gemm_grouped_table(table, len(probs), max_M)
    for prob, ref, shp in zip(probs, refs, shapes):
        assert_close(host(prob[4]), ref, f"table problem {shp}")
    assert b.fp8gemm_get_device_status() == b.OK


@pytest.mark.parametrize("max_M,shapes", [
    # entries above 64 rows: taken 64 rows at a time (last chunk partial)
    (300, [(300, 1024, 512), (65, 640, 2048), (1, 7168, 2048), (200, 384, 1040), (128, 256, 256)]),
    (129, [(129, 2048, 1024), (64, 300, 400), (100, 129, 4096)]),
])
def test_table_entries_above_64_rows(max_M, shapes):
    b = _b()
    probs, refs = zip(*[_problem(M, N, K, seed=60 + i) for i, (M, N, K) in enumerate(shapes)])
    b.fp8gemm_grouped_table(b.problem_table(probs), len(probs), max_M)
    for prob, ref, shp in zip(probs, refs, shapes):
        assert_close(host(prob[4]), ref, f"table problem {shp}")
    assert b.fp8gemm_get_device_status() == b.OK


def test_table_with_e5m2_and_mixed_entries():
    b = _b()
    spec = [((16, 640, 1024), "e5m2", "e4m3"), ((5, 300, 400), "e4m3", "e5m2"),
            ((33, 777, 2048), "e5m2", "e5m2"), ((90, 512, 272), "e5m2", "e4m3"),
            ((8, 2048, 1024), "e4m3", "e4m3")]
    probs, refs = zip(*[_problem(M, N, K, seed=80 + i, a_fmt=af, b_fmt=bf)
                        for i, ((M, N, K), af, bf) in enumerate(spec)])
    b.fp8gemm_grouped_table(b.problem_table(probs), len(probs), 90)
    for prob, ref, (shp, af, bf) in zip(probs, refs, spec):
        assert_close(host(prob[4]), ref, f"table problem {shp} {af} x {bf}")
    assert b.fp8gemm_get_device_status() == b.OK


def test_graph_replay_with_rewritten_table():
    """The launch is captured once; between replays the table is rewritten
    in place with problems of other sizes and buffers."""
    import torch
    b = _b()
    first = [_problem(M, N, K, seed=40 + i) for i, (M, N, K) in enumerate([(4, 640, 2048), (9, 2048, 512)])]
    second = [_problem(M, N, K, seed=50 + i) for i, (M, N, K) in
              enumerate([(16, 384, 1024), (1, 7168, 256), (12, 200, 400)])]
    P = 3
    table = torch.zeros(P * 56, dtype=torch.uint8, device="cuda")
    # the first set padded with an empty entry (M = 0) to the captured count
    empty = (first[0][0][0][:0], first[0][0][1][:0], first[0][0][2], first[0][0][3],
             first[0][0][4][:0])  # M = 0
    b.problem_table([p for p, _ in first] + [empty], out=table)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        b.fp8gemm_grouped_table(table, P, 16)  # warm-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        b.fp8gemm_grouped_table(table, P, 16)
    for (probs, _) in first:
        probs[4].fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    for (probs, ref) in first:
        assert_close(host(probs[4]), ref, "replay 1")
    b.problem_table([p for p, _ in second], out=table)
    g.replay()
    torch.cuda.synchronize()
    for (probs, ref) in second:
        assert_close(host(probs[4]), ref, "replay 2 (rewritten table)")
    assert b.fp8gemm_get_device_status() == b.OK


def test_bad_and_empty_entries():
    import torch
    b = _b()
    good, ref = _problem(8, 512, 1024, seed=7)
    other, ref2 = _problem(3, 256, 256, seed=8)
    import ctypes
    arr = (b.Problem * 5)()
    for e, (A, sA, B, sB, D, _, _) in zip(arr, [good, other, good, good, good]):
        e.A, e.sA, e.B, e.sB, e.D = (A.data_ptr(), sA.data_ptr(), B.data_ptr(), sB.data_ptr(),
                                     D.data_ptr())
        e.M, e.K = A.shape
        e.N = B.shape[0]
    arr[2].M = 65            # beyond max_M: skipped, status raised
    arr[3].A = arr[3].A + 4  # misaligned A: skipped, status raised
    arr[4].formats = 2       # unknown operand format: skipped, status raised
    bad_D = torch.full((8, 512), 7.0, dtype=torch.bfloat16, device="cuda")
    arr[2].D = arr[3].D = arr[4].D = bad_D.data_ptr()
    table = torch.frombuffer(bytearray(bytes(arr)), dtype=torch.uint8).cuda()
    b.fp8gemm_grouped_table(table, 5, 64)
    assert b.fp8gemm_get_device_status() == b.ERR_DEVICE_STATUS
    assert_close(host(good[4]), ref, "good entry beside bad ones")
    assert_close(host(other[4]), ref2, "second good entry")
    assert bool((bad_D == 7.0).all())  # skipped entries write nothing
    assert b.fp8gemm_get_device_status() == b.OK  # the read cleared it


def test_table_few_items_split_along_k():
    """Fewer (entry, tile) items than CTAs: the kernel splits their K ranges
    over the CTAs (stream-K) and sums the partials in a fixed order, so the
    result matches the oracle and repeats bit for bit."""
    b = _b()
    shapes = [(3, 256, 7168), (16, 128, 16384), (1, 384, 2048), (40, 128, 1040)]
    probs, refs = zip(*[_problem(M, N, K, seed=90 + i) for i, (M, N, K) in enumerate(shapes)])
    table = b.problem_table(probs)
    b.fp8gemm_grouped_table(table, len(probs), 64)
    first = [host(p[4]).copy() for p in probs]
    for got, ref, shp in zip(first, refs, shapes):
        assert_close(got, ref, f"split table problem {shp}")
    for p in probs:
        p[4].fill_(float("nan"))
    b.fp8gemm_grouped_table(table, len(probs), 64)
    for p, f in zip(probs, first):
        assert np.array_equal(host(p[4]), f)
    assert b.fp8gemm_get_device_status() == b.OK


def test_table_a_little_over_one_round_of_items():
    """310 (entry, tile) items for the 16-wide kernel: a little more than one
    round of whole items, so the units are split over the CTAs (stream-K) and
    many items are summed from several partials -- entries of 1 to 16 rows,
    K of 2 and 3 blocks, partial last K blocks, ragged N.  The result matches
    the oracle and repeats bit for bit."""
    b = _b()
    rng = np.random.default_rng(5)
    shapes = []
    for i in range(40):
        M = int(rng.integers(1, 17))
        N = [1024, 1000, 1024, 896][i % 4]
        K = [512, 272, 400, 1024, 256][i % 5]
        shapes.append((M, N, K))
    probs, refs = zip(*[_problem(M, N, K, seed=200 + i) for i, (M, N, K) in enumerate(shapes)])
    table = b.problem_table(probs)
    b.fp8gemm_grouped_table(table, len(probs), 16)
    first = [host(p[4]).copy() for p in probs]
    for got, ref, shp in zip(first, refs, shapes):
        assert_close(got, ref, f"table problem {shp}")
    for p in probs:
        p[4].fill_(float("nan"))
    b.fp8gemm_grouped_table(table, len(probs), 16)
    for p, f in zip(probs, first):
        assert np.array_equal(host(p[4]), f)
    assert b.fp8gemm_get_device_status() == b.OK
