"""Library-owned workspaces: one per (device, stream) for the decode path's
split-K reduction and for fp8gemm_dense_quant_a's quantised activations.
Cycling streams grows what the library holds; fp8gemm_release_workspaces
gives each stream's buffers back, and a later call on a released stream
allocates again and is still correct."""

import pytest

from tests.gpu_helpers import assert_close, dev, host, ogemm, oquant, quantised_dense

pytestmark = pytest.mark.gpu


def test_workspaces_follow_streams_and_are_released():
    import torch

    from fp8_fine_grained_e4m3_gb300 import binding as b
    from fp8_fine_grained_e4m3_gb300 import synthetic
    # a decode shape that takes the stream-K form (workspace), and FP32
    # activations at M > 64 without Q/sA (library-held quantised A)
    M, N, K = 17, 128, 16384
    A, sA, B, sB = quantised_dense(M, N, K, "decode", seed=31)
    ops = (dev(A), dev(sA), dev(B), dev(sB))
    ref = ogemm.gemm_dense(A, sA, B, sB)
    X, W = synthetic.dense_operands(200, 256, 512, kind="normal", seed=32)
    Aq, sAq = oquant.quant_1x128_fast(X)
    Bq, sBq = oquant.quant_128x128_fast(W)
    refq = ogemm.gemm_dense(Aq, sAq, Bq, sBq)
    tX, tB, tsB = dev(X), dev(Bq), dev(sBq)

    torch.cuda.synchronize()
    base = b.workspace_bytes()
    streams = [torch.cuda.Stream() for _ in range(4)]
    held = [base]
    for s in streams:
        with torch.cuda.stream(s):
            D = b.fp8gemm_dense(*ops)
            Dq = b.fp8gemm_dense_quant_a(tX, tB, tsB)
        s.synchronize()
        assert_close(host(D), ref, "decode on a new stream")
        assert_close(host(Dq), refq, "FP32 activations on a new stream")
        held.append(b.workspace_bytes())
    assert all(h2 > h1 for h1, h2 in zip(held, held[1:])), held
    per_stream = held[1] - held[0]
    for i, s in enumerate(streams):
        b.fp8gemm_release_workspaces(s)
        assert b.workspace_bytes() == held[-1] - (i + 1) * per_stream
    assert b.workspace_bytes() == base
    # a released stream gets fresh buffers on its next call
    with torch.cuda.stream(streams[0]):
        D = b.fp8gemm_dense(*ops)
    streams[0].synchronize()
    assert_close(host(D), ref, "decode after release")
    assert b.workspace_bytes() > base
    b.fp8gemm_release_workspaces(streams[0])
    assert b.workspace_bytes() == base
    assert b.fp8gemm_get_device_status() == b.OK


def test_tile_counter_workspaces_are_released():
    """The batched launch's counters and the ordered contiguous form's
    counters and order are per-stream workspaces too: released with the
    stream's other buffers, and allocated again (zeroed) by the next call,
    which is still correct."""
    import numpy as np
    import torch

    from fp8_fine_grained_e4m3_gb300 import binding as b
    from fp8_fine_grained_e4m3_gb300 import synthetic
    from tests.gpu_helpers import quant_weights
    shapes = [(1300, 4000, 640), (300, 520, 1024)]
    probs = [quantised_dense(M, N, K, "prefill", seed=70 + i) for i, (M, N, K) in enumerate(shapes)]
    ops = [tuple(dev(x) for x in p) for p in probs]
    refs = [ogemm.gemm_dense(*p) for p in probs]
    E, N, K = 10, 4096, 512
    counts = synthetic.zipf_counts(E, 2500, seed=71)
    X, W, lay = synthetic.contiguous_operands(E, 2500, N, K, seed=71, counts=counts)
    Ac, sAc = oquant.quant_1x128_fast(X)
    Bq = [quant_weights(W[e]) for e in range(E)]
    Bc = np.stack([q for q, _ in Bq])
    sBc = np.stack([s for _, s in Bq])
    cops = (dev(Ac), dev(sAc), dev(Bc), dev(sBc), dev(lay.m_indices))
    cref = ogemm.gemm_contiguous(Ac, sAc, Bc, sBc, lay.m_indices)

    torch.cuda.synchronize()
    base = b.workspace_bytes()
    s = torch.cuda.Stream()
    for rep in range(2):
        with torch.cuda.stream(s):
            outs = b.fp8gemm_dense_batch(ops)
            Dc = b.fp8gemm_grouped_contiguous(*cops)
        s.synchronize()
        for D, r in zip(outs, refs):
            assert_close(host(D), r, f"batch, pass {rep}")
        assert_close(host(Dc), cref, f"ordered contiguous, pass {rep}")
        assert b.workspace_bytes() > base
        b.fp8gemm_release_workspaces(s)
        assert b.workspace_bytes() == base
    assert b.fp8gemm_get_device_status() == b.OK
