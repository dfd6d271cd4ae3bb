"""fp8gemm_dense_small_m_noalloc: the decode-shape GEMM for callers that must
not let the library allocate device memory (servers with a fixed memory
budget reserved at start-up, frameworks whose own pool owns the device
memory, loops that cannot take cudaMalloc's implicit synchronisation).

It is called through the C ABI and compared with fp8gemm_dense -- the entry
point that keeps a cudaMalloc'd workspace -- on two calls in a row with
different inputs, so the second call also shows that what the first left in
the shared scratch does not leak into its result.  The file name sorts last so
that a run stopping at the first failure has already run every other test.
"""

import ctypes

import numpy as np
import pytest

from tests.gpu_helpers import assert_close, dev, host, quantised_dense

pytestmark = pytest.mark.gpu


def _lib():
    from fp8_fine_grained_e4m3_gb300 import binding
    return binding, binding.lib()


def _p(t, off=0):
    return ctypes.c_void_p(t.data_ptr() + off)


def _noalloc(L, A, sA, B, sB, M, N, K):
    import torch
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    rc = L.fp8gemm_dense_small_m_noalloc(_p(A), _p(sA), _p(B), _p(sB), _p(D), M, N, K,
                                         ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc, D


@pytest.mark.parametrize("M,N,K", [(16, 7168, 2048), (64, 2048, 7168), (1, 7168, 2048)])
def test_noalloc_matches_dense_on_two_calls(M, N, K):
    b, L = _lib()
    for call, seed in enumerate((M + 1, M + 2)):
        A, sA, B, sB = quantised_dense(M, N, K, "decode", seed=seed)
        tA, tsA, tB, tsB = dev(A), dev(sA), dev(B), dev(sB)
        rc, D = _noalloc(L, tA, tsA, tB, tsB, M, N, K)
        assert rc == b.OK, b.strerror(rc)
        ref = host(b.fp8gemm_dense(tA, tsA, tB, tsB))
        assert_close(host(D), ref, f"no-alloc call {call + 1}, {M}x{N}x{K}")
    assert b.fp8gemm_get_device_status() == b.OK


def test_noalloc_rejects_what_its_scratch_cannot_hold():
    import torch
    b, L = _lib()
    A = torch.zeros((65, 256), dtype=torch.uint8, device="cuda")
    sA = torch.ones((65, 2), dtype=torch.float32, device="cuda")
    B = torch.zeros((256, 256), dtype=torch.uint8, device="cuda")
    sB = torch.ones((2, 2), dtype=torch.float32, device="cuda")
    D = torch.empty((65, 256), dtype=torch.bfloat16, device="cuda")
    s = ctypes.c_void_p(0)
    assert L.fp8gemm_dense_small_m_noalloc(_p(A), _p(sA), _p(B), _p(sB), _p(D),
                                           65, 256, 256, s) == b.ERR_SCRATCH_LIMIT
    assert "scratch" in b.strerror(b.ERR_SCRATCH_LIMIT)
    assert L.fp8gemm_dense_small_m_noalloc(_p(A), _p(sA), _p(B), _p(sB), _p(D),
                                           4, 256, 200, s) == b.ERR_SHAPE
    assert L.fp8gemm_dense_small_m_noalloc(_p(A), _p(sA), _p(B), _p(sB), _p(D, 2),
                                           4, 256, 256, s) == b.ERR_ALIGN
