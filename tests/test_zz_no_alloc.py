"""fp8gemm_dense_small_m_noalloc: the decode-shape GEMM for callers that must
not let the library allocate device memory (servers with a fixed memory
budget reserved at start-up, frameworks whose own pool owns the device
memory, loops that cannot take cudaMalloc's implicit synchronisation).

It is called through the C ABI on two calls in a row with different inputs,
and each result is compared with the FP64 oracle (the acceptance test of the
GEMM) and with fp8gemm_dense, the entry point that keeps a cudaMalloc'd
workspace.  The second call also shows that what the first left in the shared
scratch does not leak into its result.  After the first call on the device,
further calls must leave the device's free memory unchanged.  The file name
sorts last so that a run stopping at the first failure has already run every
other test.
"""

import ctypes

import pytest

from tests.gpu_helpers import assert_close, dev, host, ogemm, quantised_dense

pytestmark = pytest.mark.gpu


def _lib():
    from fp8_fine_grained_e4m3_gb300 import binding
    return binding, binding.lib()


def _p(t, off=0):
    return ctypes.c_void_p(t.data_ptr() + off)


def _call(L, ops, D, M, N, K):
    import torch
    A, sA, B, sB = ops
    return L.fp8gemm_dense_small_m_noalloc(
        _p(A), _p(sA), _p(B), _p(sB), _p(D), M, N, K,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("M,N,K", [
    (16, 7168, 2048), (64, 2048, 7168), (1, 7168, 2048),
    (17, 128, 16384),   # one N tile: its K range shared by several CTAs (stream-K fix-up)
    (5, 777, 400),      # partial last K block (16 of 128 columns), N odd
    (33, 1000, 1280),   # N % 8 != 0, rows not a multiple of the padded width
])
def test_noalloc_matches_oracle_and_dense_on_two_calls(M, N, K):
    import torch
    b, L = _lib()
    cases = []
    for seed in (M + 1, M + 2):
        A, sA, B, sB = quantised_dense(M, N, K, "decode", seed=seed)
        ops = (dev(A), dev(sA), dev(B), dev(sB))
        cases.append((ops, ogemm.gemm_dense(A, sA, B, sB)))
    outs = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in cases]
    # first call on the device: set-up (the scratch's address, module load)
    assert _call(L, cases[0][0], outs[0], M, N, K) == b.OK
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for (ops, _), D in zip(cases, outs):
        rc = _call(L, ops, D, M, N, K)
        assert rc == b.OK, b.strerror(rc)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0, "the no-allocation call changed free memory"
    for call, ((ops, ref), D) in enumerate(zip(cases, outs)):
        got = host(D)
        assert_close(got, ref, f"no-alloc call {call + 1} vs oracle, {M}x{N}x{K}")
        assert_close(got, host(b.fp8gemm_dense(*ops)), f"no-alloc call {call + 1} vs dense")
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
