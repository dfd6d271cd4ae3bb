"""C-ABI behaviour on the GPU: validation codes, no-ops, device status."""

import ctypes

import numpy as np
import pytest

from tests.gpu_helpers import dev, host, oquant
from fp8_fine_grained_e4m3_gb300 import synthetic

pytestmark = pytest.mark.gpu


def _b():
    from fp8_fine_grained_e4m3_gb300 import binding
    return binding


def _p(t, off=0):
    return ctypes.c_void_p(t.data_ptr() + off)


def _bufs(M=128, N=256, K=256):
    import torch
    A = torch.zeros((M, K), dtype=torch.uint8, device="cuda")
    sA = torch.ones((M, K // 128), dtype=torch.float32, device="cuda")
    B = torch.zeros((N, K), dtype=torch.uint8, device="cuda")
    sB = torch.ones(((N + 127) // 128, K // 128), dtype=torch.float32, device="cuda")
    D = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    return A, sA, B, sB, D


def test_dense_validation_codes():
    b = _b()
    L = b.lib()
    A, sA, B, sB, D = _bufs()
    s = ctypes.c_void_p(0)
    ok = L.fp8gemm_dense(_p(A), _p(sA), _p(B), _p(sB), _p(D), 128, 256, 256, s)
    assert ok == b.OK
    assert L.fp8gemm_dense(_p(A, 1), _p(sA), _p(B), _p(sB), _p(D), 128, 256, 256, s) == b.ERR_ALIGN
    assert L.fp8gemm_dense(_p(A), _p(sA), _p(B), _p(sB), _p(D, 8), 128, 256, 256, s) == b.ERR_ALIGN
    assert L.fp8gemm_dense(None, _p(sA), _p(B), _p(sB), _p(D), 128, 256, 256, s) == b.ERR_NULL
    assert L.fp8gemm_dense(_p(A), _p(sA), _p(B), _p(sB), _p(D), 128, 256, 200, s) == b.ERR_SHAPE
    assert L.fp8gemm_dense(_p(A), _p(sA), _p(B), _p(sB), _p(D), 128, 256, 136, s) == b.ERR_SHAPE
    assert L.fp8gemm_dense(_p(A), _p(sA), _p(B), _p(sB), _p(D), -1, 256, 256, s) == b.ERR_SHAPE
    assert b.fp8gemm_get_device_status() == b.OK


def test_zero_m_is_noop():
    import torch
    b = _b()
    A, sA, B, sB, D = _bufs()
    D.fill_(3.0)
    assert b.lib().fp8gemm_dense(_p(A), _p(sA), _p(B), _p(sB), _p(D), 0, 256, 256,
                                 ctypes.c_void_p(0)) == b.OK
    torch.cuda.synchronize()
    assert bool((D == 3.0).all())


def test_grouped_validation_codes():
    b = _b()
    L = b.lib()
    A, sA, B, sB, D = _bufs(M=256)
    import torch
    mi = torch.zeros(256, dtype=torch.int32, device="cuda")
    s = ctypes.c_void_p(0)
    assert L.fp8gemm_grouped_contiguous(_p(A), _p(sA), _p(B), _p(sB), _p(mi), _p(D),
                                        200, 256, 256, 1, s) == b.ERR_SHAPE
    assert L.fp8gemm_grouped_contiguous(_p(A), _p(sA), _p(B), _p(sB), None, _p(D),
                                        256, 256, 256, 1, s) == b.ERR_NULL
    assert L.fp8gemm_grouped_masked(_p(A), _p(sA), _p(B), _p(sB), _p(mi, 4), _p(D),
                                    1, 256, 256, 256, s) == b.ERR_ALIGN
    assert L.fp8gemm_grouped_masked(_p(A), _p(sA), _p(B), _p(sB), _p(mi), _p(D),
                                    0, 256, 256, 256, s) == b.OK


def test_bad_expert_index_sets_status():
    import torch
    b = _b()
    X, W, lay = synthetic.contiguous_operands(2, 200, 256, 256, seed=1)
    A, sA = oquant.quant_1x128_fast(X)
    Bq = [oquant.quant_128x128_fast(W[e]) for e in range(2)]
    B = np.stack([q for q, _ in Bq])
    sB = np.stack([s for _, s in Bq])
    mi = lay.m_indices.copy()
    mi[mi == 1] = 7  # expert 7 does not exist
    b.fp8gemm_get_device_status()  # clear
    b.fp8gemm_grouped_contiguous(dev(A), dev(sA), dev(B), dev(sB), dev(mi))
    assert b.fp8gemm_get_device_status() == b.ERR_DEVICE_STATUS
    assert b.fp8gemm_get_device_status() == b.OK  # read clears it
    torch.cuda.synchronize()


def test_masked_count_above_m_max_sets_status():
    import torch
    b = _b()
    E, M_max, N, K = 2, 128, 256, 256
    A, sA, B, sB, D = _bufs(M=E * M_max, N=N, K=K)
    Bq = torch.zeros((E, N, K), dtype=torch.uint8, device="cuda")
    sBq = torch.ones((E, 2, 2), dtype=torch.float32, device="cuda")
    mm = torch.tensor([500, 3], dtype=torch.int32, device="cuda")
    b.fp8gemm_get_device_status()
    b.fp8gemm_grouped_masked(A.view(E, M_max, K), sA.view(E, M_max, 2), Bq, sBq, mm,
                             D=D.view(E, M_max, N))
    assert b.fp8gemm_get_device_status() == b.ERR_DEVICE_STATUS
    torch.cuda.synchronize()


def test_strerror_and_launch_counter():
    b = _b()
    assert "aligned" in b.strerror(b.ERR_ALIGN)
    n0 = b.num_kernel_launches()
    A, sA, B, sB, D = _bufs()
    b.fp8gemm_dense(A, sA, B, sB, D=D)
    assert b.num_kernel_launches() == n0 + 1
