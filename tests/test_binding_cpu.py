"""Argument checks of the Python binding that need no GPU: FP8 tensors whose
own dtype contradicts the stated operand format are refused before any
call reaches the library."""

import pytest

torch = pytest.importorskip("torch")


def _b():
    from fp8_fine_grained_e4m3_gb300 import binding
    return binding


def test_float8_dtype_must_agree_with_the_format():
    b = _b()
    a4 = torch.zeros((2, 128), dtype=torch.float8_e4m3fn)
    a5 = torch.zeros((2, 128), dtype=torch.float8_e5m2)
    s = torch.ones((2, 1))
    with pytest.raises(TypeError, match="format is given as 'e5m2'"):
        b.fp8gemm_dense_fmt(a4, s, "e5m2", a4, s, "e4m3")
    with pytest.raises(TypeError, match="format is given as 'e4m3'"):
        b.fp8gemm_dense_fmt(a5, s, "e4m3", a4, s, "e4m3")
    with pytest.raises(TypeError, match="A is torch.float8_e4m3fn"):
        b.fp8gemm_grouped_masked_fmt(a4.reshape(1, 2, 128), s, "e5m2",
                                     a5.reshape(1, 2, 128), s, "e5m2", torch.ones(1))
    with pytest.raises(TypeError, match="B is torch.float8_e5m2"):
        b._u8_fmt(a5, "e4m3", "B")


def test_agreeing_dtypes_pass_the_format_check():
    b = _b()
    a5 = torch.zeros((2, 128), dtype=torch.float8_e5m2)
    a4 = torch.zeros((2, 128), dtype=torch.float8_e4m3fn)
    s = torch.ones((2, 1))
    sb = torch.ones((1, 1))
    # past the format and shape checks, the next one refuses host memory
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        b.fp8gemm_dense_fmt(a5, s, "e5m2", a4, sb, "e4m3")
    with pytest.raises(ValueError, match="format must be one of"):
        b.fp8gemm_dense_fmt(a5, s, "e3m4", a4, s, "e4m3")


def test_plain_calls_refuse_e5m2_tensors():
    b = _b()
    a5 = torch.zeros((2, 128), dtype=torch.float8_e5m2)
    s = torch.ones((2, 1))
    with pytest.raises(TypeError, match="e4m3 bytes"):
        b.fp8gemm_dense(a5, s, a5, s)


# ------------------------------------------------------------------ shapes
# The C ABI sees only pointers and sizes: a tensor of the wrong size would be
# read or written out of bounds by the kernels.  The binding refuses it before
# any pointer is passed on (these run on host tensors, so the device check
# would fire next).

def _dense_ok(M=4, N=256, K=256):
    u8 = lambda *s: torch.zeros(s, dtype=torch.uint8)  # noqa: E731
    A, B = u8(M, K), u8(N, K)
    sA, sB = torch.ones((M, -(-K // 128))), torch.ones((-(-N // 128), -(-K // 128)))
    D = torch.empty((M, N), dtype=torch.bfloat16)
    return A, sA, B, sB, D


@pytest.mark.parametrize("call", ["fp8gemm_dense", "fp8gemm_dense_small_m_noalloc"])
@pytest.mark.parametrize("bad,match", [
    ("D_rows", "D has shape"), ("D_cols", "D has shape"), ("D_dtype", "D must be bfloat16"),
    ("B_k", "B has shape"), ("sA", "sA has shape"), ("sB", "sB has shape"), ("A_dim", "A has shape"),
])
def test_dense_calls_refuse_wrong_shapes(call, bad, match):
    b = _b()
    A, sA, B, sB, D = _dense_ok()
    if bad == "D_rows":
        D = torch.empty((3, 256), dtype=torch.bfloat16)
    elif bad == "D_cols":
        D = torch.empty((4, 128), dtype=torch.bfloat16)
    elif bad == "D_dtype":
        D = torch.empty((4, 256), dtype=torch.float32)
    elif bad == "B_k":
        B = torch.zeros((256, 128), dtype=torch.uint8)
    elif bad == "sA":
        sA = torch.ones((4, 1))
    elif bad == "sB":
        sB = torch.ones((1, 2))
    elif bad == "A_dim":
        A = A.reshape(-1)
    with pytest.raises((ValueError, TypeError), match=match):
        getattr(b, call)(A, sA, B, sB, D)


def test_well_shaped_dense_call_reaches_the_device_check():
    b = _b()
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        b.fp8gemm_dense(*_dense_ok())
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        b.fp8gemm_dense_small_m_noalloc(*_dense_ok())


def test_quantisers_refuse_wrong_outputs():
    b = _b()
    X = torch.zeros((4, 256))
    with pytest.raises(ValueError, match="Q has shape"):
        b.fp8_quant_1x128(X, Q=torch.zeros((4, 128), dtype=torch.uint8), sX=torch.ones((4, 2)))
    with pytest.raises(ValueError, match="sX has shape"):
        b.fp8_quant_1x128(X, Q=torch.zeros((4, 256), dtype=torch.uint8), sX=torch.ones((4, 1)))
    W = torch.zeros((2, 300, 256))
    with pytest.raises(ValueError, match="sW has shape"):
        b.fp8_quant_128x128(W, Q=torch.zeros((2, 300, 256), dtype=torch.uint8),
                            sW=torch.ones((2, 2, 2)))


def test_grouped_calls_refuse_wrong_shapes():
    b = _b()
    u8 = lambda *s: torch.zeros(s, dtype=torch.uint8)  # noqa: E731
    E, N, K = 2, 256, 256
    B, sB = u8(E, N, K), torch.ones((E, 2, 2))
    # contiguous: m_indices must cover every row, D every row x N
    A, sA = u8(256, K), torch.ones((256, 2))
    mi = torch.zeros(256, dtype=torch.int32)
    with pytest.raises(ValueError, match="index array"):
        b.fp8gemm_grouped_contiguous(A, sA, B, sB, mi[:128],
                                     D=torch.empty((256, N), dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="D has shape"):
        b.fp8gemm_grouped_contiguous(A, sA, B, sB, mi, D=torch.empty((128, N), dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="sB has shape"):
        b.fp8gemm_grouped_contiguous(A, sA, B, torch.ones((E, 1, 2)), mi,
                                     D=torch.empty((256, N), dtype=torch.bfloat16))
    # masked: B must hold E experts, masked_m E entries
    Am, sAm = u8(E, 128, K), torch.ones((E, 128, 2))
    mm = torch.zeros(E, dtype=torch.int32)
    with pytest.raises(ValueError, match="B has shape"):
        b.fp8gemm_grouped_masked(Am, sAm, u8(E + 1, N, K), torch.ones((E + 1, 2, 2)), mm,
                                 D=torch.empty((E, 128, N), dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="index array"):
        b.fp8gemm_grouped_masked(Am, sAm, B, sB, mm[:1],
                                 D=torch.empty((E, 128, N), dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="sA has shape"):
        b.fp8gemm_grouped_masked(Am, torch.ones((E, 128, 1)), B, sB, mm,
                                 D=torch.empty((E, 128, N), dtype=torch.bfloat16))


def test_problem_table_checks_every_entry():
    b = _b()
    A, sA, B, sB, D = _dense_ok()
    with pytest.raises(ValueError, match="D has shape"):
        b.problem_table([(A, sA, B, sB, D[:2])])
