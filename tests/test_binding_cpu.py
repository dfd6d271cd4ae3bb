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
    # past the format check, the next one refuses host memory
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        b.fp8gemm_dense_fmt(a5, s, "e5m2", a4, s, "e4m3")
    with pytest.raises(ValueError, match="format must be one of"):
        b.fp8gemm_dense_fmt(a5, s, "e3m4", a4, s, "e4m3")


def test_plain_calls_refuse_e5m2_tensors():
    b = _b()
    a5 = torch.zeros((2, 128), dtype=torch.float8_e5m2)
    s = torch.ones((2, 1))
    with pytest.raises(TypeError, match="e4m3 bytes"):
        b.fp8gemm_dense(a5, s, a5, s)
