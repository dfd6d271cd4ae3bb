"""The C-ABI library builds, loads and exports every declared entry point;
host-side validation answers without touching a GPU.  CPU only."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(\w+)\s*\([^;{]*\)\s*;", src, re.M)
    return names


@pytest.fixture(scope="module")
def lib():
    from fp8_fine_grained_e4m3_gb300 import build, binding
    build.build()
    return binding.lib()


def test_header_declares_the_boundary():
    names = set(_declared_functions())
    for n in ["fp8_quant_1x128", "fp8_quant_128x128", "fp8gemm_dense", "fp8gemm_dense_quant_a",
              "fp8gemm_grouped_contiguous", "fp8gemm_grouped_masked",
              "fp8gemm_get_device_status", "fp8gemm_strerror"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in _declared_functions():
        assert hasattr(lib, n), n


def test_binding_covers_every_symbol():
    from fp8_fine_grained_e4m3_gb300 import binding
    bound = {n for n, _, _ in binding.SIGNATURES}
    assert set(_declared_functions()) <= bound


def test_strerror_on_host(lib):
    from fp8_fine_grained_e4m3_gb300 import binding
    assert binding.strerror(binding.ERR_SHAPE).startswith("unsupported shape")
    assert binding.strerror(12345) == "unknown status"


def test_host_validation_needs_no_gpu(lib):
    from fp8_fine_grained_e4m3_gb300 import binding as b
    P = ctypes.c_void_p
    good = P(1 << 20)  # never dereferenced: validation fails before any CUDA call
    s = P(0)
    assert lib.fp8gemm_dense(good, good, good, good, good, 128, 256, 200, s) == b.ERR_SHAPE
    assert lib.fp8gemm_dense(good, good, good, good, good, 128, 256, 136, s) == b.ERR_SHAPE
    assert lib.fp8gemm_dense(good, good, good, good, good, 128, -1, 256, s) == b.ERR_SHAPE
    assert lib.fp8gemm_dense(good, good, good, good, good, 128, 256, 0, s) == b.ERR_SHAPE
    assert lib.fp8gemm_dense(None, good, good, good, good, 128, 256, 256, s) == b.ERR_NULL
    assert lib.fp8gemm_dense(P((1 << 20) + 4), good, good, good, good, 128, 256, 256, s) == b.ERR_ALIGN
    assert lib.fp8gemm_dense(good, good, good, good, good, 0, 256, 256, s) == b.OK
    assert lib.fp8gemm_grouped_contiguous(good, good, good, good, good, good,
                                          100, 256, 256, 2, s) == b.ERR_SHAPE
    assert lib.fp8gemm_grouped_masked(good, good, good, good, good, good,
                                      0, 128, 256, 256, s) == b.OK
    assert lib.fp8gemm_dense_quant_a(good, None, None, good, good, good, 4, 256, 200, s) == b.ERR_SHAPE
    assert lib.fp8gemm_dense_quant_a(good, good, None, good, good, good, 4, 256, 256, s) == b.ERR_NULL
    assert lib.fp8gemm_dense_quant_a(None, None, None, good, good, good, 4, 256, 256, s) == b.ERR_NULL
    assert lib.fp8gemm_dense_quant_a(P((1 << 20) + 8), None, None, good, good, good,
                                     4, 256, 256, s) == b.ERR_ALIGN
    assert lib.fp8gemm_dense_quant_a(good, None, None, good, good, good, 0, 256, 256, s) == b.OK
    assert lib.fp8_quant_1x128(good, good, good, 4, 130, s) == b.ERR_SHAPE
    assert lib.fp8_quant_1x128_fmt(good, good, good, 4, 256, 2, s) == b.ERR_FORMAT
    assert lib.fp8_quant_128x128_fmt(good, good, good, 1, 256, 256, -1, s) == b.ERR_FORMAT
    assert lib.fp8gemm_dense_fmt(good, good, 0, good, good, 5, good, 4, 256, 256, s) == b.ERR_FORMAT
    assert lib.fp8gemm_dense_fmt(good, good, 1, good, good, 1, good, 4, 256, 136, s) == b.ERR_SHAPE
    assert lib.fp8gemm_dense_fmt(None, good, 1, good, good, 0, good, 4, 256, 256, s) == b.ERR_NULL
    assert b.strerror(b.ERR_FORMAT).startswith("unknown FP8 format")
    assert lib.fp8gemm_grouped_contiguous_fmt(good, good, 0, good, good, 3, good, good,
                                              128, 256, 256, 2, s) == b.ERR_FORMAT
    assert lib.fp8gemm_grouped_masked_fmt(good, good, 9, good, good, 0, good, good,
                                          2, 128, 256, 256, s) == b.ERR_FORMAT
    assert lib.fp8_quant_128x128(good, None, good, 1, 8, 128, s) == b.ERR_NULL
    assert lib.fp8gemm_grouped_table(good, -1, 16, s) == b.ERR_SHAPE
    assert lib.fp8gemm_grouped_table(good, 4, 0, s) == b.ERR_SHAPE
    assert lib.fp8gemm_grouped_table(None, 4, 16, s) == b.ERR_NULL
    assert lib.fp8gemm_grouped_table(P((1 << 20) + 4), 4, 16, s) == b.ERR_ALIGN
    assert lib.fp8gemm_grouped_table(None, 0, 16, s) == b.OK
    assert lib.fp8gemm_get_device_status(s, None) == b.ERR_NULL
    assert isinstance(lib.fp8gemm_num_kernel_launches(), int)
    assert lib.fp8gemm_workspace_bytes() == 0  # nothing allocated without a GPU
    assert lib.fp8gemm_dense_ex(good, good, 0, good, good, 0, good, 4, 256, 256, 2, s) == b.ERR_FLAGS
    assert lib.fp8gemm_dense_ex(good, good, 0, good, good, 0, good, 4, 256, 136, 1, s) == b.ERR_SHAPE
    assert lib.fp8gemm_dense_ex(good, good, 0, good, good, 0, good, 0, 256, 256, 1, s) == b.OK
    assert b.strerror(b.ERR_FLAGS).startswith("unknown flag")
    # saturation counters: optional, 8-byte aligned; validated before any CUDA call
    assert lib.fp8_quant_1x128_ex(good, good, good, 4, 256, 0, P((1 << 20) + 4), s) == b.ERR_ALIGN
    assert lib.fp8_quant_1x128_ex(good, good, good, 4, 130, 0, good, s) == b.ERR_SHAPE
    assert lib.fp8_quant_1x128_ex(good, good, good, 4, 256, 3, None, s) == b.ERR_FORMAT
    assert lib.fp8_quant_1x128_ex(good, good, good, 0, 256, 0, good, s) == b.OK
    assert lib.fp8_quant_128x128_ex(good, good, good, 1, 8, 128, 0, P((1 << 20) + 12), s) == b.ERR_ALIGN
    assert lib.fp8_quant_128x128_ex(good, None, good, 1, 8, 128, 0, good, s) == b.ERR_NULL
    assert lib.fp8_quant_128x128_ex(good, good, good, 1, 0, 128, 1, good, s) == b.OK


def test_problem_struct_layout():
    """The binding's table entry has the C struct's size and field offsets
    (5 pointers, then M, N, K, formats)."""
    from fp8_fine_grained_e4m3_gb300 import binding as b
    assert ctypes.sizeof(b.Problem) == 56
    assert [getattr(b.Problem, f).offset for f in ("A", "sA", "B", "sB", "D", "M", "N", "K")] == \
        [0, 8, 16, 24, 32, 40, 44, 48]
    hdr = open(os.path.join(ROOT, "include", "fp8gemm.h")).read()
    body = hdr[hdr.index("typedef struct fp8gemm_problem"):hdr.index("} fp8gemm_problem;")]
    assert re.findall(r"\*\s*(\w+);", body) == ["A", "sA", "B", "sB", "D"]
    assert "int M, N, K;" in body and "int formats;" in body


def test_dense_batch_host_validation_needs_no_gpu(lib):
    """fp8gemm_dense_batch checks the count and every entry (sizes, formats,
    pointers, alignment) before any CUDA call."""
    from fp8_fine_grained_e4m3_gb300 import binding as b
    P = ctypes.c_void_p
    s = P(0)
    good = 1 << 20

    def entries(*rows):
        arr = (b.Problem * len(rows))()
        for e, (M, N, K, fmts, ptrs) in zip(arr, rows):
            e.A, e.sA, e.B, e.sB, e.D = ptrs
            e.M, e.N, e.K, e.formats = M, N, K, fmts
        return ctypes.cast(arr, P), len(rows)

    hdr = open(os.path.join(ROOT, "include", "fp8gemm.h")).read()
    assert re.search(r"#define FP8GEMM_MAX_DENSE_BATCH (\d+)", hdr).group(1) == \
        str(b.MAX_DENSE_BATCH)
    ok5 = (good,) * 5
    assert lib.fp8gemm_dense_batch(None, 0, s) == b.OK
    assert lib.fp8gemm_dense_batch(None, -1, s) == b.ERR_SHAPE
    assert lib.fp8gemm_dense_batch(None, b.MAX_DENSE_BATCH + 1, s) == b.ERR_SHAPE
    assert lib.fp8gemm_dense_batch(None, 1, s) == b.ERR_NULL
    # the second entry is bad: nothing is launched for the first either
    assert lib.fp8gemm_dense_batch(*entries((256, 256, 256, 0, ok5), (128, 256, 200, 0, ok5)), s) \
        == b.ERR_SHAPE
    assert lib.fp8gemm_dense_batch(*entries((256, 256, 0, 0, ok5)), s) == b.ERR_SHAPE
    assert lib.fp8gemm_dense_batch(*entries((256, -2, 256, 0, ok5)), s) == b.ERR_SHAPE
    assert lib.fp8gemm_dense_batch(*entries((256, 256, 256, 2, ok5)), s) == b.ERR_FORMAT
    assert lib.fp8gemm_dense_batch(*entries((256, 256, 256, 1 | (3 << 8), ok5)), s) == b.ERR_FORMAT
    assert lib.fp8gemm_dense_batch(*entries((256, 256, 256, 0, (good, None, good, good, good))),
                                   s) == b.ERR_NULL
    assert lib.fp8gemm_dense_batch(*entries((256, 256, 256, 0, (good, good, good, good + 8, good))),
                                   s) == b.ERR_ALIGN
    # empty entries are skipped (no pointer needed): nothing to launch
    assert lib.fp8gemm_dense_batch(*entries((0, 256, 256, 0, (None,) * 5),
                                            (256, 0, 128, 1 | (1 << 8), (None,) * 5)), s) == b.OK


def test_dense_batch_binding_refuses_on_host():
    """The binding refuses more entries than one launch takes, before any
    tensor is touched."""
    from fp8_fine_grained_e4m3_gb300 import binding as b
    with pytest.raises(ValueError, match="at most"):
        b.fp8gemm_dense_batch([None] * (b.MAX_DENSE_BATCH + 1))
