"""ctypes binding over libfp8gemm.so (include/fp8gemm.h).

Argument marshalling only: every function here checks tensor metadata,
allocates outputs with torch when the caller gives none, and passes raw
device pointers plus the current CUDA stream to the C ABI.  All arithmetic
runs in the library's kernels.  There is no fallback: if the library is
missing or a call fails, an exception is raised.

FP8 operands are uint8 tensors holding e4m3 bytes (a torch.float8_e4m3fn
tensor is accepted and viewed as uint8); scales are float32; outputs are
bfloat16.
"""

import ctypes
import os
import threading

from . import build as _build

OK = 0
ERR_NULL = -1
ERR_ALIGN = -2
ERR_SHAPE = -3
ERR_ARCH = -4
ERR_LAUNCH = -5
ERR_DEVICE_STATUS = -6
ERR_TIMEOUT = -7
ERR_SCRATCH_LIMIT = -8
ERR_FORMAT = -9
FMT = {"e4m3": 0, "e5m2": 1}  # FP8GEMM_FMT_*

_lib = None
_lock = threading.Lock()

# (name, restype, argtypes) for every entry point of include/fp8gemm.h
_P = ctypes.c_void_p
_I = ctypes.c_int
SIGNATURES = [
    ("fp8_quant_1x128", _I, [_P, _P, _P, _I, _I, _P]),
    ("fp8_quant_128x128", _I, [_P, _P, _P, _I, _I, _I, _P]),
    ("fp8gemm_dense", _I, [_P, _P, _P, _P, _P, _I, _I, _I, _P]),
    ("fp8_quant_1x128_fmt", _I, [_P, _P, _P, _I, _I, _I, _P]),
    ("fp8_quant_128x128_fmt", _I, [_P, _P, _P, _I, _I, _I, _I, _P]),
    ("fp8gemm_dense_fmt", _I, [_P, _P, _I, _P, _P, _I, _P, _I, _I, _I, _P]),
    ("fp8gemm_grouped_table", _I, [_P, _I, _I, _P]),
    ("fp8gemm_grouped_contiguous_fmt", _I,
     [_P, _P, _I, _P, _P, _I, _P, _P, _I, _I, _I, _I, _P]),
    ("fp8gemm_grouped_masked_fmt", _I, [_P, _P, _I, _P, _P, _I, _P, _P, _I, _I, _I, _I, _P]),
    ("fp8gemm_dense_quant_a", _I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _P]),
    ("fp8gemm_grouped_contiguous", _I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P]),
    ("fp8gemm_grouped_masked", _I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P]),
    ("fp8gemm_dense_small_m_noalloc", _I, [_P, _P, _P, _P, _P, _I, _I, _I, _P]),
    ("fp8gemm_get_device_status", _I, [_P, ctypes.POINTER(ctypes.c_int)]),
    ("fp8gemm_strerror", ctypes.c_char_p, [_I]),
    ("fp8gemm_num_kernel_launches", ctypes.c_uint64, []),
]


class FP8GemmError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        super().__init__(f"{where}: {strerror(code)} (code {code})")


def library_path():
    return _build.LIB_PATH


def lib():
    """Load libfp8gemm.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                path = library_path()
                if not os.path.exists(path):
                    raise RuntimeError(
                        f"{path} is missing: build it first "
                        "(python -c 'import __graft_entry__ as g; g.build()')")
                L = ctypes.CDLL(path)
                for name, res, args in SIGNATURES:
                    f = getattr(L, name)
                    f.restype = res
                    f.argtypes = args
                _lib = L
    return _lib


def strerror(code: int) -> str:
    return lib().fp8gemm_strerror(int(code)).decode()


def num_kernel_launches() -> int:
    return int(lib().fp8gemm_num_kernel_launches())


def _check(code, where):
    if code != OK:
        raise FP8GemmError(code, where)


# ----------------------------------------------------------------- helpers
def _torch():
    import torch
    return torch


def _stream(stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _u8(t, name):
    torch = _torch()
    if t.dtype == torch.float8_e4m3fn:
        t = t.view(torch.uint8)
    if t.dtype != torch.uint8:
        raise TypeError(f"{name} must hold e4m3 bytes (uint8 or float8_e4m3fn), got {t.dtype}")
    return _dev(t, name)


def _f32(t, name):
    if t.dtype != _torch().float32:
        raise TypeError(f"{name} must be float32, got {t.dtype}")
    return _dev(t, name)


def _i32(t, name):
    if t.dtype != _torch().int32:
        raise TypeError(f"{name} must be int32, got {t.dtype}")
    return _dev(t, name)


def _dev(t, name):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


# ------------------------------------------------------------ entry points
def fp8_quant_1x128(X, Q=None, sX=None, stream=None):
    """X f32 [..., K] -> (Q u8 [..., K], sX f32 [..., ceil(K/128)]).  Leading dims
    are flattened into M."""
    torch = _torch()
    X = _f32(X, "X")
    K = X.shape[-1]
    M = X.numel() // K if K else 0
    if Q is None:
        Q = torch.empty(X.shape, dtype=torch.uint8, device=X.device)
    if sX is None:
        sX = torch.empty((*X.shape[:-1], -(-K // 128)), dtype=torch.float32, device=X.device)
    _check(lib().fp8_quant_1x128(_ptr(X), _ptr(_u8(Q, "Q")), _ptr(_f32(sX, "sX")), M, K,
                                 _stream(stream)), "fp8_quant_1x128")
    return Q, sX


def fp8_quant_128x128(W, Q=None, sW=None, stream=None):
    """W f32 [N, K] or [E, N, K] -> (Q u8 same shape, sW f32 [(E,) ceil(N/128), K/128])."""
    torch = _torch()
    W = _f32(W, "W")
    squeeze = W.dim() == 2
    W3 = W.unsqueeze(0) if squeeze else W
    E, N, K = W3.shape
    if Q is None:
        Q = torch.empty(W.shape, dtype=torch.uint8, device=W.device)
    if sW is None:
        shp = ((N + 127) // 128, -(-K // 128))
        sW = torch.empty(shp if squeeze else (E, *shp), dtype=torch.float32, device=W.device)
    _check(lib().fp8_quant_128x128(_ptr(W3), _ptr(_u8(Q, "Q")), _ptr(_f32(sW, "sW")), E, N, K,
                                   _stream(stream)), "fp8_quant_128x128")
    return Q, sW


def fp8gemm_dense(A, sA, B, sB, D=None, stream=None):
    """A u8 [M, K], sA [M, K/128], B u8 [N, K], sB [ceil(N/128), K/128] -> D bf16 [M, N]."""
    torch = _torch()
    A, B = _u8(A, "A"), _u8(B, "B")
    M, K = A.shape
    N = B.shape[0]
    if D is None:
        D = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _check(lib().fp8gemm_dense(_ptr(A), _ptr(_f32(sA, "sA")), _ptr(B), _ptr(_f32(sB, "sB")),
                               _ptr(_dev(D, "D")), M, N, K, _stream(stream)), "fp8gemm_dense")
    return D


def _fmt(name):
    if name not in FMT:
        raise ValueError(f"format must be one of {sorted(FMT)}, got {name!r}")
    return FMT[name]


def _u8_fmt(t, fmt, name):
    """FP8 bytes in format `fmt`: a uint8 tensor, or a torch float8 tensor
    whose own format agrees with `fmt` (viewed as uint8)."""
    torch = _torch()
    _fmt(fmt)
    own = {torch.float8_e4m3fn: "e4m3", torch.float8_e5m2: "e5m2"}.get(t.dtype)
    if own is not None:
        if own != fmt:
            raise TypeError(f"{name} is {t.dtype} but its format is given as {fmt!r}")
        t = t.view(torch.uint8)
    if t.dtype != torch.uint8:
        raise TypeError(f"{name} must hold FP8 bytes (uint8 or a float8 dtype), got {t.dtype}")
    return _dev(t, name)


def fp8_quant_1x128_fmt(X, fmt, Q=None, sX=None, stream=None):
    """fp8_quant_1x128 with the output format ("e4m3" or "e5m2")."""
    torch = _torch()
    X = _f32(X, "X")
    K = X.shape[-1]
    M = X.numel() // K if K else 0
    if Q is None:
        Q = torch.empty(X.shape, dtype=torch.uint8, device=X.device)
    if sX is None:
        sX = torch.empty((*X.shape[:-1], -(-K // 128)), dtype=torch.float32, device=X.device)
    _check(lib().fp8_quant_1x128_fmt(_ptr(X), _ptr(_u8_fmt(Q, fmt, "Q")), _ptr(_f32(sX, "sX")),
                                     M, K, _fmt(fmt), _stream(stream)), "fp8_quant_1x128_fmt")
    return Q, sX


def fp8_quant_128x128_fmt(W, fmt, Q=None, sW=None, stream=None):
    """fp8_quant_128x128 with the output format ("e4m3" or "e5m2")."""
    torch = _torch()
    W = _f32(W, "W")
    squeeze = W.dim() == 2
    W3 = W.unsqueeze(0) if squeeze else W
    E, N, K = W3.shape
    if Q is None:
        Q = torch.empty(W.shape, dtype=torch.uint8, device=W.device)
    if sW is None:
        shp = ((N + 127) // 128, -(-K // 128))
        sW = torch.empty(shp if squeeze else (E, *shp), dtype=torch.float32, device=W.device)
    _check(lib().fp8_quant_128x128_fmt(_ptr(W3), _ptr(_u8_fmt(Q, fmt, "Q")), _ptr(_f32(sW, "sW")),
                                       E, N, K, _fmt(fmt), _stream(stream)),
           "fp8_quant_128x128_fmt")
    return Q, sW


def fp8gemm_dense_fmt(A, sA, a_fmt, B, sB, b_fmt, D=None, stream=None):
    """fp8gemm_dense with operand formats ("e4m3" / "e5m2") for A and B."""
    torch = _torch()
    A, B = _u8_fmt(A, a_fmt, "A"), _u8_fmt(B, b_fmt, "B")
    M, K = A.shape
    N = B.shape[0]
    if D is None:
        D = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _check(lib().fp8gemm_dense_fmt(_ptr(A), _ptr(_f32(sA, "sA")), _fmt(a_fmt), _ptr(B),
                                   _ptr(_f32(sB, "sB")), _fmt(b_fmt), _ptr(_dev(D, "D")), M, N,
                                   K, _stream(stream)), "fp8gemm_dense_fmt")
    return D


def fp8gemm_dense_quant_a(X, B, sB, D=None, Q=None, sA=None, stream=None):
    """X f32 [M, K], B u8 [N, K], sB [ceil(N/128), K/128] -> D bf16 [M, N], with A
    quantised 1x128 on load.  Q u8 [M, K] and sA f32 [M, K/128] (both or neither)
    receive the quantised activations."""
    torch = _torch()
    X, B = _f32(X, "X"), _u8(B, "B")
    M, K = X.shape
    N = B.shape[0]
    if D is None:
        D = torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    if (Q is None) != (sA is None):
        raise ValueError("Q and sA go together: give both or neither")
    qp = _ptr(_u8(Q, "Q")) if Q is not None else None
    sp = _ptr(_f32(sA, "sA")) if sA is not None else None
    _check(lib().fp8gemm_dense_quant_a(_ptr(X), qp, sp, _ptr(B), _ptr(_f32(sB, "sB")),
                                       _ptr(_dev(D, "D")), M, N, K, _stream(stream)),
           "fp8gemm_dense_quant_a")
    return D


class Problem(ctypes.Structure):
    """One entry of the fp8gemm_grouped_table problem table (C layout)."""
    _fields_ = [("A", _P), ("sA", _P), ("B", _P), ("sB", _P), ("D", _P),
                ("M", ctypes.c_int), ("N", ctypes.c_int), ("K", ctypes.c_int),
                ("reserved", ctypes.c_int)]


def problem_table(problems, out=None):
    """Device table for fp8gemm_grouped_table from (A, sA, B, sB, D) tensor
    tuples: a uint8 CUDA tensor of len(problems) * sizeof(Problem) bytes
    (written into `out` when given, e.g. to update a table a graph captured)."""
    torch = _torch()
    arr = (Problem * len(problems))()
    for e, (A, sA, B, sB, D) in zip(arr, problems):
        A, B = _u8(A, "A"), _u8(B, "B")
        e.A, e.sA, e.B = A.data_ptr(), _f32(sA, "sA").data_ptr(), B.data_ptr()
        e.sB, e.D = _f32(sB, "sB").data_ptr(), _dev(D, "D").data_ptr()
        e.M, e.K = A.shape
        e.N = B.shape[0]
        e.reserved = 0
    host = torch.frombuffer(bytearray(bytes(arr)), dtype=torch.uint8)
    if out is None:
        return host.to("cuda")
    out.copy_(host)
    return out


def fp8gemm_grouped_table(table, num_problems, max_M, stream=None):
    """Run every problem of a device table (see problem_table); max_M bounds
    every entry's M (<= 64) and picks the kernel's padded width."""
    _check(lib().fp8gemm_grouped_table(_ptr(_dev(table, "table")), int(num_problems),
                                       int(max_M), _stream(stream)), "fp8gemm_grouped_table")


def fp8gemm_grouped_contiguous(A, sA, B, sB, m_indices, D=None, stream=None):
    """A u8 [M_pad, K], B u8 [E, N, K], m_indices i32 [M_pad] -> D bf16 [M_pad, N]."""
    torch = _torch()
    A, B = _u8(A, "A"), _u8(B, "B")
    M_pad, K = A.shape
    E, N = B.shape[0], B.shape[1]
    if D is None:
        D = torch.empty((M_pad, N), dtype=torch.bfloat16, device=A.device)
    _check(lib().fp8gemm_grouped_contiguous(
        _ptr(A), _ptr(_f32(sA, "sA")), _ptr(B), _ptr(_f32(sB, "sB")),
        _ptr(_i32(m_indices, "m_indices")), _ptr(_dev(D, "D")), M_pad, N, K, E,
        _stream(stream)), "fp8gemm_grouped_contiguous")
    return D


def fp8gemm_grouped_masked(A, sA, B, sB, masked_m, D=None, stream=None):
    """A u8 [E, M_max, K], B u8 [E, N, K], masked_m i32 [E] -> D bf16 [E, M_max, N]
    (rows >= masked_m[e] are not written)."""
    torch = _torch()
    A, B = _u8(A, "A"), _u8(B, "B")
    E, M_max, K = A.shape
    N = B.shape[1]
    if D is None:
        D = torch.empty((E, M_max, N), dtype=torch.bfloat16, device=A.device)
    _check(lib().fp8gemm_grouped_masked(
        _ptr(A), _ptr(_f32(sA, "sA")), _ptr(B), _ptr(_f32(sB, "sB")),
        _ptr(_i32(masked_m, "masked_m")), _ptr(_dev(D, "D")), E, M_max, N, K,
        _stream(stream)), "fp8gemm_grouped_masked")
    return D


def fp8gemm_grouped_contiguous_fmt(A, sA, a_fmt, B, sB, b_fmt, m_indices, D=None, stream=None):
    """fp8gemm_grouped_contiguous with operand formats ("e4m3" / "e5m2")."""
    torch = _torch()
    A, B = _u8_fmt(A, a_fmt, "A"), _u8_fmt(B, b_fmt, "B")
    M_pad, K = A.shape
    E, N = B.shape[0], B.shape[1]
    if D is None:
        D = torch.empty((M_pad, N), dtype=torch.bfloat16, device=A.device)
    _check(lib().fp8gemm_grouped_contiguous_fmt(
        _ptr(A), _ptr(_f32(sA, "sA")), _fmt(a_fmt), _ptr(B), _ptr(_f32(sB, "sB")), _fmt(b_fmt),
        _ptr(_i32(m_indices, "m_indices")), _ptr(_dev(D, "D")), M_pad, N, K, E,
        _stream(stream)), "fp8gemm_grouped_contiguous_fmt")
    return D


def fp8gemm_grouped_masked_fmt(A, sA, a_fmt, B, sB, b_fmt, masked_m, D=None, stream=None):
    """fp8gemm_grouped_masked with operand formats ("e4m3" / "e5m2")."""
    torch = _torch()
    A, B = _u8_fmt(A, a_fmt, "A"), _u8_fmt(B, b_fmt, "B")
    E, M_max, K = A.shape
    N = B.shape[1]
    if D is None:
        D = torch.empty((E, M_max, N), dtype=torch.bfloat16, device=A.device)
    _check(lib().fp8gemm_grouped_masked_fmt(
        _ptr(A), _ptr(_f32(sA, "sA")), _fmt(a_fmt), _ptr(B), _ptr(_f32(sB, "sB")), _fmt(b_fmt),
        _ptr(_i32(masked_m, "masked_m")), _ptr(_dev(D, "D")), E, M_max, N, K,
        _stream(stream)), "fp8gemm_grouped_masked_fmt")
    return D


def fp8gemm_dense_small_m_noalloc(A, sA, B, sB, D, stream=None):
    """fp8gemm_dense for M <= 64 without any device allocation by the library:
    the caller provides D, and the split-K scratch is a fixed array inside the
    library (shared by every call on the device; calls must not overlap on the
    GPU)."""
    A, B = _u8(A, "A"), _u8(B, "B")
    M, K = A.shape
    N = B.shape[0]
    _check(lib().fp8gemm_dense_small_m_noalloc(
        _ptr(A), _ptr(_f32(sA, "sA")), _ptr(B), _ptr(_f32(sB, "sB")), _ptr(_dev(D, "D")),
        M, N, K, _stream(stream)), "fp8gemm_dense_small_m_noalloc")
    return D


def fp8gemm_get_device_status(stream=None) -> int:
    """Synchronise the stream, then read and clear the device status word."""
    out = ctypes.c_int(0)
    _check(lib().fp8gemm_get_device_status(_stream(stream), ctypes.byref(out)),
           "fp8gemm_get_device_status")
    return out.value
