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
ERR_FLAGS = -10
FMT = {"e4m3": 0, "e5m2": 1}  # FP8GEMM_FMT_*
FLAG_B_READ_ONLY = 1  # FP8GEMM_FLAG_B_READ_ONLY

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
    ("fp8_quant_1x128_ex", _I, [_P, _P, _P, _I, _I, _I, _P, _P]),
    ("fp8_quant_128x128_ex", _I, [_P, _P, _P, _I, _I, _I, _I, _P, _P]),
    ("fp8gemm_dense_fmt", _I, [_P, _P, _I, _P, _P, _I, _P, _I, _I, _I, _P]),
    ("fp8gemm_dense_ex", _I, [_P, _P, _I, _P, _P, _I, _P, _I, _I, _I, ctypes.c_uint, _P]),
    ("fp8gemm_grouped_table", _I, [_P, _I, _I, _P]),
    ("fp8gemm_dense_batch", _I, [_P, _I, _P]),
    ("fp8gemm_grouped_contiguous_fmt", _I,
     [_P, _P, _I, _P, _P, _I, _P, _P, _I, _I, _I, _I, _P]),
    ("fp8gemm_grouped_masked_fmt", _I, [_P, _P, _I, _P, _P, _I, _P, _P, _I, _I, _I, _I, _P]),
    ("fp8gemm_dense_quant_a", _I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _P]),
    ("fp8gemm_dense_quant_a_ex", _I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, ctypes.c_uint, _P]),
    ("fp8gemm_grouped_contiguous", _I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P]),
    ("fp8gemm_grouped_masked", _I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P]),
    ("fp8gemm_dense_small_m_noalloc", _I, [_P, _P, _P, _P, _P, _I, _I, _I, _P]),
    ("fp8gemm_get_device_status", _I, [_P, ctypes.POINTER(ctypes.c_int)]),
    ("fp8gemm_strerror", ctypes.c_char_p, [_I]),
    ("fp8gemm_num_kernel_launches", ctypes.c_uint64, []),
    ("fp8gemm_release_workspaces", _I, [_P]),
    ("fp8gemm_workspace_bytes", ctypes.c_uint64, []),
    ("fp8gemm_set_wait_limit_ns", _I, [ctypes.c_uint64]),
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
    return t


def _f32(t, name):
    if t.dtype != _torch().float32:
        raise TypeError(f"{name} must be float32, got {t.dtype}")
    return t


def _i32(t, name):
    if t.dtype != _torch().int32:
        raise TypeError(f"{name} must be int32, got {t.dtype}")
    return t


def _bf16(t, name):
    if t.dtype != _torch().bfloat16:
        raise TypeError(f"{name} must be bfloat16, got {t.dtype}")
    return t


def _cdiv(a, b):
    return -(-a // b)


def _need(t, name, elems, last=None):
    """The library reads or writes exactly `elems` contiguous elements of t
    (a row length of `last` when given): refuse a tensor of another size
    before any pointer reaches a kernel, where it would be read or written
    out of bounds."""
    if t.numel() != elems or (last is not None and elems > 0 and t.shape[-1] != last):
        want = f"{elems} elements" + (f" in rows of {last}" if last is not None else "")
        raise ValueError(f"{name} has shape {tuple(t.shape)}; the call needs {want}")
    return t


def _shape_dense(A, sA, B, sB, D, M, N, K):
    """Operand sizes of the dense forms: A [M, K], sA [M, ceil(K/128)],
    B [N, K], sB [ceil(N/128), ceil(K/128)], D bf16 [M, N]."""
    Kb = _cdiv(K, 128)
    if B.dim() != 2 or B.shape[1] != K:
        raise ValueError(f"B has shape {tuple(B.shape)}; the call needs [N, {K}]")
    _need(sA, "sA", M * Kb, Kb)
    _need(sB, "sB", _cdiv(N, 128) * Kb, Kb)
    _need(_bf16(D, "D"), "D", M * N, N)


def _dev(t, name):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _ptr(t, name="tensor"):
    return ctypes.c_void_p(_dev(t, name).data_ptr())


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
        sX = torch.empty((*X.shape[:-1], _cdiv(K, 128)), dtype=torch.float32, device=X.device)
    _need(_u8(Q, "Q"), "Q", M * K, K)
    _need(_f32(sX, "sX"), "sX", M * _cdiv(K, 128), _cdiv(K, 128))
    _check(lib().fp8_quant_1x128(_ptr(X, "X"), _ptr(_u8(Q, "Q"), "Q"), _ptr(sX, "sX"), M, K,
                                 _stream(stream)), "fp8_quant_1x128")
    return Q, sX


def _weights3(W):
    W = _f32(W, "W")
    if W.dim() not in (2, 3):
        raise ValueError(f"W has shape {tuple(W.shape)}; the call needs [N, K] or [E, N, K]")
    return W, W.dim() == 2, (W.unsqueeze(0) if W.dim() == 2 else W)


def fp8_quant_128x128(W, Q=None, sW=None, stream=None):
    """W f32 [N, K] or [E, N, K] -> (Q u8 same shape, sW f32 [(E,) ceil(N/128), K/128])."""
    torch = _torch()
    W, squeeze, W3 = _weights3(W)
    E, N, K = W3.shape
    shp = (_cdiv(N, 128), _cdiv(K, 128))
    if Q is None:
        Q = torch.empty(W.shape, dtype=torch.uint8, device=W.device)
    if sW is None:
        sW = torch.empty(shp if squeeze else (E, *shp), dtype=torch.float32, device=W.device)
    _need(_u8(Q, "Q"), "Q", E * N * K, K)
    _need(_f32(sW, "sW"), "sW", E * shp[0] * shp[1], shp[1])
    _check(lib().fp8_quant_128x128(_ptr(W3, "W"), _ptr(_u8(Q, "Q"), "Q"), _ptr(sW, "sW"), E, N,
                                   K, _stream(stream)), "fp8_quant_128x128")
    return Q, sW


def _dense_mnk(A, B, name_a="A"):
    if A.dim() != 2:
        raise ValueError(f"{name_a} has shape {tuple(A.shape)}; the call needs [M, K]")
    M, K = A.shape
    if B.dim() != 2:
        raise ValueError(f"B has shape {tuple(B.shape)}; the call needs [N, {K}]")
    return M, B.shape[0], K


def fp8gemm_dense(A, sA, B, sB, D=None, stream=None):
    """A u8 [M, K], sA [M, K/128], B u8 [N, K], sB [ceil(N/128), K/128] -> D bf16 [M, N]."""
    torch = _torch()
    A, B = _u8(A, "A"), _u8(B, "B")
    M, N, K = _dense_mnk(A, B)
    if D is None:
        D = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _shape_dense(A, _f32(sA, "sA"), B, _f32(sB, "sB"), D, M, N, K)
    _check(lib().fp8gemm_dense(_ptr(A, "A"), _ptr(sA, "sA"), _ptr(B, "B"), _ptr(sB, "sB"),
                               _ptr(D, "D"), M, N, K, _stream(stream)), "fp8gemm_dense")
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
    return t


def _counter(t):
    """Device address of a saturation counter: an int64 CUDA tensor (its
    first element is added to), or None."""
    torch = _torch()
    if t is None:
        return None
    if t.dtype != torch.int64 or t.numel() < 1:
        raise TypeError(f"sat_count must be an int64 tensor of at least one element, got {t.dtype}")
    return _ptr(t, "sat_count")


def fp8_quant_1x128_fmt(X, fmt, Q=None, sX=None, stream=None, sat_count=None):
    """fp8_quant_1x128 with the output format ("e4m3" or "e5m2").  sat_count
    (an int64 CUDA tensor) receives, added to its first element, the number of
    values the saturating encoding clamped (fp8_quant_1x128_ex)."""
    torch = _torch()
    X = _f32(X, "X")
    K = X.shape[-1]
    M = X.numel() // K if K else 0
    if Q is None:
        Q = torch.empty(X.shape, dtype=torch.uint8, device=X.device)
    if sX is None:
        sX = torch.empty((*X.shape[:-1], _cdiv(K, 128)), dtype=torch.float32, device=X.device)
    Q = _need(_u8_fmt(Q, fmt, "Q"), "Q", M * K, K)
    _need(_f32(sX, "sX"), "sX", M * _cdiv(K, 128), _cdiv(K, 128))
    if sat_count is not None:
        _check(lib().fp8_quant_1x128_ex(_ptr(X, "X"), _ptr(Q, "Q"), _ptr(sX, "sX"), M, K,
                                        _fmt(fmt), _counter(sat_count), _stream(stream)),
               "fp8_quant_1x128_ex")
        return Q, sX
    _check(lib().fp8_quant_1x128_fmt(_ptr(X, "X"), _ptr(Q, "Q"), _ptr(sX, "sX"), M, K, _fmt(fmt),
                                     _stream(stream)), "fp8_quant_1x128_fmt")
    return Q, sX


def fp8_quant_128x128_fmt(W, fmt, Q=None, sW=None, stream=None, sat_count=None):
    """fp8_quant_128x128 with the output format ("e4m3" or "e5m2"); sat_count
    as for fp8_quant_1x128_fmt (fp8_quant_128x128_ex)."""
    torch = _torch()
    W, squeeze, W3 = _weights3(W)
    E, N, K = W3.shape
    shp = (_cdiv(N, 128), _cdiv(K, 128))
    if Q is None:
        Q = torch.empty(W.shape, dtype=torch.uint8, device=W.device)
    if sW is None:
        sW = torch.empty(shp if squeeze else (E, *shp), dtype=torch.float32, device=W.device)
    Qb = _need(_u8_fmt(Q, fmt, "Q"), "Q", E * N * K, K)
    _need(_f32(sW, "sW"), "sW", E * shp[0] * shp[1], shp[1])
    if sat_count is not None:
        _check(lib().fp8_quant_128x128_ex(_ptr(W3, "W"), _ptr(Qb, "Q"), _ptr(sW, "sW"), E, N, K,
                                          _fmt(fmt), _counter(sat_count), _stream(stream)),
               "fp8_quant_128x128_ex")
        return Q, sW
    _check(lib().fp8_quant_128x128_fmt(_ptr(W3, "W"), _ptr(Qb, "Q"), _ptr(sW, "sW"), E, N, K,
                                       _fmt(fmt), _stream(stream)), "fp8_quant_128x128_fmt")
    return Q, sW


def fp8gemm_dense_fmt(A, sA, a_fmt, B, sB, b_fmt, D=None, stream=None):
    """fp8gemm_dense with operand formats ("e4m3" / "e5m2") for A and B."""
    torch = _torch()
    A, B = _u8_fmt(A, a_fmt, "A"), _u8_fmt(B, b_fmt, "B")
    M, N, K = _dense_mnk(A, B)
    if D is None:
        D = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _shape_dense(A, _f32(sA, "sA"), B, _f32(sB, "sB"), D, M, N, K)
    _check(lib().fp8gemm_dense_fmt(_ptr(A, "A"), _ptr(sA, "sA"), _fmt(a_fmt), _ptr(B, "B"),
                                   _ptr(sB, "sB"), _fmt(b_fmt), _ptr(D, "D"), M, N, K,
                                   _stream(stream)), "fp8gemm_dense_fmt")
    return D


def fp8gemm_dense_ex(A, sA, a_fmt, B, sB, b_fmt, D=None, flags=0, stream=None):
    """fp8gemm_dense_fmt with flags, e.g. FLAG_B_READ_ONLY: B and sB are not
    written by any kernel still running when this one starts (constant
    weights), so the decode path may stage them before its dependency wait."""
    torch = _torch()
    A, B = _u8_fmt(A, a_fmt, "A"), _u8_fmt(B, b_fmt, "B")
    M, N, K = _dense_mnk(A, B)
    if D is None:
        D = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _shape_dense(A, _f32(sA, "sA"), B, _f32(sB, "sB"), D, M, N, K)
    _check(lib().fp8gemm_dense_ex(_ptr(A, "A"), _ptr(sA, "sA"), _fmt(a_fmt), _ptr(B, "B"),
                                  _ptr(sB, "sB"), _fmt(b_fmt), _ptr(D, "D"), M, N, K,
                                  int(flags), _stream(stream)), "fp8gemm_dense_ex")
    return D


def fp8gemm_dense_quant_a(X, B, sB, D=None, Q=None, sA=None, stream=None, flags=0):
    """X f32 [M, K], B u8 [N, K], sB [ceil(N/128), K/128] -> D bf16 [M, N], with A
    quantised 1x128 on load.  Q u8 [M, K] and sA f32 [M, K/128] (both or neither)
    receive the quantised activations.  flags (e.g. FLAG_B_READ_ONLY) go to
    fp8gemm_dense_quant_a_ex."""
    torch = _torch()
    X, B = _f32(X, "X"), _u8(B, "B")
    M, N, K = _dense_mnk(X, B, "X")
    if D is None:
        D = torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    if (Q is None) != (sA is None):
        raise ValueError("Q and sA go together: give both or neither")
    Kb = _cdiv(K, 128)
    if B.shape[1] != K:
        raise ValueError(f"B has shape {tuple(B.shape)}; the call needs [N, {K}]")
    _need(_f32(sB, "sB"), "sB", _cdiv(N, 128) * Kb, Kb)
    _need(_bf16(D, "D"), "D", M * N, N)
    if Q is not None:
        _need(_u8(Q, "Q"), "Q", M * K, K)
        _need(_f32(sA, "sA"), "sA", M * Kb, Kb)
    qp = _ptr(_u8(Q, "Q"), "Q") if Q is not None else None
    sp = _ptr(sA, "sA") if sA is not None else None
    if flags:
        rc = lib().fp8gemm_dense_quant_a_ex(_ptr(X, "X"), qp, sp, _ptr(B, "B"), _ptr(sB, "sB"),
                                            _ptr(D, "D"), M, N, K, int(flags), _stream(stream))
    else:
        rc = lib().fp8gemm_dense_quant_a(_ptr(X, "X"), qp, sp, _ptr(B, "B"), _ptr(sB, "sB"),
                                         _ptr(D, "D"), M, N, K, _stream(stream))
    _check(rc, "fp8gemm_dense_quant_a_ex" if flags else "fp8gemm_dense_quant_a")
    return D


class Problem(ctypes.Structure):
    """One entry of the fp8gemm_grouped_table problem table (C layout)."""
    _fields_ = [("A", _P), ("sA", _P), ("B", _P), ("sB", _P), ("D", _P),
                ("M", ctypes.c_int), ("N", ctypes.c_int), ("K", ctypes.c_int),
                ("formats", ctypes.c_int)]


def problem_table(problems, out=None):
    """Device table for fp8gemm_grouped_table from (A, sA, B, sB, D) tensor
    tuples, optionally extended by the operand formats, (A, sA, B, sB, D,
    a_fmt, b_fmt) with "e4m3" / "e5m2": a uint8 CUDA tensor of
    len(problems) * sizeof(Problem) bytes (written into `out` when given, e.g.
    to update a table a graph captured).  Every entry's tensors are checked
    against its (M, N, K) here, since the kernel only sees the pointers."""
    torch = _torch()
    arr = (Problem * len(problems))()
    for e, prob in zip(arr, problems):
        A, sA, B, sB, D = prob[:5]
        a_fmt, b_fmt = (prob[5], prob[6]) if len(prob) > 5 else ("e4m3", "e4m3")
        A, B = _u8_fmt(A, a_fmt, "A"), _u8_fmt(B, b_fmt, "B")
        M, N, K = _dense_mnk(A, B)
        _shape_dense(A, _f32(sA, "sA"), B, _f32(sB, "sB"), D, M, N, K)
        e.A, e.sA, e.B = _dev(A, "A").data_ptr(), _dev(sA, "sA").data_ptr(), _dev(B, "B").data_ptr()
        e.sB, e.D = _dev(sB, "sB").data_ptr(), _dev(D, "D").data_ptr()
        e.M, e.N, e.K = M, N, K
        e.formats = _fmt(a_fmt) | (_fmt(b_fmt) << 8)
    host = torch.frombuffer(bytearray(bytes(arr)), dtype=torch.uint8)
    if out is None:
        return host.to("cuda")
    out.copy_(host)
    return out


MAX_DENSE_BATCH = 32  # FP8GEMM_MAX_DENSE_BATCH


def fp8gemm_dense_batch(problems, stream=None):
    """Independent dense problems in one launch: `problems` is a list of at
    most MAX_DENSE_BATCH tuples (A, sA, B, sB) or (A, sA, B, sB, D), optionally
    followed by (a_fmt, b_fmt); returns the list of D (bf16 [M, N], allocated
    where not given).  The entries are read on the host during the call."""
    torch = _torch()
    if len(problems) > MAX_DENSE_BATCH:
        raise ValueError(f"{len(problems)} problems; one call takes at most {MAX_DENSE_BATCH}")
    arr = (Problem * max(len(problems), 1))()
    outs = []
    for e, prob in zip(arr, problems):
        A, sA, B, sB = prob[:4]
        D = prob[4] if len(prob) in (5, 7) else None
        fmts = prob[-2:] if len(prob) in (6, 7) else ("e4m3", "e4m3")
        A, B = _u8_fmt(A, fmts[0], "A"), _u8_fmt(B, fmts[1], "B")
        M, N, K = _dense_mnk(A, B)
        if D is None:
            D = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
        _shape_dense(A, _f32(sA, "sA"), B, _f32(sB, "sB"), D, M, N, K)
        e.A, e.sA, e.B = _ptr(A, "A").value, _ptr(sA, "sA").value, _ptr(B, "B").value
        e.sB, e.D = _ptr(sB, "sB").value, _ptr(D, "D").value
        e.M, e.N, e.K = M, N, K
        e.formats = _fmt(fmts[0]) | (_fmt(fmts[1]) << 8)
        outs.append(D)
    _check(lib().fp8gemm_dense_batch(ctypes.cast(arr, _P), len(problems), _stream(stream)),
           "fp8gemm_dense_batch")
    return outs


def fp8gemm_grouped_table(table, num_problems, max_M, stream=None):
    """Run every problem of a device table (see problem_table); max_M bounds
    every entry's M and picks the kernel's padded width (16, 32 or 64 rows;
    larger entries are taken 64 rows at a time)."""
    if table.numel() < int(num_problems) * ctypes.sizeof(Problem):
        raise ValueError(f"table holds {table.numel()} bytes; {num_problems} entries need "
                         f"{int(num_problems) * ctypes.sizeof(Problem)}")
    _check(lib().fp8gemm_grouped_table(_ptr(table, "table"), int(num_problems), int(max_M),
                                       _stream(stream)), "fp8gemm_grouped_table")


def _shape_grouped(A, sA, B, sB, info, D, rows, N, K, E, info_len, a_name="A"):
    """Operand sizes of the grouped forms: A holds `rows` rows of K bytes,
    sA [rows, ceil(K/128)], B [E, N, K], sB [E, ceil(N/128), ceil(K/128)],
    the index array `info_len` int32 entries, D bf16 [rows, N]."""
    Kb = _cdiv(K, 128)
    _need(A, a_name, rows * K, K)
    _need(sA, "sA", rows * Kb, Kb)
    if B.dim() != 3 or B.shape[0] != E or B.shape[2] != K:
        raise ValueError(f"B has shape {tuple(B.shape)}; the call needs [{E}, N, {K}]")
    _need(sB, "sB", E * _cdiv(N, 128) * Kb, Kb)
    _need(info, "the index array", info_len)
    _need(_bf16(D, "D"), "D", rows * N, N)


def _contiguous(A, sA, B, sB, m_indices, D, a_fmt, b_fmt, stream, fmt_call):
    torch = _torch()
    if A.dim() != 2 or B.dim() != 3:
        raise ValueError(f"A {tuple(A.shape)} / B {tuple(B.shape)}: the call needs A [M_pad, K]"
                         " and B [E, N, K]")
    M_pad, K = A.shape
    E, N = B.shape[0], B.shape[1]
    if D is None:
        D = torch.empty((M_pad, N), dtype=torch.bfloat16, device=A.device)
    _shape_grouped(A, _f32(sA, "sA"), B, _f32(sB, "sB"), _i32(m_indices, "m_indices"), D,
                   M_pad, N, K, E, M_pad)
    if fmt_call:
        rc = lib().fp8gemm_grouped_contiguous_fmt(
            _ptr(A, "A"), _ptr(sA, "sA"), _fmt(a_fmt), _ptr(B, "B"), _ptr(sB, "sB"),
            _fmt(b_fmt), _ptr(m_indices, "m_indices"), _ptr(D, "D"), M_pad, N, K, E,
            _stream(stream))
    else:
        rc = lib().fp8gemm_grouped_contiguous(
            _ptr(A, "A"), _ptr(sA, "sA"), _ptr(B, "B"), _ptr(sB, "sB"),
            _ptr(m_indices, "m_indices"), _ptr(D, "D"), M_pad, N, K, E, _stream(stream))
    _check(rc, "fp8gemm_grouped_contiguous" + ("_fmt" if fmt_call else ""))
    return D


def _masked(A, sA, B, sB, masked_m, D, a_fmt, b_fmt, stream, fmt_call):
    torch = _torch()
    if A.dim() != 3 or B.dim() != 3:
        raise ValueError(f"A {tuple(A.shape)} / B {tuple(B.shape)}: the call needs A "
                         "[E, M_max, K] and B [E, N, K]")
    E, M_max, K = A.shape
    N = B.shape[1]
    if D is None:
        D = torch.empty((E, M_max, N), dtype=torch.bfloat16, device=A.device)
    _shape_grouped(A, _f32(sA, "sA"), B, _f32(sB, "sB"), _i32(masked_m, "masked_m"), D,
                   E * M_max, N, K, E, E)
    if fmt_call:
        rc = lib().fp8gemm_grouped_masked_fmt(
            _ptr(A, "A"), _ptr(sA, "sA"), _fmt(a_fmt), _ptr(B, "B"), _ptr(sB, "sB"),
            _fmt(b_fmt), _ptr(masked_m, "masked_m"), _ptr(D, "D"), E, M_max, N, K,
            _stream(stream))
    else:
        rc = lib().fp8gemm_grouped_masked(
            _ptr(A, "A"), _ptr(sA, "sA"), _ptr(B, "B"), _ptr(sB, "sB"),
            _ptr(masked_m, "masked_m"), _ptr(D, "D"), E, M_max, N, K, _stream(stream))
    _check(rc, "fp8gemm_grouped_masked" + ("_fmt" if fmt_call else ""))
    return D


def fp8gemm_grouped_contiguous(A, sA, B, sB, m_indices, D=None, stream=None):
    """A u8 [M_pad, K], B u8 [E, N, K], m_indices i32 [M_pad] -> D bf16 [M_pad, N]."""
    return _contiguous(_u8(A, "A"), sA, _u8(B, "B"), sB, m_indices, D, "e4m3", "e4m3", stream,
                       False)


def fp8gemm_grouped_masked(A, sA, B, sB, masked_m, D=None, stream=None):
    """A u8 [E, M_max, K], B u8 [E, N, K], masked_m i32 [E] -> D bf16 [E, M_max, N]
    (rows >= masked_m[e] are not written)."""
    return _masked(_u8(A, "A"), sA, _u8(B, "B"), sB, masked_m, D, "e4m3", "e4m3", stream, False)


def fp8gemm_grouped_contiguous_fmt(A, sA, a_fmt, B, sB, b_fmt, m_indices, D=None, stream=None):
    """fp8gemm_grouped_contiguous with operand formats ("e4m3" / "e5m2")."""
    return _contiguous(_u8_fmt(A, a_fmt, "A"), sA, _u8_fmt(B, b_fmt, "B"), sB, m_indices, D,
                       a_fmt, b_fmt, stream, True)


def fp8gemm_grouped_masked_fmt(A, sA, a_fmt, B, sB, b_fmt, masked_m, D=None, stream=None):
    """fp8gemm_grouped_masked with operand formats ("e4m3" / "e5m2")."""
    return _masked(_u8_fmt(A, a_fmt, "A"), sA, _u8_fmt(B, b_fmt, "B"), sB, masked_m, D,
                   a_fmt, b_fmt, stream, True)


def fp8gemm_dense_small_m_noalloc(A, sA, B, sB, D, stream=None):
    """fp8gemm_dense for M <= 64 without any device allocation by the library:
    the caller provides D, and the split-K scratch is a fixed array inside the
    library (shared by every call on the device; calls must not overlap on the
    GPU)."""
    A, B = _u8(A, "A"), _u8(B, "B")
    M, N, K = _dense_mnk(A, B)
    _shape_dense(A, _f32(sA, "sA"), B, _f32(sB, "sB"), D, M, N, K)
    _check(lib().fp8gemm_dense_small_m_noalloc(
        _ptr(A, "A"), _ptr(sA, "sA"), _ptr(B, "B"), _ptr(sB, "sB"), _ptr(D, "D"),
        M, N, K, _stream(stream)), "fp8gemm_dense_small_m_noalloc")
    return D


def fp8gemm_get_device_status(stream=None) -> int:
    """Synchronise the stream, then read and clear the device status word."""
    out = ctypes.c_int(0)
    _check(lib().fp8gemm_get_device_status(_stream(stream), ctypes.byref(out)),
           "fp8gemm_get_device_status")
    return out.value


def fp8gemm_release_workspaces(stream=None):
    """Free the library's workspaces of `stream` (current stream by default)
    on the current device, after synchronising it."""
    _check(lib().fp8gemm_release_workspaces(_stream(stream)), "fp8gemm_release_workspaces")


def workspace_bytes() -> int:
    """Bytes of library-owned workspaces currently held (all devices, streams)."""
    return int(lib().fp8gemm_workspace_bytes())


def set_wait_limit_ns(ns: int):
    """Time limit of every pipeline wait in kernels launched from now on
    (process-wide); 0 restores the default (2 s)."""
    _check(lib().fp8gemm_set_wait_limit_ns(int(ns)), "fp8gemm_set_wait_limit_ns")
