"""GB300-native single-precision GEMM: Python binding of the C ABI.

The names mirror ``include/precision_gemm.h``; every function only marshals
arguments (tensors or integers to device pointers, streams to handles) and
calls the shared library ``libprecision_gemm.so`` built in this directory.
All arithmetic runs in the library's CUDA kernels.  There is no fallback: if
the library has not been built, or a call fails, an exception is raised.

    sgemm(transa, transb, m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, mode, stream)

A, B, C are device pointers (ints) or CUDA torch tensors (their storage is
addressed through ``data_ptr()``); mode is 'ffma', 'tf32', '3xtf32' or the
integer SGEMM_* constant; stream is a torch.cuda.Stream, a raw handle, or None
for torch's current stream.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libprecision_gemm.so")

SGEMM_FFMA, SGEMM_TF32, SGEMM_3XTF32 = 0, 1, 2
MODES = {"ffma": SGEMM_FFMA, "tf32": SGEMM_TF32, "3xtf32": SGEMM_3XTF32}
MODE_NAMES = {v: k for k, v in MODES.items()}

SGEMM_ERR = {1: "SGEMM_ERR_CUDA", 2: "SGEMM_ERR_NO_DEVICE", 3: "SGEMM_ERR_ARCH", 4: "SGEMM_ERR_TIMEOUT",
             5: "SGEMM_ERR_ALLOC", 6: "SGEMM_ERR_TENSOR_MAP", 7: "SGEMM_ERR_CAPTURE", 8: "SGEMM_ERR_SCRATCH"}
SGEMM_ERR_SCRATCH = 8
SGEMM_ERR_TIMEOUT = 4
SGEMM_DEBUG_STALL_PRODUCER = 1
KERNELS = {0: "none", 1: "scale", 2: "ffma", 3: "tc", 4: "tc2"}
PREPS = {0: "none", 1: "copy", 2: "transpose", 3: "split"}

# Every symbol the header declares (checked by the CPU tests).
EXPORTS = ("sgemm", "sgemm_host", "sgemm_host_async", "sgemm_noalloc", "sgemm_plan", "sgemm_device_status",
           "sgemm_set_wait_timeout", "sgemm_force_plan", "sgemm_debug_flags", "sgemm_launch_count",
           "sgemm_workspace_release", "sgemm_last_error_string", "sgemm_version")


class SgemmError(RuntimeError):
    """A nonzero status from the library; .code is the status."""

    def __init__(self, code: int, message: str):
        super().__init__("%s (%d): %s" % (SGEMM_ERR.get(code, "invalid argument" if code < 0 else "error"),
                                          code, message))
        self.code = code


class sgemm_plan_t(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int) for name in (
        "kernel", "mode", "bm", "bn", "bk", "stages", "split_k", "k_blocks", "k_blocks_per_split",
        "tiles_m", "tiles_n", "prep_a", "prep_b", "threads", "ctas_per_sm")] + [
        ("ld_a", ctypes.c_int64), ("ld_b", ctypes.c_int64), ("smem_bytes", ctypes.c_size_t),
        ("workspace_bytes", ctypes.c_size_t), ("launches", ctypes.c_int), ("tail_tiles", ctypes.c_int),
        ("tail_split", ctypes.c_int)]


_lib = None
_lock = threading.Lock()


def load_library(path: str | None = None):
    """Load (once) and return the ctypes handle; raises if the library is missing."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError("the CUDA library %s is not built; run `python -c \"import __graft_entry__ as g; "
                               "g.build()\"` (or precision_gemm_gb300/build.py)" % p)
        lib = ctypes.CDLL(p)
        c, i64, f, vp, i = ctypes.c_char, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_int
        gemm_args = [c, c, i64, i64, i64, f, vp, i64, vp, i64, f, vp, i64, i, vp]
        lib.sgemm.argtypes = gemm_args
        lib.sgemm.restype = i
        lib.sgemm_host.argtypes = gemm_args
        lib.sgemm_host.restype = i
        lib.sgemm_host_async.argtypes = gemm_args
        lib.sgemm_host_async.restype = i
        lib.sgemm_noalloc.argtypes = gemm_args
        lib.sgemm_noalloc.restype = i
        lib.sgemm_plan.argtypes = gemm_args[:14] + [i, ctypes.POINTER(sgemm_plan_t)]
        lib.sgemm_plan.restype = i
        lib.sgemm_device_status.argtypes = [vp, i]
        lib.sgemm_device_status.restype = i
        lib.sgemm_set_wait_timeout.argtypes = [ctypes.c_uint64]
        lib.sgemm_set_wait_timeout.restype = ctypes.c_uint64
        lib.sgemm_force_plan.argtypes = [i, i]
        lib.sgemm_force_plan.restype = i
        lib.sgemm_debug_flags.argtypes = [i]
        lib.sgemm_debug_flags.restype = i
        lib.sgemm_launch_count.argtypes = []
        lib.sgemm_launch_count.restype = ctypes.c_uint64
        lib.sgemm_workspace_release.argtypes = []
        lib.sgemm_workspace_release.restype = i
        lib.sgemm_last_error_string.argtypes = []
        lib.sgemm_last_error_string.restype = ctypes.c_char_p
        lib.sgemm_version.argtypes = []
        lib.sgemm_version.restype = ctypes.c_char_p
        if path is None:
            _lib = lib
        return lib


def _ptr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return int(x.data_ptr())
    if hasattr(x, "ctypes"):  # numpy array (host pointer for sgemm_host)
        return int(x.ctypes.data)
    raise TypeError("cannot take a pointer from %r" % type(x))


def _stream(s) -> int:
    if s is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream) if torch.cuda.is_available() else 0
    if isinstance(s, int):
        return s
    if hasattr(s, "cuda_stream"):
        return int(s.cuda_stream)
    raise TypeError("cannot take a stream handle from %r" % type(s))


def _mode(mode) -> int:
    return MODES[mode.lower()] if isinstance(mode, str) else int(mode)


def _check(rc: int, lib) -> None:
    if rc != 0:
        raise SgemmError(rc, lib.sgemm_last_error_string().decode(errors="replace"))


def _tchar(t: str) -> bytes:
    return t.encode() if isinstance(t, str) else bytes(t)


def sgemm(transa, transb, m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, mode="ffma", stream=None) -> None:
    """C = alpha*op(A)*op(B) + beta*C on device memory (column-major); asynchronous."""
    lib = load_library()
    _check(lib.sgemm(_tchar(transa), _tchar(transb), m, n, k, alpha, _ptr(A), lda, _ptr(B), ldb, beta,
                     _ptr(C), ldc, _mode(mode), _stream(stream)), lib)


def sgemm_host(transa, transb, m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, mode="ffma", stream=None) -> None:
    """The same on host arrays (pinned tensors / numpy); returns when C holds the result."""
    lib = load_library()
    _check(lib.sgemm_host(_tchar(transa), _tchar(transb), m, n, k, alpha, _ptr(A), lda, _ptr(B), ldb, beta,
                          _ptr(C), ldc, _mode(mode), _stream(stream)), lib)


def sgemm_host_async(transa, transb, m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, mode="ffma",
                     stream=None) -> None:
    """sgemm_host queued on `stream` without waiting: C holds the result once the
    stream is synchronised; until then A, B and C must stay untouched (and alive)."""
    lib = load_library()
    _check(lib.sgemm_host_async(_tchar(transa), _tchar(transb), m, n, k, alpha, _ptr(A), lda, _ptr(B), ldb, beta,
                                _ptr(C), ldc, _mode(mode), _stream(stream)), lib)


def sgemm_noalloc(transa, transb, m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, mode="ffma",
                  stream=None) -> None:
    """sgemm for callers that cannot allocate device memory: never calls cudaMalloc;
    its split-K scratch is a fixed 16 MiB device array shared by every call (calls
    that overlap on the GPU race on it).  FFMA or TF32, untransposed 16-byte
    aligned operands with ld multiples of 4; raises SgemmError (code
    SGEMM_ERR_SCRATCH) when the call's partial sums would not fit."""
    lib = load_library()
    _check(lib.sgemm_noalloc(_tchar(transa), _tchar(transb), m, n, k, alpha, _ptr(A), lda, _ptr(B), ldb, beta,
                             _ptr(C), ldc, _mode(mode), _stream(stream)), lib)


def sgemm_rm(m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, mode="ffma", stream=None) -> None:
    """Row-major C (m x n, row stride ldc) = alpha*A*B + beta*C with row-major A (m x k,
    row stride lda) and B (k x n, row stride ldb).  A row-major buffer is the
    column-major storage of the transpose, so this is the column-major call
    C^T = B^T * A^T: operands swapped, m and n swapped."""
    sgemm("N", "N", n, m, k, alpha, B, ldb, A, lda, beta, C, ldc, mode, stream)


def sgemm_plan(transa, transb, m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, mode="ffma",
               num_sms: int = 152) -> dict:
    """What sgemm would launch (no device needed); pointers only matter for alignment."""
    lib = load_library()
    pl = sgemm_plan_t()
    _check(lib.sgemm_plan(_tchar(transa), _tchar(transb), m, n, k, alpha, _ptr(A), lda, _ptr(B), ldb, beta,
                          _ptr(C), ldc, _mode(mode), num_sms, ctypes.byref(pl)), lib)
    d = {name: getattr(pl, name) for name, _ in sgemm_plan_t._fields_}
    d["kernel_name"] = KERNELS.get(d["kernel"], "?")
    d["prep_a_name"] = PREPS.get(d["prep_a"], "?")
    d["prep_b_name"] = PREPS.get(d["prep_b"], "?")
    return d


def device_status(stream=None, clear: bool = True) -> int:
    """Synchronise the stream; 0, or SGEMM_ERR_TIMEOUT if a kernel's bounded wait expired."""
    lib = load_library()
    return int(lib.sgemm_device_status(_stream(stream), 1 if clear else 0))


def set_wait_timeout(ns: int) -> int:
    return int(load_library().sgemm_set_wait_timeout(int(ns)))


def force_plan(bn: int = 0, split_k: int = 0) -> None:
    lib = load_library()
    _check(lib.sgemm_force_plan(int(bn), int(split_k)), lib)


def debug_flags(flags: int) -> int:
    return int(load_library().sgemm_debug_flags(int(flags)))


def launch_count() -> int:
    return int(load_library().sgemm_launch_count())


def workspace_release() -> None:
    lib = load_library()
    _check(lib.sgemm_workspace_release(), lib)


def last_error() -> str:
    return load_library().sgemm_last_error_string().decode(errors="replace")


def version() -> str:
    return load_library().sgemm_version().decode()


def matmul(A, B, mode="ffma", out=None, alpha: float = 1.0, beta: float = 0.0, stream=None):
    """out = alpha * A @ B + beta * out for 2-D CUDA float32 torch tensors whose
    last dimension is contiguous (row-major with a row stride); returns out."""
    import torch
    m, k = A.shape
    k2, n = B.shape
    if k2 != k:
        raise ValueError("inner dimensions differ: %d vs %d" % (k, k2))
    for name, t in (("A", A), ("B", B)):
        if t.dtype != torch.float32 or not t.is_cuda or (t.shape[1] > 1 and t.stride(1) != 1):
            raise ValueError("%s must be a CUDA float32 tensor with unit column stride" % name)
    if out is None:
        out = torch.empty((m, n), dtype=torch.float32, device=A.device)
        beta = 0.0
    sgemm_rm(m, n, k, alpha, A, max(A.stride(0), k, 1), B, max(B.stride(0), n, 1), beta, out,
             max(out.stride(0), n, 1), mode, stream)
    return out
