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

Tensor operands are checked before the library is called, for every operand
the call reads or writes: float32, on the current CUDA device (host memory for
the sgemm_host entries), and a storage that holds the operand's whole extent
(ld * (cols - 1) + rows elements from the tensor's first element).  A failed
check raises ValueError.  Integer addresses are passed on unchecked.
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
             5: "SGEMM_ERR_ALLOC", 6: "SGEMM_ERR_TENSOR_MAP", 7: "SGEMM_ERR_CAPTURE", 8: "SGEMM_ERR_SCRATCH",
             9: "SGEMM_ERR_WORKSPACE"}
SGEMM_ERR_CAPTURE = 7
SGEMM_ERR_SCRATCH = 8
SGEMM_ERR_WORKSPACE = 9
SGEMM_ERR_TIMEOUT = 4
SGEMM_DEBUG_STALL_PRODUCER = 1
SGEMM_DEBUG_FAIL_ALLOC = 2
SGEMM_DEBUG_FAIL_TENSOR_MAP = 4
SGEMM_ERR_ALLOC = 5
SGEMM_ERR_TENSOR_MAP = 6
KERNELS = {0: "none", 1: "scale", 2: "ffma", 3: "tc", 4: "tc2"}
PREPS = {0: "none", 1: "copy", 2: "transpose", 3: "split"}

# Every symbol the header declares (checked by the CPU tests).
EXPORTS = ("sgemm", "sgemm_host", "sgemm_host_async", "sgemm_set_host_split", "sgemm_host_split_ratio",
           "sgemm_noalloc", "sgemm_set_workspace", "sgemm_plan", "sgemm_device_status",
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
        ("tail_split", ctypes.c_int), ("sk_ctas", ctypes.c_int)]


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
        lib.sgemm_set_host_split.argtypes = [ctypes.c_double]
        lib.sgemm_set_host_split.restype = i
        lib.sgemm_host_split_ratio.argtypes = [i]
        lib.sgemm_host_split_ratio.restype = ctypes.c_double
        lib.sgemm_set_workspace.argtypes = [vp, ctypes.c_size_t, vp]
        lib.sgemm_set_workspace.restype = i
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


_torch = None


def _torch_mod():
    global _torch
    if _torch is None:
        import torch
        _torch = torch
    return _torch


def _check_operand(x, name: str, rows: int, cols: int, ld: int, on_device: bool, cur_dev=None) -> None:
    """Raise ValueError unless tensor / array x can serve as a rows x cols operand
    with leading dimension ld: float32, in device memory of the current CUDA
    device (on_device; cur_dev is that device's index when the caller has it) or
    in host memory (not on_device), with storage for the whole extent.  ints are
    not checked; None is left to the library, which rejects a null pointer the
    call needs."""
    if x is None or isinstance(x, int):
        return
    torch = _torch_mod()
    if isinstance(x, torch.Tensor):
        if x.dtype != torch.float32:
            raise ValueError("%s: expected a float32 tensor, got %s" % (name, x.dtype))
        if on_device:
            if not x.is_cuda:
                raise ValueError("%s: expected a CUDA tensor, got one on %s" % (name, x.device))
            cur = torch.cuda.current_device() if cur_dev is None else cur_dev
            if x.get_device() != cur:
                raise ValueError("%s: the tensor is on %s, the current device is cuda:%d" % (name, x.device, cur))
        elif x.is_cuda:
            raise ValueError("%s: expected a host (CPU) tensor, got one on %s" % (name, x.device))
        avail = (x.untyped_storage().nbytes() - x.storage_offset() * 4) // 4
    elif hasattr(x, "ctypes") and hasattr(x, "dtype"):  # numpy array
        if on_device:
            raise ValueError("%s: a numpy array is host memory; this call takes device memory" % name)
        if str(x.dtype) != "float32":
            raise ValueError("%s: expected a float32 array, got %s" % (name, x.dtype))
        if not (x.flags["C_CONTIGUOUS"] or x.flags["F_CONTIGUOUS"]):
            raise ValueError("%s: the array must be contiguous" % name)
        avail = int(x.size)
    else:
        raise TypeError("%s: cannot take a pointer from %r" % (name, type(x)))
    if ld < max(1, rows):
        return  # the library reports the bad leading dimension as an invalid argument
    need = 0 if rows <= 0 or cols <= 0 else ld * (cols - 1) + rows  # the last column needs only its rows
    if avail < need:
        raise ValueError("%s: a %d x %d operand with leading dimension %d spans %d elements; the storage from the "
                         "tensor's first element holds %d" % (name, rows, cols, ld, need, avail))


def _check_gemm_operands(transa, transb, m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, on_device: bool) -> None:
    """The operand checks of one call: A and B when the product reads them, C when
    the call reads or writes it (the library's own rules for what it touches)."""
    if m <= 0 or n <= 0:
        return
    cur = None
    if on_device and any(getattr(x, "is_cuda", False) for x in (A, B, C)):
        cur = _torch_mod().cuda.current_device()
    reads_ab = k > 0 and alpha != 0.0
    if reads_ab:
        ra, ca = (m, k) if transa in ("N", "n", b"N", b"n") else (k, m)
        rb, cb = (k, n) if transb in ("N", "n", b"N", b"n") else (n, k)
        _check_operand(A, "A", ra, ca, lda, on_device, cur)
        _check_operand(B, "B", rb, cb, ldb, on_device, cur)
    if reads_ab or beta != 1.0:
        _check_operand(C, "C", m, n, ldc, on_device, cur)


def _stream(s) -> int:
    if s is None:
        torch = _torch_mod()
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
    _check_gemm_operands(transa, transb, m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, on_device=True)
    _check(lib.sgemm(_tchar(transa), _tchar(transb), m, n, k, alpha, _ptr(A), lda, _ptr(B), ldb, beta,
                     _ptr(C), ldc, _mode(mode), _stream(stream)), lib)


def sgemm_host(transa, transb, m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, mode="ffma", stream=None) -> None:
    """The same on host arrays (pinned tensors / numpy); returns when C holds the result."""
    lib = load_library()
    _check_gemm_operands(transa, transb, m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, on_device=False)
    _check(lib.sgemm_host(_tchar(transa), _tchar(transb), m, n, k, alpha, _ptr(A), lda, _ptr(B), ldb, beta,
                          _ptr(C), ldc, _mode(mode), _stream(stream)), lib)


def sgemm_host_async(transa, transb, m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, mode="ffma",
                     stream=None) -> None:
    """sgemm_host queued on `stream` without waiting: C holds the result once the
    stream is synchronised; until then A, B and C must stay untouched (and alive)."""
    lib = load_library()
    _check_gemm_operands(transa, transb, m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, on_device=False)
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
    _check_gemm_operands(transa, transb, m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, on_device=True)
    _check(lib.sgemm_noalloc(_tchar(transa), _tchar(transb), m, n, k, alpha, _ptr(A), lda, _ptr(B), ldb, beta,
                             _ptr(C), ldc, _mode(mode), _stream(stream)), lib)


def sgemm_rm(m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, mode="ffma", stream=None) -> None:
    """Row-major C (m x n, row stride ldc) = alpha*A*B + beta*C with row-major A (m x k,
    row stride lda) and B (k x n, row stride ldb).  A row-major buffer is the
    column-major storage of the transpose, so this is the column-major call
    C^T = B^T * A^T: operands swapped, m and n swapped."""
    sgemm("N", "N", n, m, k, alpha, B, ldb, A, lda, beta, C, ldc, mode, stream)


def set_host_split(q: float) -> None:
    """Hybrid CPU + GPU column split of sgemm_host / sgemm_host_async: q > 0 gives
    the last floor(n / (q + 1)) columns of C to the host cores, q < 0 measures q
    call by call (starting at 15), 0 turns the split off (the default)."""
    lib = load_library()
    _check(lib.sgemm_set_host_split(float(q)), lib)


def host_split_ratio(mode="ffma") -> float:
    """The ratio Q the next host call in `mode` would use (0 when the split is off)."""
    return float(load_library().sgemm_host_split_ratio(_mode(mode)))


_ws_refs = {}  # (device, stream handle) -> the tensor given to set_workspace, kept alive here


def set_workspace(buf, nbytes: int | None = None, stream=None) -> None:
    """Give calls on `stream` (torch's current stream when None) on the current
    device a workspace of the caller's own instead of one the library allocates:
    a CUDA tensor (its storage from its first element; 256-byte aligned, as the
    caching allocator gives) or an integer address with nbytes; None returns the
    stream to the library's own workspace.  The tensor is kept alive here until
    it is replaced.  Calls needing more than its size raise SgemmError with code
    SGEMM_ERR_WORKSPACE; sgemm_plan(...)["workspace_bytes"] gives the need."""
    lib = load_library()
    st = _stream(stream)
    if buf is None:
        ptr, size = 0, 0
    elif isinstance(buf, int):
        if nbytes is None:
            raise ValueError("an integer workspace address needs nbytes")
        ptr, size = buf, int(nbytes)
    else:
        import torch
        if not getattr(buf, "is_cuda", False):
            raise ValueError("the workspace must be a CUDA tensor")
        if buf.device.index != torch.cuda.current_device():
            raise ValueError("the workspace is on %s, the current device is cuda:%d"
                             % (buf.device, torch.cuda.current_device()))
        avail = buf.untyped_storage().nbytes() - buf.storage_offset() * buf.element_size()
        size = avail if nbytes is None else int(nbytes)
        if size > avail:
            raise ValueError("nbytes %d exceeds the tensor's storage (%d bytes)" % (size, avail))
        ptr = int(buf.data_ptr())
    _check(lib.sgemm_set_workspace(ptr, size, st), lib)
    import torch
    key = (torch.cuda.current_device() if torch.cuda.is_available() else 0, st)
    if buf is None:
        _ws_refs.pop(key, None)
    else:
        _ws_refs[key] = buf


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
