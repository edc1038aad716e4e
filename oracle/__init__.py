"""CPU oracle for single-precision GEMM -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
(and its ``--impl reference`` arm) may import this package.  The CUDA library
and its Python binding never import it, and it imports nothing from them.

The arithmetic lives in ``sgemm_oracle.c`` (plain C, double accumulation, no
blocking); this module compiles it with gcc, calls it through ctypes, and holds
the acceptance check.

Acceptance (normalised error), per output entry::

    err = |C_out - Cref| / den,   den = sum_p |alpha*opA[i,p]*opB[p,j]| + |beta*Cin[i,j]|

An optional absolute ``floor`` loosens this to |C_out - Cref| <= tol*den + floor.
FP32 with gradual underflow rounds a result below the normal range (2^-126) to
a multiple of 2^-149, so each operation may add an absolute error of up to
2^-149 that no relative bound covers; an output whose products underflow needs
floor = (number of roundings) * 2^-149, e.g. (k + 2) * 2^-149 for a dot product
of k terms followed by the alpha/beta update.  The floor is 0 unless a test
passes one (it matters only where den is below about k * 2^-130).

The pages state no tolerance ("V3. Vectorized and double buffer", section 3,
prints only a max_abs_err and PASS); the bounds used by the tests are 1e-5 for
the exact-FP32 and split-TF32 modes and 5e-3 for plain TF32.  Extra rules:
an output that is NaN or Inf where Cref is finite fails; where den == 0 the
output must equal Cref exactly (either signed zero is accepted).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sgemm_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", "-std=c11"]


def build(force: bool = False) -> str:
    """Compile the oracle library in place (gcc, OpenMP); returns its path."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + ".tmp%d" % os.getpid()
    subprocess.run(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, _LIB)
    return _LIB


def build_from(src: str, out: str) -> str:
    """Compile another copy of the oracle source (the mutation tests use this)."""
    subprocess.run(["gcc", *CFLAGS, src, "-o", out, "-lm"], check=True)
    return out


def _bind(lib):
    f32p = ctypes.POINTER(ctypes.c_float)
    f64p = ctypes.POINTER(ctypes.c_double)
    i64p = ctypes.POINTER(ctypes.c_int64)
    c, i64, f = ctypes.c_char, ctypes.c_int64, ctypes.c_float
    common = [c, c, i64, i64, i64, f, f32p, i64, f32p, i64, f, f32p, i64]
    lib.oracle_sgemm_full.argtypes = common + [f64p, f64p, ctypes.c_int]
    lib.oracle_sgemm_full.restype = ctypes.c_int
    lib.oracle_sgemm_entries.argtypes = common + [i64, i64p, i64p, f64p, f64p, ctypes.c_int]
    lib.oracle_sgemm_entries.restype = ctypes.c_int
    lib.oracle_sgemm_ikj.argtypes = common + [f64p]
    lib.oracle_sgemm_ikj.restype = ctypes.c_int
    lib.oracle_max_threads.argtypes = []
    lib.oracle_max_threads.restype = ctypes.c_int
    return lib


def load(path: str | None = None):
    """The ctypes handle (building the default library on first use)."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
        return _lib


def _f32(x) -> np.ndarray:
    if hasattr(x, "detach"):  # a CPU torch tensor
        x = x.detach().cpu().numpy()
    a = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    return a


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _empty_if_none(a):
    return np.zeros(1, np.float32) if a is None else _f32(a)


class Oracle:
    """Thin caller around one loaded oracle library (the default, or a mutant)."""

    def __init__(self, lib=None):
        self.lib = lib if lib is not None else load()

    def max_threads(self) -> int:
        return int(self.lib.oracle_max_threads())

    def full(self, transa, transb, m, n, k, alpha, A, lda, B, ldb, beta, C, ldc,
             threads: int = 0):
        """(Cref, den), each an (m, n) float64 array (Fortran order)."""
        A, B, C = _empty_if_none(A), _empty_if_none(B), _empty_if_none(C)
        cref = np.zeros(max(m * n, 1), np.float64)
        den = np.zeros(max(m * n, 1), np.float64)
        rc = self.lib.oracle_sgemm_full(
            transa.encode(), transb.encode(), m, n, k, float(alpha),
            _ptr(A, ctypes.c_float), lda, _ptr(B, ctypes.c_float), ldb, float(beta),
            _ptr(C, ctypes.c_float), ldc, _ptr(cref, ctypes.c_double),
            _ptr(den, ctypes.c_double), int(threads))
        if rc != 0:
            raise ValueError("oracle_sgemm_full rejected its arguments (%d)" % rc)
        shape = (m, n)
        return (cref[: m * n].reshape(shape, order="F"),
                den[: m * n].reshape(shape, order="F"))

    def entries(self, transa, transb, m, n, k, alpha, A, lda, B, ldb, beta, C, ldc,
                ii, jj, threads: int = 0):
        """(Cref, den) at the listed (ii[e], jj[e]) entries, each a 1-D float64 array."""
        A, B, C = _empty_if_none(A), _empty_if_none(B), _empty_if_none(C)
        ii = np.ascontiguousarray(ii, dtype=np.int64)
        jj = np.ascontiguousarray(jj, dtype=np.int64)
        cnt = ii.size
        cref = np.zeros(max(cnt, 1), np.float64)
        den = np.zeros(max(cnt, 1), np.float64)
        rc = self.lib.oracle_sgemm_entries(
            transa.encode(), transb.encode(), m, n, k, float(alpha),
            _ptr(A, ctypes.c_float), lda, _ptr(B, ctypes.c_float), ldb, float(beta),
            _ptr(C, ctypes.c_float), ldc, cnt, _ptr(ii, ctypes.c_int64),
            _ptr(jj, ctypes.c_int64), _ptr(cref, ctypes.c_double),
            _ptr(den, ctypes.c_double), int(threads))
        if rc != 0:
            raise ValueError("oracle_sgemm_entries rejected its arguments (%d)" % rc)
        return cref[:cnt], den[:cnt]

    def ikj(self, transa, transb, m, n, k, alpha, A, lda, B, ldb, beta, C, ldc):
        A, B, C = _empty_if_none(A), _empty_if_none(B), _empty_if_none(C)
        cref = np.zeros(max(m * n, 1), np.float64)
        rc = self.lib.oracle_sgemm_ikj(
            transa.encode(), transb.encode(), m, n, k, float(alpha),
            _ptr(A, ctypes.c_float), lda, _ptr(B, ctypes.c_float), ldb, float(beta),
            _ptr(C, ctypes.c_float), ldc, _ptr(cref, ctypes.c_double))
        if rc != 0:
            raise ValueError("oracle_sgemm_ikj rejected its arguments (%d)" % rc)
        return cref[: m * n].reshape((m, n), order="F")


def full(*args, **kw):
    return Oracle().full(*args, **kw)


def entries(*args, **kw):
    return Oracle().entries(*args, **kw)


def ikj(*args, **kw):
    return Oracle().ikj(*args, **kw)


def max_threads() -> int:
    return Oracle().max_threads()


# Tolerances on the normalised error, per mode name.
TOL = {"ffma": 1e-5, "3xtf32": 1e-5, "tf32": 5e-3}


def normalised_error(out, cref, den, floor: float = 0.0):
    """Per-entry normalised error (see the module docstring); with floor > 0 the
    absolute error is first reduced by floor (an error within the floor counts 0)."""
    out = np.asarray(out, dtype=np.float64)
    cref = np.asarray(cref, dtype=np.float64)
    den = np.asarray(den, dtype=np.float64)
    finite_ref = np.isfinite(cref)
    with np.errstate(divide="ignore", invalid="ignore"):
        diff = np.abs(out - cref)
        if floor > 0:
            diff = np.maximum(diff - floor, 0.0)
        err = np.where(den > 0, diff / np.where(den > 0, den, 1.0), np.where(diff == 0, 0.0, np.inf))
    bad_nonfinite = finite_ref & ~np.isfinite(out)
    err = np.where(bad_nonfinite, np.inf, err)
    # A non-finite reference (overflow or NaN inputs) must be matched in kind.
    nonfinite_ref = ~finite_ref
    same_kind = (np.isnan(cref) & np.isnan(out)) | (np.isinf(cref) & (cref == out))
    err = np.where(nonfinite_ref, np.where(same_kind, 0.0, np.inf), err)
    return err


def check(out, cref, den, tol: float, floor: float = 0.0) -> dict:
    """Summary dict: max normalised error, count above tol, max abs error, ok flag."""
    err = normalised_error(out, cref, den, floor)
    out64 = np.asarray(out, dtype=np.float64)
    with np.errstate(invalid="ignore"):
        abs_err = np.abs(out64 - np.asarray(cref, dtype=np.float64))
    n_bad = int(np.count_nonzero(~(err <= tol)))
    finite = np.isfinite(abs_err)
    return {
        "max_err": float(np.max(err)) if err.size else 0.0,
        "n_bad": n_bad,
        "n": int(err.size),
        "max_abs_err": float(np.max(abs_err[finite])) if finite.any() else 0.0,
        "tol": tol,
        "ok": n_bad == 0,
    }
