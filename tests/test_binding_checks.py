"""The Python binding refuses operands it cannot pass safely, before the library
is called: a tensor of the wrong dtype, on the wrong side of the host link, or
with storage too small for the operand's extent (ld * (cols - 1) + rows
elements).  Without these checks such a tensor reaches the kernels as a raw
address.  Every refusal here happens on the host; no test needs a GPU.  (On a
machine without a GPU, a call that passes the checks fails in the library with
SGEMM_ERR_NO_DEVICE, which shows that the binding let it through.)"""
import ctypes

import numpy as np
import pytest
import torch

import precision_gemm_gb300 as pg
from precision_gemm_gb300 import build as pgbuild

NO_GPU = not torch.cuda.is_available()


@pytest.fixture(scope="module", autouse=True)
def lib():
    pgbuild.build()
    return pg.load_library()


def _host_call(entry, m, n, k, A, lda, B, ldb, C, ldc, transa="N", transb="N", alpha=1.0, beta=0.5):
    getattr(pg, entry)(transa, transb, m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, "ffma", stream=0)


def _passes_binding(fn):
    """fn() got past the binding's checks: on this GPU-less machine the library
    then answers SGEMM_ERR_NO_DEVICE."""
    with pytest.raises(pg.SgemmError) as e:
        fn()
    assert e.value.code == 2, e.value


@pytest.mark.skipif(not NO_GPU, reason="relies on the library failing without a device")
@pytest.mark.parametrize("entry", ["sgemm_host", "sgemm_host_async"])
def test_host_entries_check_extent_exactly(entry):
    m, n, k, lda, ldb, ldc = 5, 4, 3, 7, 6, 9
    need_a, need_b, need_c = lda * (k - 1) + m, ldb * (n - 1) + k, ldc * (n - 1) + m
    A, B, C = torch.zeros(need_a), torch.zeros(need_b), torch.zeros(need_c)
    _passes_binding(lambda: _host_call(entry, m, n, k, A, lda, B, ldb, C, ldc))
    for short in ("A", "B", "C"):
        args = dict(A=A, B=B, C=C)
        args[short] = args[short][:-1].clone()  # a fresh storage one element short
        with pytest.raises(ValueError, match="^%s: .*spans %d elements" % (short, dict(A=need_a, B=need_b,
                                                                                         C=need_c)[short])):
            _host_call(entry, m, n, k, args["A"], lda, args["B"], ldb, args["C"], ldc)


@pytest.mark.skipif(not NO_GPU, reason="relies on the library failing without a device")
def test_extent_follows_the_transpose_flags_and_the_storage_offset():
    m, n, k = 6, 5, 4
    # transa = 'T': A is stored k x m; transb = 'T': B is stored n x k
    lda, ldb, ldc = k + 1, n + 2, m
    A = torch.zeros(lda * (m - 1) + k)
    B = torch.zeros(ldb * (k - 1) + n)
    C = torch.zeros(ldc * n)
    _passes_binding(lambda: _host_call("sgemm_host", m, n, k, A, lda, B, ldb, C, ldc, transa="T", transb="T"))
    with pytest.raises(ValueError, match="^A: "):
        _host_call("sgemm_host", m, n, k, A[:-1].clone(), lda, B, ldb, C, ldc, transa="T", transb="T")
    # a view that starts 3 elements into its storage holds 3 fewer
    big = torch.zeros(A.numel() + 2)
    with pytest.raises(ValueError, match="holds %d$" % (A.numel() - 1)):
        _host_call("sgemm_host", m, n, k, big[3:], lda, B, ldb, C, ldc, transa="T", transb="T")


def test_device_entries_refuse_host_tensors_and_other_dtypes():
    m = n = k = 8
    good = torch.zeros(64)
    for entry in ("sgemm", "sgemm_noalloc"):
        with pytest.raises(ValueError, match="^A: expected a CUDA tensor"):
            getattr(pg, entry)("N", "N", m, n, k, 1.0, good, m, good, k, 0.0, good, m, "ffma", 0)
        with pytest.raises(ValueError, match="^B: expected a float32 tensor"):
            getattr(pg, entry)("N", "N", m, n, k, 1.0, 4096, m, good.double(), k, 0.0, 8192, m, "ffma", 0)
        with pytest.raises(ValueError, match="^C: a numpy array is host memory"):
            getattr(pg, entry)("N", "N", m, n, k, 1.0, 4096, m, 8192, k, 0.0, np.zeros(64, np.float32), m, "ffma",
                               0)
    with pytest.raises(ValueError, match="^A: expected a CUDA tensor"):
        pg.sgemm_rm(m, n, k, 1.0, 4096, k, good, n, 0.0, 8192, n, "ffma", 0)  # row-major A is the column-major B


def test_host_entries_refuse_other_dtypes_and_strided_arrays():
    m = n = k = 8
    f32 = np.zeros(64, np.float32)
    with pytest.raises(ValueError, match="^A: expected a float32 array"):
        pg.sgemm_host("N", "N", m, n, k, 1.0, np.zeros(64), m, f32, k, 0.0, f32, m, "ffma", 0)
    with pytest.raises(ValueError, match="^B: the array must be contiguous"):
        pg.sgemm_host("N", "N", m, n, k, 1.0, f32, m, np.zeros(128, np.float32)[::2], k, 0.0, f32, m, "ffma", 0)
    with pytest.raises(ValueError, match="^C: expected a float32 tensor"):
        pg.sgemm_host("N", "N", m, n, k, 1.0, f32, m, f32, k, 0.0, torch.zeros(64, dtype=torch.float16), m, "ffma",
                      0)


def test_operands_the_call_does_not_touch_are_not_checked():
    # alpha = 0, beta = 1: nothing is read or written, so even a wrong tensor passes
    # and the library returns 0 without a device.
    wrong = torch.zeros(1, dtype=torch.float64)
    pg.sgemm("N", "N", 64, 64, 64, 0.0, wrong, 64, wrong, 64, 1.0, wrong, 64, "tf32", 0)
    pg.sgemm("N", "N", 0, 64, 64, 1.0, wrong, 1, wrong, 64, 0.0, wrong, 1, "tf32", 0)
    # k = 0 with beta != 1: only C is touched; A and B go unchecked, C is checked
    with pytest.raises(ValueError, match="^C: "):
        pg.sgemm("N", "N", 8, 8, 0, 1.0, wrong, 8, wrong, 1, 2.0, wrong, 8, "ffma", 0)


def test_bad_leading_dimension_is_left_to_the_library():
    # lda < m: the binding does not guess an extent; the library answers -8 before any device work
    t = torch.zeros(64)
    with pytest.raises(pg.SgemmError) as e:
        pg.sgemm_host("N", "N", 8, 8, 8, 1.0, t, 4, t, 8, 0.0, t, 8, "ffma", 0)
    assert e.value.code == -8


def test_set_workspace_checks(lib):
    # argument checks of the C entry point come before any device work
    assert lib.sgemm_set_workspace(ctypes.c_void_p(4096 + 16), 1024, None) == -1
    assert "argument 1" in pg.last_error()
    assert lib.sgemm_set_workspace(None, 1024, None) == -2
    assert "argument 2" in pg.last_error()
    with pytest.raises(ValueError, match="CUDA tensor"):
        pg.set_workspace(torch.zeros(1024), stream=0)
    with pytest.raises(ValueError, match="nbytes"):
        pg.set_workspace(4096, stream=0)
