"""The host co-worker of the hybrid CPU + GPU column split, on the CPU.

The co-worker (precision_gemm_gb300/csrc/host_sgemm.cpp, inside the library and
reached there only through sgemm_host with a split set) is compiled here on its
own, with a three-line shim that calls it, and held to the oracle: FP32 fused
multiply-add chains in increasing p meet the FFMA tolerance, integer inputs
match bit for bit, results are identical for any thread count, the ld gaps are
never written, C is not read when beta = 0.  The split's setter is checked too.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
import precision_gemm_gb300 as pg
from precision_gemm_gb300 import build as pgbuild
from precision_gemm_gb300 import synth
from tests import _harness as H

SHIM = r'''
#include <cstdint>
#include "host_sgemm.h"
extern "C" __attribute__((visibility("default")))
void coworker(char ta, char tb, int64_t m, int64_t n, int64_t k, float alpha, const float* A, int64_t lda,
              const float* B, int64_t ldb, float beta, float* C, int64_t ldc, int threads) {
    pg::host_sgemm(ta, tb, m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, threads);
}
'''


@pytest.fixture(scope="module")
def coworker(tmp_path_factory):
    d = tmp_path_factory.mktemp("coworker")
    shim = d / "shim.cpp"
    shim.write_text(SHIM)
    so = d / "libcoworker.so"
    cmd = ["g++", "-shared", *pgbuild.HOST_FLAGS, "-I", pgbuild.CSRC, str(shim),
           os.path.join(pgbuild.CSRC, "host_sgemm.cpp"), "-o", str(so)]
    subprocess.run(cmd, check=True)
    lib = ctypes.CDLL(str(so))
    c, i64, f, vp = ctypes.c_char, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p
    lib.coworker.argtypes = [c, c, i64, i64, i64, f, vp, i64, vp, i64, f, vp, i64, ctypes.c_int]
    lib.coworker.restype = None
    return lib


def _run(lib, p, A, B, C, threads=0):
    out = C.clone()
    lib.coworker(p.transa.encode(), p.transb.encode(), p.m, p.n, p.k, p.alpha, A.data_ptr(), p.lda, B.data_ptr(),
                 p.ldb, p.beta, out.data_ptr(), p.ldc, threads)
    return out


@pytest.mark.parametrize("trans", ["NN", "NT", "TN", "TT"])
@pytest.mark.parametrize("mnk", [(1, 1, 1), (130, 37, 300), (17, 200, 513), (300, 66, 1)])
def test_coworker_matches_oracle(coworker, trans, mnk):
    m, n, k = mnk
    p = synth.Problem(m, n, k, transa=trans[0], transb=trans[1], alpha=1.25, beta=-0.5, dist="normal", seed=7)
    p = p.with_(lda=p.lda + 3, ldb=p.ldb + 1, ldc=p.ldc + 2)
    A, B, C = synth.make(p)
    out = _run(coworker, p, A, B, C)
    cref, den = H.reference_full(p, A, B, C)
    res = oracle.check(H.logical(p, out), cref, den, oracle.TOL["ffma"])
    assert res["ok"], res
    assert H.padding_intact(p, out, C)


def test_coworker_integers_exact_and_thread_independent(coworker):
    p = synth.Problem(333, 129, 700, lda=337, ldc=335, alpha=1.0, beta=1.0, dist="int", seed=5)
    A, B, C = synth.make(p)
    outs = [_run(coworker, p, A, B, C, threads=t) for t in (1, 3, 8)]
    cref, _ = H.reference_full(p, A, B, C)
    assert np.array_equal(H.logical(p, outs[0]), cref)
    q = synth.Problem(257, 70, 1000, alpha=0.75, beta=0.25, dist="normal", seed=9)
    A, B, C = synth.make(q)
    outs += [_run(coworker, q, A, B, C, threads=t) for t in (1, 2, 7)]
    for a, b in ((outs[0], outs[1]), (outs[0], outs[2]), (outs[3], outs[4]), (outs[3], outs[5])):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_coworker_beta_and_alpha_rules(coworker):
    p = synth.Problem(70, 40, 90, alpha=1.0, beta=0.0, dist="normal", seed=11)
    A, B, C = synth.make(p)
    C.fill_(float("nan"))
    out = _run(coworker, p, A, B, C)  # beta = 0: C is not read
    cref, den = H.reference_full(p, A, B, C)
    assert np.all(np.isfinite(H.logical(p, out)))
    assert oracle.check(H.logical(p, out), cref, den, oracle.TOL["ffma"])["ok"]
    q = p.with_(alpha=0.0, beta=2.0)
    A2, B2, C2 = synth.make(q)
    A2.fill_(float("nan"))
    B2.fill_(float("nan"))
    out = _run(coworker, q, A2, B2, C2)  # alpha = 0: A and B are not read
    assert np.array_equal(H.logical(q, out), 2.0 * H.logical(q, C2))


def test_host_split_setter():
    lib = pg.load_library()
    try:
        assert lib.sgemm_set_host_split(float("nan")) == -1 and "argument 1" in pg.last_error()
        assert lib.sgemm_set_host_split(float("inf")) == -1
        pg.set_host_split(0.0)
        assert pg.host_split_ratio("tf32") == 0.0
        pg.set_host_split(3.0)
        assert pg.host_split_ratio("ffma") == 3.0
        pg.set_host_split(-1.0)
        assert pg.host_split_ratio("3xtf32") > 0  # automatic: the last measured ratio (15 before any call)
        assert lib.sgemm_host_split_ratio(7) == -1.0
    finally:
        pg.set_host_split(0.0)
