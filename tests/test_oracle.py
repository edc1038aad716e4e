"""Pins for the CPU oracle: it is checked against things other than itself.

Each pin below is a plain function of an ``oracle.Oracle`` so the mutation test
at the end can run the whole set against copies of the oracle with a planted
mistake (a swapped index, a wrong sign, a dropped term) and show that at least
one pin fails for every such mistake.
"""
import json
import os
import shutil
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
from precision_gemm_gb300 import synth
from tests._golden import colmajor_storage, load_worked

NAN = np.float32(np.nan)


def _rand_storage(rows, cols, ld, rng, dist="normal"):
    if dist == "normal":
        vals = rng.standard_normal((cols, ld)).astype(np.float32)
    else:
        vals = rng.integers(-8, 9, size=(cols, ld)).astype(np.float32)
    vals[:, rows:] = NAN
    return vals.reshape(-1)


def _dense(storage, rows, cols, ld):
    """(rows, cols) float64 view of a column-major storage buffer (test-side read)."""
    return storage.reshape(cols, ld)[:, :rows].T.astype(np.float64)


def _op(storage, trans, r_op, c_op, ld):
    """op(X) as a dense float64 matrix of shape (r_op, c_op)."""
    if trans in "Nn":
        return _dense(storage, r_op, c_op, ld)
    return _dense(storage, c_op, r_op, ld).T


# ---------------------------------------------------------------- pins


def pin_worked_example(O):
    """The hand-worked 2x3x2 product in tests/golden, column- and row-major."""
    w = load_worked()
    m, n, k = w["m"], w["n"], w["k"]
    for alpha, beta, exp in w["cases"]:
        # column-major, every leading dimension padded by one NaN row
        A = colmajor_storage(w["opA"], m + 1)
        B = colmajor_storage(w["opB"], k + 1)
        C = colmajor_storage(w["Cin"], m + 1)
        cref, _ = O.full("N", "N", m, n, k, alpha, A, m + 1, B, k + 1, beta, C, m + 1)
        assert np.array_equal(cref, exp), (alpha, beta, cref, exp)
        # row-major storage as the lecture's host wrapper addresses it (i*ld + j):
        # that buffer is the column-major storage of the transpose.
        At = colmajor_storage(w["opA"].T, k + 2)   # A row-major, lda = k+2
        Bt = colmajor_storage(w["opB"].T, n + 2)   # B row-major, ldb = n+2
        cref_t, _ = O.full("T", "T", m, n, k, alpha, At, k + 2, Bt, n + 2, beta, C, m + 1)
        assert np.array_equal(cref_t, exp)


def pin_identity(O):
    rng = np.random.default_rng(1)
    m, n = 37, 23
    A = colmajor_storage(np.eye(m), m + 4)
    B = _rand_storage(m, n, m + 2, rng)
    C = _rand_storage(m, n, m + 3, rng)
    alpha, beta = np.float32(1.5), np.float32(-0.25)
    cref, den = O.full("N", "N", m, n, m, alpha, A, m + 4, B, m + 2, beta, C, m + 3)
    exp = float(alpha) * _dense(B, m, n, m + 2) + float(beta) * _dense(C, m, n, m + 3)
    assert np.array_equal(cref, exp)
    assert np.array_equal(den, np.abs(float(alpha) * _dense(B, m, n, m + 2))
                          + np.abs(float(beta) * _dense(C, m, n, m + 3)))


def pin_permutations(O):
    rng = np.random.default_rng(2)
    m, k, n = 19, 19, 11
    sigma = rng.permutation(m)
    P = np.zeros((m, k))
    P[np.arange(m), sigma] = 1.0
    X = _rand_storage(k, n, k, rng)
    cref, _ = O.full("N", "N", m, n, k, 1.0, colmajor_storage(P, m), m, X, k, 0.0, None, m)
    assert np.array_equal(cref, _dense(X, k, n, k)[sigma, :])
    # permutation on the right: C[i, j] = A[i, tau(j)]
    k2, n2 = 13, 13
    tau = rng.permutation(n2)
    Q = np.zeros((k2, n2))
    Q[tau, np.arange(n2)] = 1.0
    Y = _rand_storage(m, k2, m + 1, rng)
    cref2, _ = O.full("N", "N", m, n2, k2, 1.0, Y, m + 1, colmajor_storage(Q, k2), k2, 0.0, None, m)
    assert np.array_equal(cref2, _dense(Y, m, k2, m + 1)[:, tau])


def pin_all_ones(O):
    m, n, k = 9, 14, 1000
    A = np.ones(m * k, np.float32)
    B = np.ones(k * n, np.float32)
    cref, den = O.full("N", "N", m, n, k, 1.0, A, m, B, k, 0.0, None, m)
    assert np.all(cref == k) and np.all(den == k)


def pin_rank_one(O):
    rng = np.random.default_rng(3)
    m, n = 31, 17
    u = rng.standard_normal(m).astype(np.float32)
    v = rng.standard_normal(n).astype(np.float32)
    C = _rand_storage(m, n, m, rng)
    alpha, beta = np.float32(0.75), np.float32(2.0)
    cref, _ = O.full("N", "N", m, n, 1, alpha, u, m, v, 1, beta, C, m)
    exp = float(alpha) * np.outer(u.astype(np.float64), v.astype(np.float64)) \
        + float(beta) * _dense(C, m, n, m)
    assert np.allclose(cref, exp, rtol=1e-15, atol=0)


def pin_alpha_beta_algebra(O):
    rng = np.random.default_rng(4)
    m, n, k = 21, 18, 40
    A = _rand_storage(m, k, m, rng)
    B = _rand_storage(k, n, k, rng)
    C = _rand_storage(m, n, m, rng)
    alpha, beta = np.float32(-1.25), np.float32(0.5)
    full, den = O.full("N", "N", m, n, k, alpha, A, m, B, k, beta, C, m)
    prod, _ = O.full("N", "N", m, n, k, 1.0, A, m, B, k, 0.0, None, m)
    assert np.all(np.abs(full - (float(alpha) * prod + float(beta) * _dense(C, m, n, m)))
                  <= 1e-15 * den)
    # alpha = 0: A and B are not read (NaN there changes nothing)
    An = np.full_like(A, np.nan)
    Bn = np.full_like(B, np.nan)
    c0, _ = O.full("N", "N", m, n, k, 0.0, An, m, Bn, k, beta, C, m)
    assert np.array_equal(c0, float(beta) * _dense(C, m, n, m))
    # beta = 0: Cin is not read
    Cn = np.full_like(C, np.nan)
    cb, _ = O.full("N", "N", m, n, k, alpha, A, m, B, k, 0.0, Cn, m)
    assert np.all(np.isfinite(cb))
    assert np.array_equal(cb, float(alpha) * prod)
    # k = 0: only the beta term remains
    ck, dk = O.full("N", "N", m, n, 0, alpha, A, m, B, 1, beta, C, m)
    assert np.array_equal(ck, float(beta) * _dense(C, m, n, m))


def pin_transpose_identities(O):
    rng = np.random.default_rng(5)
    m, n, k = 23, 29, 31
    A = _rand_storage(m, k, m + 1, rng)
    B = _rand_storage(k, n, k + 2, rng)
    Ad, Bd = _dense(A, m, k, m + 1), _dense(B, k, n, k + 2)
    At = colmajor_storage(Ad.T, k + 3)
    Bt = colmajor_storage(Bd.T, n + 1)
    ref, _ = O.full("N", "N", m, n, k, 1.0, A, m + 1, B, k + 2, 0.0, None, m)
    for ta, tb, a, la, b, lb in (("T", "N", At, k + 3, B, k + 2), ("N", "T", A, m + 1, Bt, n + 1),
                                 ("T", "T", At, k + 3, Bt, n + 1), ("t", "c", At, k + 3, Bt, n + 1)):
        got, _ = O.full(ta, tb, m, n, k, 1.0, a, la, b, lb, 0.0, None, m)
        assert np.array_equal(got, ref), (ta, tb)
    # (A B)^T = B^T A^T
    swapped, _ = O.full("N", "N", n, m, k, 1.0, Bt, n + 1, At, k + 3, 0.0, None, n)
    assert np.array_equal(swapped, ref.T)


def pin_second_loop_order(O):
    rng = np.random.default_rng(6)
    sizes = (0, 1, 2, 5, 17)
    for m in sizes:
        for n in sizes:
            for k in sizes:
                ta, tb = rng.choice(["N", "T"]), rng.choice(["N", "T"])
                ra, ca = (m, k) if ta == "N" else (k, m)
                rb, cb = (k, n) if tb == "N" else (n, k)
                lda, ldb, ldc = max(1, ra) + 1, max(1, rb) + 2, max(1, m) + 1
                A = _rand_storage(ra, ca, lda, rng)
                B = _rand_storage(rb, cb, ldb, rng)
                C = _rand_storage(m, n, ldc, rng)
                alpha, beta = np.float32(rng.standard_normal()), np.float32(rng.standard_normal())
                a, _ = O.full(ta, tb, m, n, k, alpha, A, lda, B, ldb, beta, C, ldc)
                b = O.ikj(ta, tb, m, n, k, alpha, A, lda, B, ldb, beta, C, ldc)
                assert np.array_equal(a, b), (m, n, k, ta, tb)


def pin_library_matmul(O):
    """Against numpy's float64 matmul of the same fp32 values."""
    rng = np.random.default_rng(7)
    for (m, n, k) in ((33, 47, 129), (64, 1, 300), (1, 70, 65)):
        for ta in "NT":
            for tb in "NT":
                ra, ca = (m, k) if ta == "N" else (k, m)
                rb, cb = (k, n) if tb == "N" else (n, k)
                lda, ldb, ldc = ra + 3, rb + 1, m + 2
                A = _rand_storage(ra, ca, lda, rng)
                B = _rand_storage(rb, cb, ldb, rng)
                C = _rand_storage(m, n, ldc, rng)
                alpha, beta = np.float32(0.8), np.float32(-1.5)
                cref, den = O.full(ta, tb, m, n, k, alpha, A, lda, B, ldb, beta, C, ldc)
                exp = float(alpha) * (_op(A, ta, m, k, lda) @ _op(B, tb, k, n, ldb)) \
                    + float(beta) * _dense(C, m, n, ldc)
                assert np.all(np.abs(cref - exp) <= 1e-13 * den), (m, n, k, ta, tb)


def pin_integer_exact(O):
    """Integer inputs: exact against int64 arithmetic."""
    rng = np.random.default_rng(8)
    m, n, k = 40, 36, 250
    A = _rand_storage(m, k, m, rng, dist="int")
    B = _rand_storage(k, n, k + 1, rng, dist="int")
    C = _rand_storage(m, n, m, rng, dist="int")
    Ai = _dense(A, m, k, m).astype(np.int64)
    Bi = _dense(B, k, n, k + 1).astype(np.int64)
    Ci = _dense(C, m, n, m).astype(np.int64)
    cref, _ = O.full("N", "N", m, n, k, 1.0, A, m, B, k + 1, 1.0, C, m)
    assert np.array_equal(cref, (Ai @ Bi + Ci).astype(np.float64))
    cref3, _ = O.full("N", "N", m, n, k, 3.0, A, m, B, k + 1, -2.0, C, m)
    assert np.array_equal(cref3, (3 * (Ai @ Bi) - 2 * Ci).astype(np.float64))


def pin_entries_equal_full(O):
    rng = np.random.default_rng(9)
    m, n, k = 50, 45, 60
    A = _rand_storage(m, k, m + 2, rng)
    B = _rand_storage(k, n, k, rng)
    C = _rand_storage(m, n, m + 1, rng)
    cref, den = O.full("N", "N", m, n, k, 1.5, A, m + 2, B, k, 0.25, C, m + 1)
    ii, jj = synth.sample_entries(m, n, count=200, seed=3, edges=(8, 16))
    ce, de = O.entries("N", "N", m, n, k, 1.5, A, m + 2, B, k, 0.25, C, m + 1, ii, jj)
    assert np.array_equal(ce, cref[ii, jj]) and np.array_equal(de, den[ii, jj])


def pin_padding_never_read(O):
    """NaN in every leading-dimension gap leaves the result finite."""
    rng = np.random.default_rng(10)
    m, n, k = 30, 20, 25
    for ta in "NT":
        for tb in "NT":
            ra, ca = (m, k) if ta == "N" else (k, m)
            rb, cb = (k, n) if tb == "N" else (n, k)
            A = _rand_storage(ra, ca, ra + 7, rng)
            B = _rand_storage(rb, cb, rb + 5, rng)
            C = _rand_storage(m, n, m + 3, rng)
            cref, den = O.full(ta, tb, m, n, k, 1.0, A, ra + 7, B, rb + 5, 1.0, C, m + 3)
            assert np.all(np.isfinite(cref)) and np.all(np.isfinite(den))


def pin_denominator(O):
    rng = np.random.default_rng(11)
    m, n, k = 12, 13, 14
    A = np.abs(_rand_storage(m, k, m, rng))
    B = np.abs(_rand_storage(k, n, k, rng))
    C = np.abs(_rand_storage(m, n, m, rng))
    cref, den = O.full("N", "N", m, n, k, 2.0, A, m, B, k, 0.5, C, m)
    assert np.allclose(den, cref, rtol=1e-15, atol=0)
    A2 = _rand_storage(m, k, m, rng)
    cref2, den2 = O.full("N", "N", m, n, k, -2.0, A2, m, B, k, -0.5, C, m)
    assert np.all(den2 >= np.abs(cref2) * (1 - 1e-15))
    # den is the same sum with every sign made positive
    cabs, _ = O.full("N", "N", m, n, k, 2.0, np.abs(A2), m, B, k, 0.5, C, m)
    assert np.allclose(den2, cabs, rtol=1e-15, atol=0)


PINS = [pin_worked_example, pin_identity, pin_permutations, pin_all_ones, pin_rank_one,
        pin_alpha_beta_algebra, pin_transpose_identities, pin_second_loop_order,
        pin_library_matmul, pin_integer_exact, pin_entries_equal_full,
        pin_padding_never_read, pin_denominator]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(oracle_lib, pin):
    pin(oracle_lib)


# ------------------------------------------------- checker (acceptance rule)


def test_checker_flags_errors():
    cref = np.array([1.0, -2.0, 0.0, 3.0])
    den = np.array([1.0, 2.0, 0.0, 3.0])
    ok = oracle.check(np.array([1.0, -2.0, -0.0, 3.0], np.float32), cref, den, 1e-5)
    assert ok["ok"] and ok["max_err"] == 0.0
    bad = oracle.check(np.array([1.0 + 1e-4, -2.0, 0.0, 3.0], np.float32), cref, den, 1e-5)
    assert not bad["ok"] and bad["n_bad"] == 1
    nan = oracle.check(np.array([np.nan, -2.0, 0.0, 3.0], np.float32), cref, den, 1.0)
    assert not nan["ok"]
    inf = oracle.check(np.array([1.0, -np.inf, 0.0, 3.0], np.float32), cref, den, 1.0)
    assert not inf["ok"]
    zero_den = oracle.check(np.array([1.0, -2.0, 1e-30, 3.0], np.float32), cref, den, 1.0)
    assert not zero_den["ok"]
    # a non-finite reference must be matched in kind
    r = np.array([np.inf, np.nan])
    assert oracle.check(np.array([np.inf, np.nan]), r, np.array([np.inf, np.nan]), 1e-5)["ok"]
    assert not oracle.check(np.array([1.0, np.nan]), r, np.array([np.inf, np.nan]), 1e-5)["ok"]


def test_checker_floor_covers_fp32_underflow(oracle_lib):
    """Why the check has an absolute floor: FP32 with gradual underflow rounds a
    result below 2^-126 to a multiple of 2^-149, so a dot product whose products
    underflow carries an absolute error no relative bound covers.  Modelled here
    on the CPU: a sequential FP32 fused multiply-add loop (the product and the
    running sum added exactly in double, then rounded once to float32, which
    keeps subnormals) over k products near 2^-144 misses tol * den, and stays
    within tol * den + (k + 2) * 2^-149."""
    rng = np.random.default_rng(3)
    k = 512
    a = (rng.uniform(1.0, 2.0, k) * np.where(rng.random(k) < 0.5, -1.0, 1.0) * 2.0 ** -72).astype(np.float32)
    b = (rng.uniform(1.0, 2.0, k) * 2.0 ** -72).astype(np.float32)
    acc = np.float32(0.0)
    for p in range(k):
        acc = np.float32(np.float64(acc) + np.float64(a[p]) * np.float64(b[p]))
    assert 0 < abs(float(acc)) < 2.0 ** -126
    A = torch.from_numpy(a.copy())            # 1 x k, lda 1
    B = torch.from_numpy(b.copy())            # k x 1, ldb k
    C = torch.zeros(1)
    cref, den = oracle_lib.full("N", "N", 1, 1, k, 1.0, A, 1, B, k, 0.0, C, 1)
    out = np.array([[float(acc)]])
    assert not oracle.check(out, cref, den, 1e-5)["ok"]
    assert oracle.check(out, cref, den, 1e-5, floor=(k + 2) * 2.0 ** -149)["ok"]
    # the floor is a bound, not a pass for anything: an error of 10x the floor fails
    assert not oracle.check(out + 10 * (k + 2) * 2.0 ** -149, cref, den, 1e-5, floor=(k + 2) * 2.0 ** -149)["ok"]
    # and with floor = 0 the check is the plain normalised criterion
    assert np.array_equal(oracle.normalised_error(out, cref, den), oracle.normalised_error(out, cref, den, 0.0))


def test_synth_draws_are_seeded_and_padded():
    p = synth.Problem(5, 4, 3, lda=8, ldb=3, ldc=6, dist="normal", seed=42)
    A1, B1, C1 = synth.make(p)
    A2, B2, C2 = synth.make(p)
    assert torch.equal(A1.view(torch.int32), A2.view(torch.int32))
    assert A1.numel() == 8 * 3 and B1.numel() == 3 * 4 and C1.numel() == 6 * 4
    pad = A1.view(torch.int32).view(3, 8)[:, 5:]
    assert torch.all(pad == synth.NAN_BITS)
    assert torch.all(torch.isfinite(A1.view(3, 8)[:, :5]))
    # the draw order is A, then B, then C, each as its full storage buffer
    g = torch.Generator().manual_seed(42)
    a = torch.randn(24, generator=g)
    b = torch.randn(12, generator=g)
    assert torch.equal(a.view(3, 8)[:, :5], A1.view(3, 8)[:, :5]) and torch.equal(b, B1)


def test_sample_entries_cover_edges():
    ii, jj = synth.sample_entries(300, 200, count=100, seed=1, edges=(128,))
    pairs = set(zip(ii.tolist(), jj.tolist()))
    for corner in ((0, 0), (299, 0), (0, 199), (299, 199)):
        assert corner in pairs
    assert any(i in (127, 128) for i in ii) and any(j in (127, 128) for j in jj)
    assert len(pairs) == ii.size  # no duplicates
    assert ii.max() < 300 and jj.max() < 200


# ------------------------------------------------------- planted mistakes

MUTATIONS = {
    "a_index_transposed": ("? (double)A[i + p * lda]", "? (double)A[p + i * lda]"),
    "b_index_transposed": ("? (double)B[p + j * ldb]", "? (double)B[j + p * ldb]"),
    "trans_flag_ignored": ("return t == 'N' || t == 'n';", "return 1;"),
    "sum_wrong_sign": ("sum += prod;", "sum -= prod;"),
    "first_term_dropped": ("for (int64_t p = 0; p < k; ++p) {\n            double prod",
                           "for (int64_t p = 1; p < k; ++p) {\n            double prod"),
    "last_term_dropped": ("for (int64_t p = 0; p < k; ++p) {\n            double prod",
                          "for (int64_t p = 0; p + 1 < k; ++p) {\n            double prod"),
    "beta_term_dropped": ("*cref = a * sum + c_term;", "*cref = a * sum;"),
    "c_index_transposed": ("c_term = b * (double)C[i + j * ldc];",
                           "c_term = b * (double)C[j + i * ldc];"),
    "alpha_ignored": ("*cref = a * sum + c_term;", "*cref = sum + c_term;"),
    "beta_reads_c_when_zero": ("if (b != 0.0)\n        c_term", "if (1)\n        c_term"),
    "den_without_abs": ("abs_sum += fabs(a * prod);", "abs_sum += a * prod;"),
    "den_without_c": ("*den = abs_sum + fabs(c_term);", "*den = abs_sum;"),
    "wrong_ld_for_a": ("op_a(transa, A, lda, i, p)", "op_a(transa, A, ldb, i, p)"),
    "wrong_ld_for_c": ("(double)C[i + j * ldc];\n    *cref", "(double)C[i + j * (ldc - 1)];\n    *cref"),
}


def _run_pins(O):
    failed = []
    for pin in PINS:
        try:
            pin(O)
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    return failed


_CHILD = """
import json, sys
sys.path.insert(0, {root!r})
import oracle
from tests.test_oracle import _run_pins
print(json.dumps(_run_pins(oracle.Oracle(oracle.load({lib!r})))))
"""


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(tmp_path, name):
    """Each planted mistake fails at least one pin.  The pins run in a child
    process because a mutant that indexes out of bounds may crash; a crash is
    also a caught mistake."""
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = open(os.path.join(os.path.dirname(oracle.__file__), "sgemm_oracle.c")).read()
    old, new = MUTATIONS[name]
    assert src.count(old) >= 1, "mutation anchor not found: %s" % name
    mutant_src = tmp_path / "mutant.c"
    mutant_src.write_text(src.replace(old, new, 1))
    lib = oracle.build_from(str(mutant_src), str(tmp_path / "libmutant.so"))
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    proc = subprocess.run([sys.executable, "-c", _CHILD.format(root=root, lib=lib)],
                          capture_output=True, text=True, timeout=300,
                          env={**os.environ, "OMP_NUM_THREADS": "2"})
    if proc.returncode != 0:
        return  # the mutant crashed or raised: caught
    failed = json.loads(proc.stdout.strip().splitlines()[-1])
    assert failed, "no pin caught the planted mistake %s" % name


def test_unmutated_oracle_passes_every_pin(oracle_lib):
    assert _run_pins(oracle_lib) == []


def test_acceptance_workloads_match_their_specification():
    """The named workloads carry the acceptance suite's sizes, leading dimensions,
    scalars, distributions and seed, and their draws have the stated ranges."""
    P = synth.config_problems()
    want = {
        "c1_256": (256, 256, 256, 256, 256, 256, 1.0, 0.0, "uniform", "uniform", "col"),
        "c2_rm1024": (1024, 1024, 1024, 1024, 1024, 1024, 1.0, 0.0, "uniform", "uniform", "row"),
        "c2_rm2048": (2048, 2048, 2048, 2048, 2048, 2048, 1.0, 0.0, "uniform", "uniform", "row"),
        "c2_rm4096": (4096, 4096, 4096, 4096, 4096, 4096, 1.0, 0.0, "uniform", "uniform", "row"),
        # ragged: lda = m + 13, ldb = k + 7, ldc = m + 5, C_in ~ N(0, 1)
        "c3_ragged": (3000, 1500, 777, 3013, 784, 3005, 1.5, -0.5, "normal", "normal", "col"),
        "c4_8192": (8192, 8192, 8192, 8192, 8192, 8192, 1.0, 1.0, "uniform", "uniform", "col"),
        "c4_16384": (16384, 16384, 16384, 16384, 16384, 16384, 1.0, 1.0, "uniform", "uniform", "col"),
        "c5a_16384x16384x64": (16384, 16384, 64, 16384, 64, 16384, 1.0, 0.0, "normal", "normal", "col"),
        "c5b_128x128x262144": (128, 128, 262144, 128, 262144, 128, 1.0, 0.0, "normal", "normal", "col"),
        "c5c_8192x64x8192": (8192, 64, 8192, 8192, 8192, 8192, 1.0, 0.0, "normal", "normal", "col"),
    }
    assert sorted(P) == sorted(want)
    for name, (m, n, k, lda, ldb, ldc, alpha, beta, dist, c_dist, layout) in want.items():
        p = P[name]
        got = (p.m, p.n, p.k, p.lda, p.ldb, p.ldc, p.alpha, p.beta, p.dist, p.c_dist, p.layout)
        assert got == (m, n, k, lda, ldb, ldc, alpha, beta, dist, c_dist, layout), name
        assert p.transa == "N" and p.transb == "N" and p.seed == 0, name
    # draws: U[-1, 1) and N(0, 1); the ragged problem's padding rows hold the NaN sentinel
    A, B, C = synth.make(P["c1_256"])
    for x in (A, B):
        assert float(x.min()) >= -1.0 and float(x.max()) < 1.0 and abs(float(x.mean())) < 0.01
    A, B, C = synth.make(P["c3_ragged"])
    a = A.view(777, 3013)
    assert torch.all(a[:, 3000:].view(torch.int32) == synth.NAN_BITS)
    body = a[:, :3000]
    assert torch.isfinite(body).all() and abs(float(body.mean())) < 0.01 and abs(float(body.std()) - 1) < 0.01
    assert torch.all(B.view(1500, 784)[:, 777:].view(torch.int32) == synth.NAN_BITS)
    assert torch.all(C.view(1500, 3005)[:, 3000:].view(torch.int32) == synth.NAN_BITS)
    assert abs(float(C.view(1500, 3005)[:, :3000].std()) - 1) < 0.01
