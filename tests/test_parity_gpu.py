"""GPU parity: the CUDA path, called through the C ABI, against the CPU oracle.

Tolerance on the normalised error |C - Cref| / (sum_p |alpha a b| + |beta c|):
1e-5 for FFMA and 3xTF32, 5e-3 for TF32.  Integer-valued inputs must match
bit for bit in every mode.  Every run also checks that the leading-dimension
gaps of C and guard words around every buffer are unchanged.
"""
import numpy as np
import pytest
import torch

import oracle
import precision_gemm_gb300 as pg
from precision_gemm_gb300 import synth
from tests import _harness as H
from tests._golden import colmajor_storage, load_worked

pytestmark = pytest.mark.gpu
MODES = ("ffma", "tf32", "3xtf32")
CFG = synth.config_problems()


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pg.load_library()
    pg.force_plan(0, 0)
    yield
    pg.force_plan(0, 0)
    assert pg.device_status() == 0


def _assert_ok(res, what):
    assert res["ok"], "%s: %d/%d entries above tol %.0e (max err %.3e)" % (
        what, res["n_bad"], res["n"], res["tol"], res["max_err"])
    assert res["canaries"], "%s: guard words around a buffer changed" % what
    assert res["padding"], "%s: the ld gap of C changed" % what


# ------------------------------------------------------------ the five workloads

@pytest.mark.parametrize("mode", MODES)
def test_config1_256_full(mode):
    _assert_ok(H.check_problem(CFG["c1_256"], mode), "256^3 " + mode)


@pytest.mark.parametrize("mode", MODES)
def test_config2_rowmajor_1024_full(mode):
    _assert_ok(H.check_problem(CFG["c2_rm1024"], mode), "row-major 1024^3 " + mode)


@pytest.mark.parametrize("size", (2048, 4096))
@pytest.mark.parametrize("mode", MODES)
def test_config2_rowmajor_sampled(mode, size):
    _assert_ok(H.check_problem(CFG["c2_rm%d" % size], mode, sample=4096), "row-major %d^3 %s" % (size, mode))


@pytest.mark.parametrize("mode", MODES)
def test_config3_ragged_full(mode):
    _assert_ok(H.check_problem(CFG["c3_ragged"], mode), "ragged 3000x1500x777 " + mode)


@pytest.mark.parametrize("mode", ("ffma", "3xtf32", "tf32"))
def test_config4_8192_sampled(mode):
    _assert_ok(H.check_problem(CFG["c4_8192"], mode, sample=4096), "8192^3 " + mode)


@pytest.mark.parametrize("mode", ("ffma", "3xtf32"))
def test_config4_16384_sampled(mode):
    _assert_ok(H.check_problem(CFG["c4_16384"], mode, sample=4096), "16384^3 " + mode)


@pytest.mark.parametrize("mode", MODES)
def test_config5a_k64_sampled(mode):
    _assert_ok(H.check_problem(CFG["c5a_16384x16384x64"], mode, sample=4096), "16384^2x64 " + mode)


@pytest.mark.parametrize("mode", MODES)
def test_config5b_splitk_full(mode):
    p = CFG["c5b_128x128x262144"]
    plan = pg.sgemm_plan(p.transa, p.transb, p.m, p.n, p.k, p.alpha, 256, p.lda, 256, p.ldb, p.beta, 256,
                         p.ldc, mode)
    assert plan["split_k"] > 1, plan
    _assert_ok(H.check_problem(p, mode), "128x128x262144 " + mode)


@pytest.mark.parametrize("mode", MODES)
def test_config5c_tall_thin_sampled(mode):
    _assert_ok(H.check_problem(CFG["c5c_8192x64x8192"], mode, sample=4096), "8192x64x8192 " + mode)


# ------------------------------------------------------------ exactness and structure

@pytest.mark.parametrize("mode", MODES)
def test_worked_example_exact(mode):
    """The hand-worked 2x3x2 product of tests/golden, bit for bit."""
    w = load_worked()
    m, n, k = w["m"], w["n"], w["k"]
    for alpha, beta, exp in w["cases"]:
        A = torch.from_numpy(colmajor_storage(w["opA"], m + 1))
        B = torch.from_numpy(colmajor_storage(w["opB"], k + 1))
        C = torch.from_numpy(colmajor_storage(w["Cin"], m + 1))
        p = synth.Problem(m, n, k, lda=m + 1, ldb=k + 1, ldc=m + 1, alpha=alpha, beta=beta)
        out, ok = H.run_gpu(p, mode, A, B, C)
        assert ok and np.array_equal(H.logical(p, out), exp), (mode, alpha, beta, H.logical(p, out))


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("shape", [(300, 260, 1000), (129, 257, 64), (640, 96, 4096)])
def test_integer_inputs_bitwise(mode, shape):
    """Integers in [-8, 8]: every product and partial sum is exact in FP32 and in
    TF32 (11-bit integers are representable), so every mode must agree with the
    oracle bit for bit, whatever the summation order."""
    m, n, k = shape
    p = synth.Problem(m, n, k, lda=m + 3, ldb=k, ldc=m + 1, alpha=1.0, beta=1.0, dist="int", seed=5)
    A, B, C = synth.make(p)
    out, ok = H.run_gpu(p, mode, A, B, C)
    cref, _ = H.reference_full(p, A, B, C)
    assert ok and H.padding_intact(p, out, C)
    assert np.array_equal(H.logical(p, out), cref)


@pytest.mark.parametrize("mode", MODES)
def test_deterministic(mode):
    """Two runs give bitwise identical C, split-K included."""
    for p in (CFG["c3_ragged"], CFG["c5b_128x128x262144"].with_(k=65536)):
        A, B, C = synth.make(p)
        o1, _ = H.run_gpu(p, mode, A, B, C)
        o2, _ = H.run_gpu(p, mode, A, B, C)
        assert torch.equal(o1.view(torch.int32), o2.view(torch.int32)), (p, mode)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("trans", ["NT", "TN", "TT", "tc"])
def test_transposed_operands(mode, trans):
    p = synth.Problem(333, 222, 181, transa=trans[0], transb=trans[1], alpha=0.5, beta=2.0,
                      dist="normal", seed=7)
    p = p.with_(lda=p.lda + 5, ldb=p.ldb + 3, ldc=p.ldc + 2)
    _assert_ok(H.check_problem(p, mode), "trans %s %s" % (trans, mode))


@pytest.mark.parametrize("mode", ("tf32", "3xtf32"))
@pytest.mark.parametrize("trans", ["NT", "TN", "TT"])
@pytest.mark.parametrize("mnk", [(512, 384, 256), (96, 64, 1000), (1024, 96, 333), (640, 1024, 2048)])
def test_transposed_operands_read_in_place(mode, trans, mnk):
    """The tensor-core kernels read transposed operands through K-major / N-major
    descriptors (3-D boxes when the extent is a multiple of 32) instead of a
    transposing copy; covers the SM-pair and single-SM kernels."""
    m, n, k = mnk
    p = synth.Problem(m, n, k, transa=trans[0], transb=trans[1], alpha=1.5, beta=-1.0, dist="normal", seed=31)
    plan = pg.sgemm_plan(p.transa, p.transb, m, n, k, p.alpha, 256, p.lda, 256, p.ldb, p.beta, 256, p.ldc, mode)
    if mode == "tf32":  # no transposing copy; an ld that is not a multiple of 4 still needs a plain copy
        assert plan["prep_a_name"] == ("none" if p.lda % 4 == 0 else "copy")
        assert plan["prep_b_name"] == ("none" if p.ldb % 4 == 0 else "copy")
    _assert_ok(H.check_problem(p, mode), "in-place trans %s %s %s" % (trans, mode, mnk))


@pytest.mark.parametrize("mode", ("tf32", "3xtf32"))
@pytest.mark.parametrize("trans", ["NN", "NT", "TN", "TT"])
@pytest.mark.parametrize("case", [
    # (m, n, k, forced bn): SM-pair tiles with ragged rows/columns and split-K (the
    # smaller shapes would run on single-SM 128 x 64 tiles unless bn is forced)
    (1024, 1024, 512, 256),
    (700, 2148, 300, 0),
    (640, 640, 1000, 256),
    (1000, 512, 777, 128),   # 128-wide pair tiles, 2-D A boxes when M-major
    (512, 512, 8192, 256),   # split-K on the pair kernel
])
def test_pair_kernel_shapes(mode, trans, case):
    """The SM-pair kernel (256-row tiles) with every operand orientation,
    ragged edges, both tile widths, and split-K; beta != 0 so the epilogue's
    batched reads of C are checked."""
    m, n, k, bn = case
    p = synth.Problem(m, n, k, transa=trans[0], transb=trans[1], alpha=0.75, beta=1.5, dist="normal", seed=37)
    try:
        pg.force_plan(bn, 0)
        plan = pg.sgemm_plan(p.transa, p.transb, m, n, k, p.alpha, 256, p.lda, 256, p.ldb, p.beta, 256, p.ldc, mode)
        assert plan["kernel_name"] == "tc2", plan
        _assert_ok(H.check_problem(p, mode), "pair %s %s %s" % (case, trans, mode))
    finally:
        pg.force_plan(0, 0)


@pytest.mark.parametrize("mode", ("tf32", "3xtf32"))
@pytest.mark.parametrize("mnk", [(2500, 2000, 1000), (2560, 2048, 700), (4000, 1100, 2048)])
def test_last_wave_split(mode, mnk):
    """SM pairs: tiles past the last whole wave run as K slices whose partials the
    last slice to finish sums in slice order -- ragged edges included, beta != 0,
    bitwise repeatable."""
    m, n, k = mnk
    p = synth.Problem(m, n, k, ldc=m + 3, alpha=-1.25, beta=0.5, dist="normal", seed=43)
    plan = pg.sgemm_plan("N", "N", m, n, k, p.alpha, 256, p.lda, 256, p.ldb, p.beta, 256, p.ldc, mode)
    assert plan["kernel_name"] == "tc2" and plan["tail_split"] > 1, plan
    A, B, C = synth.make(p)
    out1, ok1 = H.run_gpu(p, mode, A, B, C)
    out2, ok2 = H.run_gpu(p, mode, A, B, C)
    assert ok1 and ok2 and torch.equal(out1.view(torch.int32), out2.view(torch.int32))
    cref, den = H.reference_full(p, A, B, C)
    res = oracle.check(H.logical(p, out1), cref, den, oracle.TOL[mode])
    assert res["ok"], res
    assert H.padding_intact(p, out1, C)


@pytest.mark.parametrize("mnk,tb", [((3000, 1700, 777), "N"), ((2048, 1536, 512), "T"), ((700, 2600, 1300), "N"),
                                    ((1000, 1100, 300), "T"), ((5000, 1900, 600), "N")])
def test_pair_kernel_512_tiles(mnk, tb):
    """TF32 on SM pairs with 256x512 tiles (two N = 256 MMAs per k-step, one TMEM
    accumulator of 512 columns, each CTA's B columns staged as two halves of 128):
    ragged edges, N-major B as 3-D and as 2-D boxes, beta != 0, and a last-wave split
    (5000 x 1900: 80 tiles on 76 pairs)."""
    m, n, k = mnk
    p = synth.Problem(m, n, k, transb=tb, ldc=m + 3, alpha=1.25, beta=-0.5, dist="normal", seed=59)
    pg.load_library()
    try:
        pg.force_plan(512, 0)
        plan = pg.sgemm_plan("N", tb, m, n, k, p.alpha, 256, p.lda, 256, p.ldb, p.beta, 256, p.ldc, "tf32")
        assert plan["kernel_name"] == "tc2" and plan["bn"] == 512, plan
        if m == 5000:
            assert plan["tail_split"] > 1, plan
        _assert_ok(H.check_problem(p, "tf32"), "512 %s %s" % (mnk, tb))
    finally:
        pg.force_plan(0, 0)


@pytest.mark.parametrize("mnk,tb,ld_pad,beta", [((2000, 64, 4100), "N", 1, -0.5), ((1100, 100, 5000), "T", 0, 0.75),
                                                 ((4096, 128, 4096), "N", 2, 0.0), ((600, 40, 4500), "T", 3, 1.0)])
def test_single_sm_3xtf32_presplit_b(mnk, tb, ld_pad, beta):
    """3xTF32 on single SMs with B split by a pre-pass (four or more rows of tiles share
    B, K >= 4096): TMA brings B's remainders into the room in front of B and one
    N = 2 BN MMA takes big * [small | big]; ragged m, n and K, N-major B as 2-D boxes
    (n % 32 != 0), unaligned leading dimensions, beta 0 and not; bitwise repeatable."""
    m, n, k = mnk
    lda = m + ld_pad
    ldb = (k if tb == "N" else n) + ld_pad
    p = synth.Problem(m, n, k, transb=tb, lda=lda, ldb=ldb, ldc=m + 3, alpha=1.5, beta=beta, dist="normal", seed=61)
    plan = pg.sgemm_plan("N", tb, m, n, k, p.alpha, 256, p.lda, 256, p.ldb, p.beta, 256, p.ldc, "3xtf32")
    assert plan["kernel_name"] == "tc" and plan["prep_b_name"] == "split" and plan["bn"] <= 128, plan
    A, B, C = synth.make(p)
    out1, ok1 = H.run_gpu(p, "3xtf32", A, B, C)
    out2, ok2 = H.run_gpu(p, "3xtf32", A, B, C)
    assert ok1 and ok2 and torch.equal(out1.view(torch.int32), out2.view(torch.int32))
    cref, den = H.reference_full(p, A, B, C)
    res = oracle.check(H.logical(p, out1), cref, den, oracle.TOL["3xtf32"])
    assert res["ok"], res
    assert H.padding_intact(p, out1, C)


@pytest.mark.parametrize("mnk,bn", [((2500, 2000, 1000), 0), ((2560, 2048, 700), 0), ((4100, 2500, 600), 128),
                                    ((2048, 2048, 2048), 0), ((4000, 4090, 1000), 0)])
def test_last_wave_split_ffma(mnk, bn):
    """FFMA: the last partial wave's tiles run as 2-8 K slices (2048^3: 128 x 64 tiles,
    eight slices); the warp of the last slice to finish sums the partial blocks in
    slice order -- ragged edges, beta != 0, bitwise repeatable.  128-wide tiles are
    forced where the planner would take 64-wide ones."""
    m, n, k = mnk
    p = synth.Problem(m, n, k, ldc=m + 3, alpha=-1.25, beta=0.5, dist="normal", seed=47)
    A, B, C = synth.make(p)
    try:
        pg.force_plan(bn, 0)
        plan = pg.sgemm_plan("N", "N", m, n, k, p.alpha, 256, p.lda, 256, p.ldb, p.beta, 256, p.ldc, "ffma")
        assert plan["kernel_name"] == "ffma" and plan["tail_split"] > 1, plan
        assert bn == 0 or plan["bn"] == bn, plan
        out1, ok1 = H.run_gpu(p, "ffma", A, B, C)
        out2, ok2 = H.run_gpu(p, "ffma", A, B, C)
    finally:
        pg.force_plan(0, 0)
    assert ok1 and ok2 and torch.equal(out1.view(torch.int32), out2.view(torch.int32))
    cref, den = H.reference_full(p, A, B, C)
    res = oracle.check(H.logical(p, out1), cref, den, oracle.TOL["ffma"])
    assert res["ok"], res
    assert H.padding_intact(p, out1, C)


@pytest.mark.parametrize("mnk,ldc_pad,beta,bn", [((2048, 2048, 2048), 3, 0.5, 128), ((1000, 1300, 4000), 0, -1.0, 0),
                                                  ((1024, 1024, 8192), 4, 0.0, 128), ((12000, 50, 5200), 1, 1.5, 0),
                                                  ((1100, 700, 6000), 2, 0.25, 0), ((1250, 1650, 5000), 0, 0.0, 128)])
def test_ffma_stream_k(mnk, ldc_pad, beta, bn):
    """FFMA products whose tiles fill less than one wave of CTA slots run stream-K:
    every CTA takes an equal range of (tile, k-block) iterations across tile
    boundaries and a fix-up adds each tile's partial blocks in k order.  The
    planner's 64-wide tiles (three CTAs per SM) and, forced, the 128-wide ones;
    ragged edges, 2 to 6 segments per tile, beta 0 and not: the oracle within
    1e-5 and bitwise repeatable."""
    m, n, k = mnk
    p = synth.Problem(m, n, k, ldc=m + ldc_pad, alpha=0.75, beta=beta, dist="normal", seed=101)
    A, B, C = synth.make(p)
    try:
        pg.force_plan(bn, 0)
        plan = pg.sgemm_plan("N", "N", m, n, k, p.alpha, 256, p.lda, 256, p.ldb, p.beta, 256, p.ldc, "ffma")
        preps = (plan["prep_a_name"] != "none") + (plan["prep_b_name"] != "none")
        assert plan["sk_ctas"] > 0 and plan["launches"] == 2 + preps, plan
        assert plan["bn"] == (bn or 64), plan
        out1, ok1 = H.run_gpu(p, "ffma", A, B, C)
        out2, ok2 = H.run_gpu(p, "ffma", A, B, C)
    finally:
        pg.force_plan(0, 0)
    assert ok1 and ok2 and torch.equal(out1.view(torch.int32), out2.view(torch.int32))
    if m * n <= 2 ** 21:
        cref, den = H.reference_full(p, A, B, C)
        res = oracle.check(H.logical(p, out1), cref, den, oracle.TOL["ffma"])
    else:
        ii, jj = synth.sample_entries(p.m, p.n, count=4096, seed=12345)
        cref, den = H.reference_entries(p, A, B, C, ii, jj)
        res = oracle.check(H.gather(p, out1, ii, jj), cref, den, oracle.TOL["ffma"])
    assert res["ok"], res
    assert H.padding_intact(p, out1, C)


@pytest.mark.parametrize("mnk,trans,beta", [((8192, 128, 8192), "NN", 0.0), ((4096, 128, 8192), "NN", 1.5),
                                              ((128, 4096, 8192), "NN", -0.5), ((5100, 100, 9000), "TN", 0.25),
                                              ((5000, 120, 12000), "NT", 1.0), ((120, 5000, 9000), "TT", 0.0)])
def test_tc_stream_k(mnk, trans, beta):
    """3xTF32 on single SMs whose tiles would fill less than 90 % of the SMs runs
    stream-K: every SM an equal range of (tile, k-block) iterations, the
    accumulator drained to a partial block at each tile boundary and restarted,
    a fix-up adding the blocks in k order.  128-wide tiles, B split by the
    pre-pass or on chip, K- and N-major operands, ragged edges, beta 0 and not:
    the oracle within 1e-5, bitwise repeatable."""
    m, n, k = mnk
    p = synth.Problem(m, n, k, transa=trans[0], transb=trans[1], alpha=0.75, beta=beta, dist="normal", seed=113)
    p = p.with_(ldc=p.ldc + 3)
    plan = pg.sgemm_plan(p.transa, p.transb, m, n, k, p.alpha, 256, p.lda, 256, p.ldb, p.beta, 256, p.ldc, "3xtf32")
    assert plan["kernel_name"] == "tc" and plan["sk_ctas"] > 0, plan
    A, B, C = synth.make(p)
    out1, ok1 = H.run_gpu(p, "3xtf32", A, B, C)
    out2, ok2 = H.run_gpu(p, "3xtf32", A, B, C)
    assert ok1 and ok2 and torch.equal(out1.view(torch.int32), out2.view(torch.int32))
    if m * n <= 2 ** 20:
        cref, den = H.reference_full(p, A, B, C)
        res = oracle.check(H.logical(p, out1), cref, den, oracle.TOL["3xtf32"])
    else:
        ii, jj = synth.sample_entries(p.m, p.n, count=4096, seed=12345)
        cref, den = H.reference_entries(p, A, B, C, ii, jj)
        res = oracle.check(H.gather(p, out1, ii, jj), cref, den, oracle.TOL["3xtf32"])
    assert res["ok"], res
    assert H.padding_intact(p, out1, C)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("mnk", [(1, 1, 1), (1, 300, 7), (300, 1, 7), (5, 3, 1), (127, 129, 33), (131, 67, 255),
                                 (128, 256, 32), (257, 513, 1031), (64, 64, 200000), (160, 200, 300), (288, 130, 77),
                                 (416, 1000, 2048)])
def test_ragged_and_small(mode, mnk):
    m, n, k = mnk
    p = synth.Problem(m, n, k, lda=m + 1, ldb=k + 2, ldc=m + 3, alpha=1.25, beta=-0.75, dist="normal", seed=11)
    _assert_ok(H.check_problem(p, mode), "%s %s" % (mnk, mode))


@pytest.mark.parametrize("mode", MODES)
def test_forced_split_and_tiles(mode):
    p = synth.Problem(300, 200, 2000, alpha=1.0, beta=0.5, dist="normal", seed=13)
    try:
        for bn, split in ((64, 3), (128, 5), (256, 2), (64, 1)):
            pg.force_plan(bn, split)
            _assert_ok(H.check_problem(p, mode), "bn=%d split=%d %s" % (bn, split, mode))
    finally:
        pg.force_plan(0, 0)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("mnk", [(256, 64, 512), (600, 520, 300), (2048, 64, 4096)])
def test_special_values_match_in_kind(mode, mnk):
    """Infinities and NaN in A and in B, met by finite values, by zeros and by values
    whose TF32 remainder is zero, and (FFMA, 3xTF32) the largest float, whose TF32
    rounding would overflow: every non-finite result must match the oracle's in kind
    (NaN, or an infinity of the same sign) and every finite one stay within tolerance
    -- on the single-SM kernel (A split on chip, B on chip or by the pre-pass) and on
    SM pairs (both split by the pre-pass)."""
    m, n, k = mnk
    p = synth.Problem(m, n, k, alpha=1.0, beta=0.0, dist="normal", seed=73)
    A, B, C = synth.make(p)
    a = A[: p.lda * k].view(k, p.lda)    # a[q, i] = A(i, q)
    b = B[: p.ldb * n].view(n, p.ldb)    # b[j, q] = B(q, j)
    inf, nan = float("inf"), float("nan")
    a[3, 1], a[7, 5], a[11, 9] = inf, -inf, nan
    b[:, 3] = torch.round(b[:, 3] * 2)          # integers (zero remainder), some of them 0
    b[:, 7] = torch.round(b[:, 7] * 2)
    b[2, 20], b[4, 21], b[6, 20] = inf, nan, -inf
    if mode != "tf32":
        a[17, 13] = float(np.finfo(np.float32).max)
        b[:, 17] = b[:, 17].clamp(-1.0, 1.0) * 0.5   # keeps FLT_MAX * b inside FP32
    out, ok = H.run_gpu(p, mode, A, B, C)
    assert ok
    cref, den = H.reference_full(p, A, B, C)
    got = H.logical(p, out)
    assert (~np.isfinite(cref)).sum() > 0
    res = oracle.check(got, cref, den, oracle.TOL[mode])
    assert res["ok"], res


TF32_SUBNORMAL_ZERO = 2.0 ** -137  # below this, a TF32 operand part reads as zero


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("mnk", [(256, 64, 512), (512, 512, 1024), (128, 128, 4096)])
def test_subnormal_operands(mode, mnk):
    """Subnormal operands and products that underflow, on the single-SM kernel
    (256 x 64, 128 x 128) and on SM pairs (512 x 512):
      rows 0-7 of A   subnormals that TF32 holds exactly (j * 2^-136, j < 1024)
      rows 8-15       subnormals below 2^-137 (j * 2^-149, j < 4096)
      rows 16-23      normal values in [2^-117, 2^-116): 3xTF32 remainders subnormal
      rows 24-31      2^-70 scale, times columns 0-7 of B at 2^-70: products underflow
      cols 8-11 of B  TF32-exact subnormals; col 12 below 2^-137
      A(40, 3) = inf, met by B(3, 8) (a subnormal) and B(3, 12) (below 2^-137).
    FFMA is held to the oracle on these inputs.  The tensor-core modes read each
    operand (3xTF32: each of its two parts) in TF32, whose 10 mantissa-field bits
    hold a subnormal only to 2^-136: the tensor core does not flush what TF32
    holds (rows 0-7 and cols 8-11 are exact), values below 2^-137 read as zero,
    and 3xTF32 keeps 1e-5 for operands from 2^-118 up.  So they are held to the
    oracle on the same inputs with the values below 2^-137 set to zero.  Every
    check allows FP32's absolute underflow error, (k + 2) * 2^-149 per output."""
    m, n, k = mnk
    p = synth.Problem(m, n, k, alpha=1.0, beta=0.0, dist="normal", seed=89)
    A, B, C = synth.make(p)
    g = torch.Generator().manual_seed(90)
    a = A[: p.lda * k].view(k, p.lda)    # a[q, i] = A(i, q)
    b = B[: p.ldb * n].view(n, p.ldb)    # b[j, q] = B(q, j)

    def signs(*shape):
        return torch.where(torch.rand(*shape, generator=g) < 0.5, -1.0, 1.0)

    a[:, 0:8] = signs(k, 8) * torch.randint(1, 1024, (k, 8), generator=g).float() * 2.0 ** -136
    a[:, 8:16] = signs(k, 8) * torch.randint(1, 4096, (k, 8), generator=g).float() * 2.0 ** -149
    a[:, 16:24] = signs(k, 8) * (1.0 + torch.rand(k, 8, generator=g)) * 2.0 ** -117
    a[:, 24:32] = signs(k, 8) * (1.0 + torch.rand(k, 8, generator=g)) * 2.0 ** -70
    b[0:8, :] = signs(8, k) * (1.0 + torch.rand(8, k, generator=g)) * 2.0 ** -70
    b[8:12, :] = signs(4, k) * torch.randint(1, 1024, (4, k), generator=g).float() * 2.0 ** -136
    b[12, :] = signs(k) * torch.randint(1, 4096, (k,), generator=g).float() * 2.0 ** -149
    a[3, 40] = float("inf")
    assert bool((a[:, 8:16].abs() < TF32_SUBNORMAL_ZERO).all()) and bool((b[12].abs() < TF32_SUBNORMAL_ZERO).all())
    out, ok = H.run_gpu(p, mode, A, B, C)
    assert ok
    got = H.logical(p, out)
    if mode == "ffma":
        Ar, Br = A, B
    else:
        tiny = lambda t: (t.abs() < TF32_SUBNORMAL_ZERO) & (t != 0)  # noqa: E731
        Ar = torch.where(tiny(A), torch.zeros_like(A), A)
        Br = torch.where(tiny(B), torch.zeros_like(B), B)
    cref, den = H.reference_full(p, Ar, Br, C)
    res = oracle.check(got, cref, den, oracle.TOL[mode], floor=(k + 2) * 2.0 ** -149)
    assert res["ok"], res
    # the inputs did reach the cases: underflowing products, and a non-zero TF32-exact subnormal product
    assert 0 < np.abs(cref[24:32, 0:8]).max() < 2.0 ** -126
    assert np.isinf(cref[40, 8]) and np.isinf(got[40, 8])
    assert np.all(got[0:8, 13:20] != 0)


@pytest.mark.parametrize("bn", [64, 128, 256])
@pytest.mark.parametrize("m,ldc", [(1, 4), (31, 36), (33, 36), (100, 104), (160, 164), (167, 172), (256, 256),
                                   (167, 171)])
@pytest.mark.parametrize("beta,split", [(0.0, 1), (0.75, 1), (0.0, 3)])
def test_ffma_epilogue_paths(bn, m, ldc, beta, split):
    """The FFMA epilogue of a CTA that owns its tile or K slice: with beta = 0 and
    C 16-byte aligned with ldc % 4 == 0 the tile leaves as TMA boxes of 32 rows
    (the box that m cuts is stored by the threads); otherwise, or with K split,
    the threads store whole columns from the staged tile.  Rows cut inside a
    box, columns cut inside a tile, every tile width; every entry against the
    oracle, the ld gaps and the canaries untouched."""
    p = synth.Problem(m, 200, 70, ldc=ldc, alpha=-1.5, beta=beta, dist="normal", seed=31 + m)
    A, B, C = synth.make(p)
    try:
        pg.force_plan(bn, split)
        out, canaries = H.run_gpu(p, "ffma", A, B, C)
    finally:
        pg.force_plan(0, 0)
    cref, den = H.reference_full(p, A, B, C)
    res = oracle.check(H.logical(p, out), cref, den, oracle.TOL["ffma"])
    assert res["ok"], res
    assert canaries and H.padding_intact(p, out, C)
    assert pg.device_status() == 0


@pytest.mark.parametrize("mode", MODES)
def test_beta_zero_ignores_nan_c(mode):
    p = synth.Problem(200, 150, 100, alpha=1.0, beta=0.0, dist="normal", seed=17)
    A, B, C = synth.make(p)
    C.view(torch.int32).fill_(synth.NAN_BITS)
    out, ok = H.run_gpu(p, mode, A, B, C)
    cref, den = H.reference_full(p, A, B, C)
    assert ok and np.all(np.isfinite(H.logical(p, out)))
    assert oracle.check(H.logical(p, out), cref, den, oracle.TOL[mode])["ok"]


@pytest.mark.parametrize("mode", MODES)
def test_alpha_zero_and_k_zero(mode):
    p = synth.Problem(70, 50, 30, alpha=0.0, beta=-2.0, dist="normal", seed=19)
    A, B, C = synth.make(p)
    A.fill_(float("nan"))
    B.fill_(float("nan"))
    out, ok = H.run_gpu(p, mode, A, B, C)
    assert ok and np.array_equal(H.logical(p, out), -2.0 * H.logical(p, C))
    pk = p.with_(alpha=1.0, beta=0.0, k=0, ldb=1)
    out0, _ = H.run_gpu(pk, mode, A[:1], B[:50], C)
    assert np.all(H.logical(pk, out0) == 0.0)
    # beta == 1 with nothing to add leaves C untouched
    out1, _ = H.run_gpu(p.with_(beta=1.0), mode, A, B, C)
    assert torch.equal(out1.view(torch.int32), C.view(torch.int32))


@pytest.mark.parametrize("shape", [(70001, 5), (100, 3000), (33, 1)])
def test_scale_sweep_shapes(shape):
    """C = beta*C (alpha = 0) over tall, wide and tiny C: the sweep batches a
    thread's rows when it owns fewer columns than its batch, else its columns."""
    m, n = shape
    p = synth.Problem(m, n, 3, ldc=m + 3, alpha=0.0, beta=-1.25, dist="normal", seed=23)
    A, B, C = synth.make(p)
    out, ok = H.run_gpu(p, "tf32", A, B, C)
    assert ok and H.padding_intact(p, out, C)
    expect = np.float32(-1.25) * H.logical(p, C).astype(np.float32)  # one fp32 rounding, as on the GPU
    assert np.array_equal(H.logical(p, out), expect.astype(np.float64))


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("m,ldc", [(301, 304), (301, 303), (300, 300), (2, 8)])
@pytest.mark.parametrize("split", [2, 3, 9])
def test_splitk_reduce_rows_in_fours(mode, m, ldc, split):
    """The split-K reduction takes 4 rows of a column per thread: whole and ragged
    last chunks (m % 4 != 0), C read and written as float4 (16-byte aligned,
    ldc % 4 == 0) or element by element, beta != 0, and more slices than one
    batch of loads (9 > 8); bitwise repeatable."""
    p = synth.Problem(m, 77, 864, lda=m + 1, ldc=ldc, alpha=-0.75, beta=1.25, dist="normal", seed=97)  # 27 k-blocks
    A, B, C = synth.make(p)
    try:
        pg.force_plan(0, split)
        plan = pg.sgemm_plan("N", "N", p.m, p.n, p.k, p.alpha, 256, p.lda, 256, p.ldb, p.beta, 256, p.ldc, mode)
        assert plan["split_k"] == split, plan
        out1, ok1 = H.run_gpu(p, mode, A, B, C)
        out2, ok2 = H.run_gpu(p, mode, A, B, C)
    finally:
        pg.force_plan(0, 0)
    assert ok1 and ok2 and torch.equal(out1.view(torch.int32), out2.view(torch.int32))
    cref, den = H.reference_full(p, A, B, C)
    res = oracle.check(H.logical(p, out1), cref, den, oracle.TOL[mode])
    assert res["ok"], res
    assert H.padding_intact(p, out1, C)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("mnk", [(96, 3, 50000), (5000, 3, 70), (130, 130, 100000)])
def test_split_prep_and_reduce_shapes(mode, mnk):
    """Operand copies / TF32 splits of tall-narrow and short-wide operands, and
    split-K reductions over many slices, against the oracle (beta != 0)."""
    m, n, k = mnk
    p = synth.Problem(m, n, k, lda=m + 1, ldb=k + 1, ldc=m + 2, alpha=1.5, beta=0.5, dist="normal", seed=29)
    _assert_ok(H.check_problem(p, mode), "%s %s" % (mnk, mode))


def test_empty_sizes_are_no_ops():
    C = torch.full((16,), 3.0, device="cuda")
    pg.sgemm("N", "N", 0, 4, 4, 1.0, None, 1, None, 4, 0.0, C, 1)
    pg.sgemm("N", "N", 4, 0, 4, 1.0, None, 4, None, 4, 0.0, C, 4)
    torch.cuda.synchronize()
    assert torch.all(C == 3.0)


@pytest.mark.parametrize("mode", MODES)
def test_host_buffers_match_device_path(mode):
    p = synth.Problem(517, 389, 263, lda=520, ldb=270, ldc=530, alpha=0.75, beta=1.5, dist="normal", seed=23)
    A, B, C = synth.make(p)
    dev_out, _ = H.run_gpu(p, mode, A, B, C)
    Ch = C.clone().pin_memory()
    pg.sgemm_host("N", "N", p.m, p.n, p.k, p.alpha, A.pin_memory(), p.lda, B.pin_memory(), p.ldb, p.beta, Ch,
                  p.ldc, mode)
    assert torch.equal(Ch.view(torch.int32), dev_out.view(torch.int32))


@pytest.mark.parametrize("mode", MODES)
def test_host_buffers_pipelined_slabs(mode):
    """n >= 4096: sgemm_host overlaps the copies of column slabs with the arithmetic
    of their neighbours (internal copy streams); the result must still match the
    oracle, and the ld gap of the host C must stay untouched.  Two slabs of 3000
    columns here; A is prepared once for all slabs (3xTF32 on SM pairs: one split
    of A, then one split of each B slab and the slab's product)."""
    p = synth.Problem(2304, 6000, 300, lda=2307, ldb=301, ldc=2309, alpha=1.25, beta=0.5, dist="normal", seed=29)
    A, B, C = synth.make(p)
    Ch = C.clone().pin_memory()
    before = pg.launch_count()
    pg.sgemm_host("N", "N", p.m, p.n, p.k, p.alpha, A.pin_memory(), p.lda, B.pin_memory(), p.ldb, p.beta, Ch,
                  p.ldc, mode)
    launched = pg.launch_count() - before
    assert launched == {"ffma": 2, "tf32": 2, "3xtf32": 5}[mode], launched
    cref, den = H.reference_full(p, A, B, C)
    res = oracle.check(H.logical(p, Ch), cref, den, oracle.TOL[mode])
    assert res["ok"], res
    assert H.padding_intact(p, Ch, C)
    # pageable host memory takes the same path
    Cp = C.clone()
    pg.sgemm_host("N", "N", p.m, p.n, p.k, p.alpha, A, p.lda, B, p.ldb, p.beta, Cp, p.ldc, mode)
    assert oracle.check(H.logical(p, Cp), cref, den, oracle.TOL[mode])["ok"]


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("q,tb,mnk", [(3.0, "N", (700, 530, 900)), (1.5, "T", (300, 97, 2000)),
                                      (-1.0, "N", (700, 530, 900)), (7.0, "N", (2304, 6000, 300))])
def test_host_split(mode, q, tb, mnk):
    """The hybrid CPU + GPU column split of the host entry: the last
    floor(n / (q + 1)) columns of C on the host co-worker, the rest on the GPU
    path (with n >= 4096 its pipelined column slabs), concurrently; a fixed
    ratio, and the automatic one re-measured by the call.  The whole C matches
    the oracle, its ld gaps stay untouched; the asynchronous entry gives the same
    result after a stream synchronisation."""
    m, n, k = mnk
    p = synth.Problem(m, n, k, transb=tb, ldc=m + 5, alpha=1.25, beta=0.5, dist="normal", seed=103)
    p = p.with_(lda=p.lda + 3)
    A, B, C = synth.make(p)
    Ah, Bh = A.pin_memory(), B.pin_memory()
    Ch, Ca = C.clone().pin_memory(), C.clone().pin_memory()
    try:
        pg.set_host_split(q)
        before = pg.host_split_ratio(mode)
        pg.sgemm_host(p.transa, p.transb, m, n, k, p.alpha, Ah, p.lda, Bh, p.ldb, p.beta, Ch, p.ldc, mode)
        if q < 0:
            assert pg.host_split_ratio(mode) != before  # re-measured from this call's two parts
        s = torch.cuda.Stream()
        pg.sgemm_host_async(p.transa, p.transb, m, n, k, p.alpha, Ah, p.lda, Bh, p.ldb, p.beta, Ca, p.ldc, mode, s)
        s.synchronize()
    finally:
        pg.set_host_split(0.0)
    cref, den = H.reference_full(p, A, B, C)
    for out in (Ch, Ca):
        res = oracle.check(H.logical(p, out), cref, den, oracle.TOL[mode])
        assert res["ok"], res
        assert H.padding_intact(p, out, C)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("weights,transb", [([1, 1, 1, 1], "N"), ([15, 1], "N"), ([3, 2], "T")])
def test_column_slabs_through_the_library(mode, weights, transb):
    """The column partition of the multi-worker path, each slab computed by the
    library: a slab of C needs all of A and only its own columns of B (rows of
    a transposed B), so the slabs are independent products.  Stitched, they
    match the oracle on the whole product, and bit for bit with integer inputs
    (every sum exact, whichever plan each slab gets)."""
    from precision_gemm_gb300.partition import column_slabs, slab_views
    for dist_name in ("normal", "int"):
        p = synth.Problem(3000, 1500, 777, transb=transb, lda=3013, ldc=3005, alpha=1.5, beta=-0.5, dist=dist_name,
                          seed=107)
        A, B, C = synth.make(p)
        dA, dB, dC = A.cuda(), B.cuda(), C.cuda()
        for j0, j1 in column_slabs(p.n, weights):
            b_off, c_off, w = slab_views(j0, j1, p.ldb, p.ldc, transb)
            if w == 0:
                continue
            pg.sgemm("N", transb, p.m, w, p.k, p.alpha, dA, p.lda, dB.data_ptr() + 4 * b_off, p.ldb, p.beta,
                     dC.data_ptr() + 4 * c_off, p.ldc, mode)
        torch.cuda.synchronize()
        out = dC.cpu()
        cref, den = H.reference_full(p, A, B, C)
        if dist_name == "int":
            assert np.array_equal(H.logical(p, out), cref)
        else:
            res = oracle.check(H.logical(p, out), cref, den, oracle.TOL[mode])
            assert res["ok"], res
        assert H.padding_intact(p, out, C)


@pytest.mark.parametrize("mode", MODES)
def test_launch_counter_counts_kernels(mode):
    for p in (synth.Problem(256, 256, 256), synth.Problem(4096, 4096, 512)):
        A, B, C = synth.make(p)
        plan = pg.sgemm_plan("N", "N", p.m, p.n, p.k, p.alpha, 256, p.lda, 256, p.ldb, p.beta, 256, p.ldc, mode,
                             num_sms=torch.cuda.get_device_properties(0).multi_processor_count)
        before = pg.launch_count()
        H.run_gpu(p, mode, A, B, C)
        assert pg.launch_count() - before == plan["launches"]


# ------------------------------------------------------------ failure detection

@pytest.mark.parametrize("mode", MODES)
def test_bounded_wait_reports_timeout(mode):
    """The operand loader is told to issue nothing, so every other wait in the
    CTA runs out after the (short) limit; the kernel records SGEMM_ERR_TIMEOUT,
    exits cleanly, and the context stays usable for the next call."""
    p = synth.Problem(256, 256, 256, seed=3)
    A, B, C = synth.make(p)
    assert pg.device_status() == 0
    old = pg.set_wait_timeout(20_000_000)  # 20 ms
    pg.debug_flags(pg.SGEMM_DEBUG_STALL_PRODUCER)
    try:
        H.run_gpu(p, mode, A, B, C)
    finally:
        pg.debug_flags(0)
        pg.set_wait_timeout(old)
    assert pg.device_status(clear=True) == pg.SGEMM_ERR_TIMEOUT
    assert pg.device_status() == 0
    _assert_ok(H.check_problem(p, mode), "after a timeout " + mode)


@pytest.mark.parametrize("mode", MODES)
def test_injected_host_faults_fail_cleanly(mode):
    """Failures injected on the host (an allocation that fails, a tensor map that
    cannot be encoded) come back as SGEMM_ERR_ALLOC / SGEMM_ERR_TENSOR_MAP from
    the call itself, leave C untouched and the context usable: the next call on
    the same stream is correct."""
    # lda not a multiple of 4: the call needs workspace for an operand copy
    p = synth.Problem(300, 200, 5000, lda=301, alpha=1.0, beta=0.5, dist="normal", seed=127)
    A, B, C = synth.make(p)
    dA, dB, dC = A.cuda(), B.cuda(), C.cuda()
    s = torch.cuda.Stream()  # a fresh stream: its workspace must be allocated
    old = pg.debug_flags(0)
    try:
        for flag, code in ((pg.SGEMM_DEBUG_FAIL_ALLOC, pg.SGEMM_ERR_ALLOC),
                           (pg.SGEMM_DEBUG_FAIL_TENSOR_MAP, pg.SGEMM_ERR_TENSOR_MAP)):
            pg.debug_flags(flag)
            with pytest.raises(pg.SgemmError) as e:
                pg.sgemm("N", "N", p.m, p.n, p.k, p.alpha, dA, p.lda, dB, p.ldb, p.beta, dC, p.ldc, mode, s)
            assert e.value.code == code and "injected" in str(e.value)
    finally:
        pg.debug_flags(old)
    s.synchronize()
    assert torch.equal(dC.cpu().view(torch.int32), C.view(torch.int32))
    pg.sgemm("N", "N", p.m, p.n, p.k, p.alpha, dA, p.lda, dB, p.ldb, p.beta, dC, p.ldc, mode, s)
    s.synchronize()
    cref, den = H.reference_full(p, A, B, C)
    assert oracle.check(H.logical(p, dC.cpu()), cref, den, oracle.TOL[mode])["ok"]
    assert pg.device_status() == 0
