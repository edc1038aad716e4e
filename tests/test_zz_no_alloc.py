"""sgemm_noalloc: the entry point for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc -- their device memory is reserved up front
by another allocator, or they run in a latency-critical loop where an
allocation (which may synchronise the device) is not allowed.  sgemm_noalloc
keeps its only scratch, the split-K partial sums, in a fixed device array, so
it never allocates.  These tests call it through the C ABI and compare it with
the ordinary sgemm entry point on two calls in a row, within the normalised
error tolerance the parity tests use; they also check its documented refusals.
The file is named to run last, so a stop at the first failure has already run
every other test; it passes alone in a fresh process as well.
"""
import numpy as np
import pytest
import torch

import oracle
import precision_gemm_gb300 as pg
from precision_gemm_gb300 import synth
from tests import _harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _plain_plan():
    pg.load_library()
    pg.force_plan(0, 0)
    yield
    pg.force_plan(0, 0)


def _num_sms():
    return torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count


@pytest.mark.parametrize("mode", ("ffma", "tf32"))
def test_noalloc_matches_sgemm_on_two_calls_in_a_row(mode):
    for seed in (1, 2):
        # A skinny-K product, so the call uses split-K and therefore the scratch array.
        p = synth.Problem(192, 160, 65536, alpha=1.25, beta=0.5, dist="normal", seed=seed)
        A, B, C = synth.make(p)
        plan = pg.sgemm_plan("N", "N", p.m, p.n, p.k, p.alpha, 256, p.lda, 256, p.ldb, p.beta, 256, p.ldc, mode,
                             num_sms=_num_sms())
        assert plan["split_k"] > 1
        dA, dB = A.cuda(), B.cuda()
        c_ref = C.cuda()
        c_new = C.cuda()
        pg.sgemm("N", "N", p.m, p.n, p.k, p.alpha, dA, p.lda, dB, p.ldb, p.beta, c_ref, p.ldc, mode)
        pg.sgemm_noalloc("N", "N", p.m, p.n, p.k, p.alpha, dA, p.lda, dB, p.ldb, p.beta, c_new, p.ldc, mode)
        torch.cuda.synchronize()
        got = H.logical(p, c_new.cpu())
        ref = H.logical(p, c_ref.cpu())
        _, den = H.reference_full(p, A, B, C)
        res = oracle.check(got, ref, den, oracle.TOL[mode])
        assert res["ok"], (mode, seed, res)
        # and both agree with the oracle itself
        cref, den = H.reference_full(p, A, B, C)
        assert oracle.check(got, cref, den, oracle.TOL[mode])["ok"]
    assert pg.device_status() == 0


def test_noalloc_second_call_with_another_layout():
    """The shared array keeps whatever the last call left in it.  A second call
    with another m (so another row pitch of the partial sums) and another number
    of K slices must still match the oracle: every partial it reads it wrote."""
    shapes = [(192, 160, 65536, 1), (100, 70, 40000, 2), (192, 160, 65536, 3)]
    splits = []
    for m, n, k, seed in shapes:
        p = synth.Problem(m, n, k, alpha=0.75, beta=-1.5, dist="normal", seed=seed)
        plan = pg.sgemm_plan("N", "N", m, n, k, p.alpha, 256, p.lda, 256, p.ldb, p.beta, 256, p.ldc, "ffma",
                             num_sms=_num_sms())
        assert plan["split_k"] > 1
        splits.append(plan["split_k"])
        A, B, C = synth.make(p)
        dA, dB, dC = A.cuda(), B.cuda(), C.cuda()
        pg.sgemm_noalloc("N", "N", m, n, k, p.alpha, dA, p.lda, dB, p.ldb, p.beta, dC, p.ldc, "ffma")
        torch.cuda.synchronize()
        cref, den = H.reference_full(p, A, B, C)
        res = oracle.check(H.logical(p, dC.cpu()), cref, den, oracle.TOL["ffma"])
        assert res["ok"], ((m, n, k), res)
    assert splits[0] != splits[1]


@pytest.mark.parametrize("mode", ("ffma", "tf32"))
def test_noalloc_where_sgemm_splits_the_last_wave(mode):
    """sgemm splits a last wave at most half full along K; sgemm_noalloc does not
    (it would need scratch for the partial blocks).  The two agree within the
    mode's tolerance."""
    p = synth.Problem(2500, 2000, 1000, alpha=-1.25, beta=0.5, dist="normal", seed=47)
    plan = pg.sgemm_plan("N", "N", p.m, p.n, p.k, p.alpha, 256, p.lda, 256, p.ldb, p.beta, 256, p.ldc, mode,
                         num_sms=_num_sms())
    assert plan["tail_split"] > 1, plan
    A, B, C = synth.make(p)
    dA, dB = A.cuda(), B.cuda()
    c_ref, c_new = C.cuda(), C.cuda()
    pg.sgemm("N", "N", p.m, p.n, p.k, p.alpha, dA, p.lda, dB, p.ldb, p.beta, c_ref, p.ldc, mode)
    pg.sgemm_noalloc("N", "N", p.m, p.n, p.k, p.alpha, dA, p.lda, dB, p.ldb, p.beta, c_new, p.ldc, mode)
    torch.cuda.synchronize()
    cref, den = H.reference_full(p, A, B, C)
    got = H.logical(p, c_new.cpu())
    assert oracle.check(got, H.logical(p, c_ref.cpu()), den, oracle.TOL[mode])["ok"]
    assert oracle.check(got, cref, den, oracle.TOL[mode])["ok"]


def test_noalloc_without_split_and_trivial_calls():
    p = synth.Problem(300, 200, 100, alpha=1.0, beta=-1.0, dist="normal", seed=4)
    A, B, C = synth.make(p)
    dA, dB, dC = A.cuda(), B.cuda(), C.cuda()
    pg.sgemm_noalloc("N", "N", p.m, p.n, p.k, p.alpha, dA, p.lda, dB, p.ldb, p.beta, dC, p.ldc, "ffma")
    # alpha = 0: C = beta * C, nothing read from A or B
    d2 = C.cuda()
    pg.sgemm_noalloc("N", "N", p.m, p.n, p.k, 0.0, None, p.lda, None, p.ldb, 2.0, d2, p.ldc, "tf32")
    # a call that only scales C is not held to the limits on how A and B are read:
    # transposed A, an ld that is not a multiple of 4, 3xTF32
    d3 = C.cuda()
    pg.sgemm_noalloc("T", "T", p.m, p.n, p.k, 0.0, None, p.k + 1, None, p.n + 3, -0.5, d3, p.ldc, "3xtf32")
    torch.cuda.synchronize()
    cref, den = H.reference_full(p, A, B, C)
    assert oracle.check(H.logical(p, dC.cpu()), cref, den, oracle.TOL["ffma"])["ok"]
    assert np.array_equal(H.logical(p, d2.cpu()), 2.0 * H.logical(p, C))
    assert np.array_equal(H.logical(p, d3.cpu()), -0.5 * H.logical(p, C))


def test_noalloc_refuses_what_it_cannot_do_without_allocating():
    # Buffers cover the full extents of the refused 512 x 512 x 65536 call (A 512 x
    # 65536, B 65536 x 512), so that even a call the library wrongly let through
    # would stay inside its allocations.
    m = n = 512
    k = 65536
    dA = torch.zeros(m * k, device="cuda")
    dB = torch.zeros(k * n, device="cuda")
    dC = torch.zeros(m * n, device="cuda")
    c0 = dC.clone()
    # more K slices than the fixed array holds: 64 * 512 * 512 * 4 B = 64 MiB > 16 MiB
    pg.force_plan(0, 64)
    before = pg.launch_count()
    with pytest.raises(pg.SgemmError) as e:
        pg.sgemm_noalloc("N", "N", m, n, k, 1.0, dA, m, dB, k, 0.0, dC, m, "ffma")
    assert e.value.code == pg.SGEMM_ERR_SCRATCH and "16777216" in str(e.value)
    assert pg.launch_count() == before
    pg.force_plan(0, 0)
    # limits on how A and B are read, reported in signature order
    for kw, code in ((dict(mode="3xtf32"), -14), (dict(transa="T"), -1), (dict(transb="T"), -2),
                     (dict(lda=513), -8), (dict(A=dA.data_ptr() + 4), -7), (dict(transa="T", lda=513), -1)):
        args = dict(transa="N", transb="N", mode="ffma", lda=512, A=dA)
        args.update(kw)
        with pytest.raises(pg.SgemmError) as e:
            pg.sgemm_noalloc(args["transa"], args["transb"], 256, 256, 256, 1.0, args["A"], args["lda"], dB, 512,
                             0.0, dC, 512, args["mode"])
        assert e.value.code == code, kw
    torch.cuda.synchronize()
    assert torch.equal(dC, c0)
