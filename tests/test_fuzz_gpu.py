"""Seeded random problems through the C ABI against the oracle, entry by entry.

Each case draws sizes (1..600, including 1 and tile-edge neighbours), both
operand orientations, leading-dimension padding, alpha/beta (including 0 and
negative values) and a plan override (tile width, split-K count), so that the
kernels' edge predication, the in-place transposed reads, the operand copies,
the split-K and last-wave paths and the epilogue variants meet combinations
no hand-written case lists.  The draws are fixed by the seed: a failure names a
reproducible case.
"""
import numpy as np
import pytest

import oracle
import precision_gemm_gb300 as pg
from precision_gemm_gb300 import synth
from tests import _harness as H

pytestmark = pytest.mark.gpu
MODES = ("ffma", "tf32", "3xtf32")


def _cases(count=60, seed=2026):
    rng = np.random.default_rng(seed)
    edge = [1, 2, 31, 32, 33, 63, 64, 65, 127, 128, 129, 255, 256, 257]
    out = []
    for c in range(count):
        dims = [int(rng.choice(edge)) if rng.random() < 0.4 else int(rng.integers(1, 601)) for _ in range(3)]
        m, n, k = dims
        ta, tb = ("N", "T")[int(rng.integers(0, 2))], ("N", "T")[int(rng.integers(0, 2))]
        pads = [int(rng.integers(0, 6)) for _ in range(3)]
        alpha = float(rng.choice([1.0, -0.5, 2.25, 0.0], p=[0.4, 0.25, 0.25, 0.1]))
        beta = float(rng.choice([0.0, 1.0, -1.5], p=[0.4, 0.3, 0.3]))
        bn = int(rng.choice([0, 0, 64, 128, 256]))
        split = int(rng.choice([0, 0, 0, 1, 2, 3, 7]))
        out.append((c, m, n, k, ta, tb, pads, alpha, beta, bn, split))
    return out


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("case", _cases(), ids=lambda c: "case%d" % c[0])
def test_random_problem(mode, case):
    c, m, n, k, ta, tb, pads, alpha, beta, bn, split = case
    p = synth.Problem(m, n, k, transa=ta, transb=tb, alpha=alpha, beta=beta, dist="normal", seed=1000 + c)
    p = p.with_(lda=p.lda + pads[0], ldb=p.ldb + pads[1], ldc=p.ldc + pads[2])
    pg.load_library()
    try:
        pg.force_plan(bn, split)
        A, B, C = synth.make(p)
        out, canaries = H.run_gpu(p, mode, A, B, C)
    finally:
        pg.force_plan(0, 0)
    cref, den = H.reference_full(p, A, B, C)
    res = oracle.check(H.logical(p, out), cref, den, oracle.TOL[mode])
    assert res["ok"], (case, mode, res)
    assert canaries and H.padding_intact(p, out, C), (case, mode)
    assert pg.device_status() == 0
