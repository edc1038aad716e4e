"""Seeded synthetic inputs for the tests, the benchmark and the smoke check.

This module holds no GEMM arithmetic: only random draws, NaN padding of the
leading-dimension gaps, and the choice of which output entries a sampled check
looks at.  Both the CUDA path and the CPU oracle read the same buffers it makes.

Workloads follow the pages: square fp32 matrices with uniform or normal entries
("V3. Vectorized and double buffer", section 3 runs N x N; "HPC - Lecture 13 -
MatMat GPU" sweeps square N), extended to the shapes the acceptance suite names
(ragged sizes, padded leading dimensions, skinny products).

Draw order is fixed: A, then B, then Cin, each as its FULL storage buffer
(ld * cols values, column-major), from one ``torch.Generator`` seeded with the
problem's seed.  Padding rows (ld > rows) are then overwritten with the quiet-NaN
bit pattern 0x7fc00000, so any read or write of the padding is visible.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np
import torch

NAN_BITS = 0x7FC00000


def storage(rows: int, cols: int, ld: int, dist: str, gen: torch.Generator) -> torch.Tensor:
    """One column-major fp32 storage buffer of ld*cols elements on the CPU.

    Element (i, j) sits at i + j*ld.  Rows i >= rows are padding and hold NAN_BITS.
    dist: 'uniform' = U[-1, 1); 'normal' = N(0, 1); 'int' = integers in [-8, 8];
    'ones' = all 1.0; 'zeros' = all 0.0.
    """
    if ld < max(1, rows):
        raise ValueError("ld %d < rows %d" % (ld, rows))
    count = ld * cols
    if dist == "uniform":
        x = torch.rand(count, generator=gen, dtype=torch.float32).mul_(2.0).sub_(1.0)
    elif dist == "normal":
        x = torch.randn(count, generator=gen, dtype=torch.float32)
    elif dist == "int":
        x = torch.randint(-8, 9, (count,), generator=gen, dtype=torch.int32).to(torch.float32)
    elif dist == "ones":
        x = torch.ones(count, dtype=torch.float32)
    elif dist == "zeros":
        x = torch.zeros(count, dtype=torch.float32)
    else:
        raise ValueError("unknown distribution %r" % dist)
    if ld > rows and cols > 0:
        x.view(torch.int32).view(cols, ld)[:, rows:] = NAN_BITS
    return x


@dataclass(frozen=True)
class Problem:
    """One GEMM instance: C = alpha*op(A)*op(B) + beta*C.

    layout 'col' means BLAS column-major storage; 'row' means row-major storage
    (A is m x k with row stride lda, and so on), which the binding maps onto the
    column-major call by swapping operands.
    """
    m: int
    n: int
    k: int
    transa: str = "N"
    transb: str = "N"
    lda: int = 0
    ldb: int = 0
    ldc: int = 0
    alpha: float = 1.0
    beta: float = 0.0
    dist: str = "uniform"
    c_dist: str = ""
    seed: int = 0
    layout: str = "col"

    def __post_init__(self):
        object.__setattr__(self, "lda", self.lda or self.a_dims()[0])
        object.__setattr__(self, "ldb", self.ldb or self.b_dims()[0])
        object.__setattr__(self, "ldc", self.ldc or self.c_dims()[0])
        if not self.c_dist:
            object.__setattr__(self, "c_dist", self.dist)

    # Storage shapes as (contiguous extent, other extent), i.e. (rows, cols) of the
    # column-major buffer that holds the operand.
    def a_dims(self):
        notr = self.transa in "Nn"
        if self.layout == "col":
            return (self.m, self.k) if notr else (self.k, self.m)
        return (self.k, self.m) if notr else (self.m, self.k)

    def b_dims(self):
        notr = self.transb in "Nn"
        if self.layout == "col":
            return (self.k, self.n) if notr else (self.n, self.k)
        return (self.n, self.k) if notr else (self.k, self.n)

    def c_dims(self):
        return (self.m, self.n) if self.layout == "col" else (self.n, self.m)

    def flops(self) -> int:
        return 2 * self.m * self.n * self.k

    def with_(self, **kw) -> "Problem":
        return replace(self, **kw)


def make(p: Problem):
    """(A, B, C) CPU fp32 storage buffers for problem p (see the module docstring)."""
    gen = torch.Generator().manual_seed(p.seed)
    ra, ca = p.a_dims()
    rb, cb = p.b_dims()
    rc, cc = p.c_dims()
    A = storage(ra, ca, p.lda, p.dist, gen)
    B = storage(rb, cb, p.ldb, p.dist, gen)
    C = storage(rc, cc, p.ldc, p.c_dist, gen)
    return A, B, C


def sample_entries(m: int, n: int, count: int = 4096, seed: int = 12345,
                   edges=(64, 128, 256)):
    """Output entries a sampled check evaluates: `count` uniform picks without
    replacement, plus the four corners, the last row and column (strided when
    long), and strips at multiples of each tile edge (i or j in {t-1, t})."""
    rng = np.random.default_rng(seed)
    total = m * n
    if total == 0:
        return np.zeros(0, np.int64), np.zeros(0, np.int64)
    picks = rng.choice(total, size=min(count, total), replace=False)
    ii = list(picks % m)
    jj = list(picks // m)
    extra = [(0, 0), (m - 1, 0), (0, n - 1), (m - 1, n - 1)]
    step_r = max(1, m // 64)
    step_c = max(1, n // 64)
    extra += [(i, n - 1) for i in range(0, m, step_r)]
    extra += [(m - 1, j) for j in range(0, n, step_c)]
    for t in edges:
        rows = sorted({x for q in range(t, m + 1, t) for x in (q - 1, q) if x < m})
        cols = sorted({x for q in range(t, n + 1, t) for x in (q - 1, q) if x < n})
        rows = rows[:: max(1, len(rows) // 16)]
        cols = cols[:: max(1, len(cols) // 16)]
        for r in rows:
            extra += [(r, int(j)) for j in rng.integers(0, n, size=4)]
        for c in cols:
            extra += [(int(i), c) for i in rng.integers(0, m, size=4)]
    for i, j in extra:
        ii.append(i)
        jj.append(j)
    pairs = np.unique(np.stack([np.asarray(ii, np.int64), np.asarray(jj, np.int64)], 1), axis=0)
    return pairs[:, 0].copy(), pairs[:, 1].copy()


# The acceptance workloads, by name (sizes, distributions and scalars of the suite).
def config_problems():
    """Name -> Problem for every workload of the acceptance suite."""
    P = {}
    P["c1_256"] = Problem(256, 256, 256, alpha=1.0, beta=0.0, dist="uniform", seed=0)
    for N in (1024, 2048, 4096):
        P["c2_rm%d" % N] = Problem(N, N, N, alpha=1.0, beta=0.0, dist="uniform", seed=0,
                                  layout="row")
    P["c3_ragged"] = Problem(3000, 1500, 777, lda=3013, ldb=784, ldc=3005, alpha=1.5,
                             beta=-0.5, dist="normal", seed=0)
    for N in (8192, 16384):
        P["c4_%d" % N] = Problem(N, N, N, alpha=1.0, beta=1.0, dist="uniform", seed=0)
    P["c5a_16384x16384x64"] = Problem(16384, 16384, 64, dist="normal", seed=0)
    P["c5b_128x128x262144"] = Problem(128, 128, 262144, dist="normal", seed=0)
    P["c5c_8192x64x8192"] = Problem(8192, 64, 8192, dist="normal", seed=0)
    return P
