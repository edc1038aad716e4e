"""Test-side glue: run a synth.Problem through the CUDA library and through the
oracle, and compare.  No GEMM arithmetic here; the oracle computes references."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import precision_gemm_gb300 as pg
from precision_gemm_gb300 import synth

CANARY_BITS = 0x7F8CA1A5  # a signalling-NaN pattern no kernel writes
GUARD = 64                # guard words before and after every device buffer


class Guarded:
    """A device copy of a CPU storage buffer with canary words on both sides."""

    def __init__(self, host: torch.Tensor, device="cuda"):
        n = host.numel()
        self.full = torch.empty(n + 2 * GUARD, dtype=torch.float32, device=device)
        self.full.view(torch.int32).fill_(CANARY_BITS)
        self.full[GUARD:GUARD + n].copy_(host)
        self.n = n

    @property
    def t(self) -> torch.Tensor:
        return self.full[GUARD:GUARD + self.n]

    def canaries_intact(self) -> bool:
        bits = self.full.view(torch.int32)
        return bool(torch.all(bits[:GUARD] == CANARY_BITS)) and bool(torch.all(bits[GUARD + self.n:] == CANARY_BITS))


def run_gpu(p: synth.Problem, mode, A: torch.Tensor, B: torch.Tensor, C: torch.Tensor, stream=None,
            guards: bool = True):
    """Run p on the device; returns (C storage on the CPU, canaries_ok)."""
    gA, gB, gC = Guarded(A), Guarded(B), Guarded(C)
    if p.layout == "col":
        pg.sgemm(p.transa, p.transb, p.m, p.n, p.k, p.alpha, gA.t, p.lda, gB.t, p.ldb, p.beta, gC.t, p.ldc,
                 mode, stream)
    else:
        if p.transa not in "Nn" or p.transb not in "Nn":
            raise ValueError("row-major problems are tested without transposes")
        pg.sgemm_rm(p.m, p.n, p.k, p.alpha, gA.t, p.lda, gB.t, p.ldb, p.beta, gC.t, p.ldc, mode, stream)
    torch.cuda.synchronize()
    ok = gA.canaries_intact() and gB.canaries_intact() and gC.canaries_intact()
    return gC.t.cpu(), ok


def _oracle_args(p: synth.Problem, A, B, C):
    """The column-major oracle call that evaluates problem p.

    Row-major storage of X is the column-major storage of X^T, so a row-major
    problem is evaluated as C^T = B^T * A^T (m and n swapped); the oracle's
    transpose identities pin that rewriting."""
    if p.layout == "col":
        return (p.transa, p.transb, p.m, p.n, p.k, p.alpha, A, p.lda, B, p.ldb, p.beta, C, p.ldc), False
    return ("N", "N", p.n, p.m, p.k, p.alpha, B, p.ldb, A, p.lda, p.beta, C, p.ldc), True


def logical(p: synth.Problem, Cst: torch.Tensor) -> np.ndarray:
    """The m x n result (float64) read out of a C storage buffer."""
    rows, cols = p.c_dims()
    mat = Cst.numpy().reshape(cols, p.ldc)[:, :rows].T.astype(np.float64)
    return mat if p.layout == "col" else mat.T


def reference_full(p: synth.Problem, A, B, C, threads: int = 0):
    """(Cref, den) for every entry, as (m, n) arrays."""
    args, swapped = _oracle_args(p, A, B, C)
    cref, den = oracle.Oracle().full(*args, threads=threads)
    return (cref.T, den.T) if swapped else (cref, den)


def reference_entries(p: synth.Problem, A, B, C, ii, jj, threads: int = 0):
    args, swapped = _oracle_args(p, A, B, C)
    if swapped:
        return oracle.Oracle().entries(*args, jj, ii, threads=threads)
    return oracle.Oracle().entries(*args, ii, jj, threads=threads)


def gather(p: synth.Problem, Cst: torch.Tensor, ii, jj) -> np.ndarray:
    flat = Cst.numpy()
    if p.layout == "col":
        return flat[ii + jj * p.ldc].astype(np.float64)
    return flat[jj + ii * p.ldc].astype(np.float64)


def padding_intact(p: synth.Problem, Cst: torch.Tensor, Cin: torch.Tensor) -> bool:
    """Bits of the ld gaps of C are unchanged."""
    rows, cols = p.c_dims()
    if p.ldc == rows:
        return True
    a = Cst.view(torch.int32).view(cols, p.ldc)[:, rows:]
    b = Cin.view(torch.int32).view(cols, p.ldc)[:, rows:]
    return bool(torch.equal(a, b))


def check_problem(p: synth.Problem, mode: str, sample: int = 0, threads: int = 0, seed_entries: int = 12345):
    """Run p in `mode` and compare with the oracle (all entries, or `sample`
    sampled ones plus tile edges).  Returns the oracle.check dict plus flags."""
    A, B, C = synth.make(p)
    out, canaries = run_gpu(p, mode, A, B, C)
    if sample:
        ii, jj = synth.sample_entries(p.m, p.n, count=sample, seed=seed_entries)
        cref, den = reference_entries(p, A, B, C, ii, jj, threads=threads)
        got = gather(p, out, ii, jj)
    else:
        cref, den = reference_full(p, A, B, C, threads=threads)
        got = logical(p, out)
    res = oracle.check(got, cref, den, oracle.TOL[mode])
    res["canaries"] = canaries
    res["padding"] = padding_intact(p, out, C)
    return res
