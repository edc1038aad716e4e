"""Column partition of C across workers (host arithmetic only).

"HPC - Lecture 13 - MatMat GPU", section "Load distribution" and the hybrid
function matmatgpu3, splits the columns of C between two devices in proportion
to their speed (GPU share Q/(Q+1), CPU share 1/(Q+1), Q = 15).  Each column
slab of C needs all of A and only its own columns of B, so the slabs are
independent problems: no exchange between workers on the data path.

The lecture's integer formulas (N3*Q/(Q+1) and N3/(Q+1)) can leave columns
unassigned when N3 is not a multiple of Q+1; here the slab boundaries are
rounded cumulative shares, so the slabs always cover every column exactly once.
"""
from __future__ import annotations


def column_slabs(n: int, weights) -> list[tuple[int, int]]:
    """Contiguous [j0, j1) slabs of range(n), one per weight, sizes proportional
    to the weights (non-negative, not all zero); together they cover range(n)."""
    w = [float(x) for x in weights]
    if n < 0 or not w or any(x < 0 for x in w) or sum(w) <= 0:
        raise ValueError("need n >= 0 and non-negative weights with a positive sum")
    total = sum(w)
    bounds, acc = [0], 0.0
    for x in w[:-1]:
        acc += x
        bounds.append(int(round(n * acc / total)))
    bounds.append(n)
    return [(bounds[i], bounds[i + 1]) for i in range(len(w))]


def even_slabs(n: int, parts: int) -> list[tuple[int, int]]:
    return column_slabs(n, [1.0] * parts)


def slab_views(j0: int, j1: int, ldb: int, ldc: int, transb: str = "N"):
    """Element offsets of the slab's first column in B and C, and its width, for a
    column-major call on columns [j0, j1) of C (B not transposed: its columns
    j0..j1 are contiguous at offset j0*ldb; transposed B: rows j0..j1 at offset j0)."""
    b_off = j0 * ldb if transb in "Nn" else j0
    return b_off, j0 * ldc, j1 - j0
