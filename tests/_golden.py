"""Reader for the hand-worked fixtures under tests/golden/ (no GEMM arithmetic)."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _matrix(text):
    rows = [r.split() for r in text.split(";")]
    return np.array([[float(x) for x in r] for r in rows], dtype=np.float64)


def load_worked(name="worked_2x3x2.txt"):
    fields, cases = {}, []
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val = [s.strip() for s in line.split("=", 1)]
            if key == "case":
                scal, exp = val.split("|")
                alpha, beta = [float(x) for x in scal.split()]
                cases.append((alpha, beta, _matrix(exp)))
            else:
                fields[key] = val
    return {
        "m": int(fields["m"]), "n": int(fields["n"]), "k": int(fields["k"]),
        "opA": _matrix(fields["opA"]), "opB": _matrix(fields["opB"]),
        "Cin": _matrix(fields["Cin"]), "cases": cases,
    }


def colmajor_storage(mat, ld, pad_value=np.nan):
    """Column-major storage (ld x cols) of a rows x cols matrix, padding = pad_value."""
    rows, cols = mat.shape
    buf = np.full((cols, ld), pad_value, dtype=np.float32)
    buf[:, :rows] = mat.T
    return buf.reshape(-1)
