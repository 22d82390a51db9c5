"""fp64 CPU oracle for the row-sparse projection backward.

TEST INFRASTRUCTURE ONLY: the tests and the benchmark's CPU-baseline leg use
it; the library never imports it, and this module never imports the library.

"POC: stop-gradient through context tokens" (prime-rl), section "Mechanism",
row_sparse_linear: a linear layer Y = X W^T keeps its full-row forward, and
its backward runs on the kept rows only, since the gradient reaching Y is
exactly zero on every other row.  With dY_keep holding the gradient of the
kept rows (row i belongs to row keep[i] of X and Y):

    dW          = dY_keep^T  X[keep]          ([out, in])
    dX[keep[i]] = dY_keep[i] W                 ([in] per kept row)
    dX[r]       = 0 for every row r not kept

Inputs are converted exactly (bf16 -> fp64); the products and sums are a
numpy matmul in fp64 (the library routine the definition names), with no
blocking or reordering of our own.  Pinned in tests/test_oracle_rowsparse.py
against torch fp64 autograd of the dense layer with the gradient masked to
the kept rows, brute-force loops on tiny inputs, and invariants (row order,
linearity in the kept set, all rows kept = the dense backward).  The tests
plant mistakes in edited copies of this file (tests/oracle_mutants.py).
"""
from __future__ import annotations

import numpy as np


def _f64(a) -> np.ndarray:
    if hasattr(a, "detach"):  # a torch tensor (bf16 converts exactly)
        return a.detach().double().cpu().numpy()
    return np.asarray(a, dtype=np.float64)


def rowsparse_dw(dy_keep, x, keep) -> np.ndarray:
    """dW = dY_keep^T X[keep] in fp64, shape [out, in]."""
    dy = _f64(dy_keep)
    xs = _f64(x)
    idx = np.asarray(keep, dtype=np.int64)
    rows = xs[idx]
    dw = dy.T @ rows
    return dw


def rowsparse_dx(dy_keep, w, keep, n_rows: int) -> np.ndarray:
    """dX in fp64, shape [n_rows, in]: row keep[i] = dY_keep[i] W, zero
    elsewhere."""
    dy = _f64(dy_keep)
    ws = _f64(w)
    idx = np.asarray(keep, dtype=np.int64)
    out = np.zeros((n_rows, ws.shape[1]), dtype=np.float64)
    vals = dy @ ws
    out[idx] = vals
    return out
