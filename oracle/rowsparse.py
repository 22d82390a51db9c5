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
linearity in the kept set, all rows kept = the dense backward).
"""
from __future__ import annotations

import numpy as np


def _f64(a) -> np.ndarray:
    if hasattr(a, "detach"):  # a torch tensor (bf16 converts exactly)
        return a.detach().double().cpu().numpy()
    return np.asarray(a, dtype=np.float64)


def rowsparse_dw(dy_keep, x, keep, mutation: int = 0) -> np.ndarray:
    """dW = dY_keep^T X[keep] in fp64, shape [out, in].

    ``mutation`` plants a mistake for the pin tests (0 = none): 1 reads the
    first n_keep rows of X instead of the kept ones, 2 returns the transpose
    of the gradient's transpose (X[keep]^T dY_keep)."""
    dy = _f64(dy_keep)
    xs = _f64(x)
    idx = np.asarray(keep, dtype=np.int64)
    rows = xs[: len(idx)] if mutation == 1 else xs[idx]
    dw = dy.T @ rows
    if mutation == 2:
        dw = rows.T @ dy
    return dw


def rowsparse_dx(dy_keep, w, keep, n_rows: int, mutation: int = 0) -> np.ndarray:
    """dX in fp64, shape [n_rows, in]: row keep[i] = dY_keep[i] W, zero
    elsewhere.

    ``mutation``: 1 writes row i instead of row keep[i], 2 multiplies by W^T's
    leading block instead of W (a transposed operand, square W only)."""
    dy = _f64(dy_keep)
    ws = _f64(w)
    idx = np.asarray(keep, dtype=np.int64)
    out = np.zeros((n_rows, ws.shape[1]), dtype=np.float64)
    vals = dy @ (ws.T if mutation == 2 else ws)
    if mutation == 1:
        out[: len(idx)] = vals
    else:
        out[idx] = vals
    return out
