"""Pins for the row-sparse projection backward oracle (oracle/rowsparse.py).

"POC: stop-gradient through context tokens", "Mechanism": the row-sparse
linear backward must equal the dense backward of Y = X W^T when the gradient
reaching Y is zero on every row that is not kept (the POC's own check is the
same comparison against a masked dense reference).  Pinned here by
  * torch fp64 autograd of the dense layer with the masked gradient,
  * brute-force loops on tiny inputs and one hand-worked case,
  * invariants: the order of the kept rows does not matter, the result is
    linear in the kept set, and keeping every row gives the dense backward,
and each planted mistake in the oracle (an edited copy of its source,
tests/oracle_mutants.py) fails at least one of them.
"""
import numpy as np
import pytest
import torch

from oracle import rowsparse as rs
from tests import oracle_mutants as mutants


def _case(n_rows, n_keep, d_in, d_out, seed, sort=True):
    g = np.random.default_rng(seed)
    x = g.standard_normal((n_rows, d_in))
    w = g.standard_normal((d_out, d_in))
    keep = g.choice(n_rows, size=n_keep, replace=False)
    if sort:
        keep = np.sort(keep)
    dy = g.standard_normal((n_keep, d_out))
    return x, w, keep, dy


def _dense_autograd(x, w, keep, dy):
    xt = torch.tensor(x, dtype=torch.float64, requires_grad=True)
    wt = torch.tensor(w, dtype=torch.float64, requires_grad=True)
    y = torch.nn.functional.linear(xt, wt)
    g = torch.zeros_like(y)
    g[torch.as_tensor(keep, dtype=torch.long)] = torch.tensor(dy, dtype=torch.float64)
    y.backward(g)
    return wt.grad.numpy(), xt.grad.numpy()


def _rel(a, b):
    if a.shape != b.shape:
        return np.inf
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


SHAPES = [  # n_rows, n_keep, in, out
    (40, 9, 16, 24),
    (33, 33, 8, 8),     # every row kept
    (50, 1, 12, 5),
    (64, 20, 32, 32),
]


def _pin_autograd(shape, seed, m=rs):
    x, w, keep, dy = _case(*shape, seed, sort=seed % 2 == 0)
    rw, rx = _dense_autograd(x, w, keep, dy)
    dw = m.rowsparse_dw(dy, x, keep)
    dx = m.rowsparse_dx(dy, w, keep, x.shape[0])
    return _rel(dw, rw) <= 1e-12 and _rel(dx, rx) <= 1e-12


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("seed", [0, 1])
def test_matches_dense_autograd_with_masked_gradient(shape, seed):
    assert _pin_autograd(shape, seed)


def test_no_kept_rows_gives_zero_gradients():
    x, w, _, _ = _case(10, 3, 4, 6, 0)
    keep = np.zeros(0, dtype=np.int64)
    dy = np.zeros((0, 6))
    assert np.all(rs.rowsparse_dw(dy, x, keep) == 0) and rs.rowsparse_dw(dy, x, keep).shape == (6, 4)
    assert np.all(rs.rowsparse_dx(dy, w, keep, 10) == 0)


def _brute(x, w, keep, dy):
    n_keep, d_out = dy.shape
    d_in = x.shape[1]
    dw = [[0.0] * d_in for _ in range(d_out)]
    dx = [[0.0] * d_in for _ in range(x.shape[0])]
    for i in range(n_keep):
        r = int(keep[i])
        for o in range(d_out):
            for c in range(d_in):
                dw[o][c] += dy[i][o] * x[r][c]
                dx[r][c] += dy[i][o] * w[o][c]
    return np.array(dw), np.array(dx)


def _pin_brute(seed, m=rs):
    x, w, keep, dy = _case(7, 3, 4, 4, seed, sort=False)
    bw, bx = _brute(x, w, keep, dy)
    dw = m.rowsparse_dw(dy, x, keep)
    dx = m.rowsparse_dx(dy, w, keep, 7)
    return _rel(dw, bw) <= 1e-13 and _rel(dx, bx) <= 1e-13


@pytest.mark.parametrize("seed", [3, 4, 5])
def test_matches_brute_force_loops(seed):
    assert _pin_brute(seed)


def test_hand_worked_case():
    # X rows 0..2 = (1,2), (3,4), (5,6); kept rows 2 then 0; out = 2.
    # dY_keep = [[1, 0], [2, 1]]: row 0 of dY_keep belongs to X row 2.
    # dW[o] = sum_i dY_keep[i, o] X[keep[i]]:
    #   dW[0] = 1*(5,6) + 2*(1,2) = (7, 10);  dW[1] = 0*(5,6) + 1*(1,2) = (1, 2)
    # W = [[1, 0], [1, 1]]: dX[2] = 1*(1,0) + 0*(1,1) = (1, 0),
    #   dX[0] = 2*(1,0) + 1*(1,1) = (3, 1), dX[1] = 0
    x = np.array([[1., 2.], [3., 4.], [5., 6.]])
    w = np.array([[1., 0.], [1., 1.]])
    keep = np.array([2, 0])
    dy = np.array([[1., 0.], [2., 1.]])
    assert np.array_equal(rs.rowsparse_dw(dy, x, keep), [[7., 10.], [1., 2.]])
    assert np.array_equal(rs.rowsparse_dx(dy, w, keep, 3), [[3., 1.], [0., 0.], [1., 0.]])


def _pin_invariants(seed, m=rs):
    x, w, keep, dy = _case(30, 12, 8, 8, seed)
    dw = m.rowsparse_dw(dy, x, keep)
    dx = m.rowsparse_dx(dy, w, keep, 30)
    ok = True
    # any order of the kept rows (dY rows moved with them)
    p = np.random.default_rng(seed + 100).permutation(len(keep))
    ok &= _rel(m.rowsparse_dw(dy[p], x, keep[p]), dw) <= 1e-13
    ok &= _rel(m.rowsparse_dx(dy[p], w, keep[p], 30), dx) <= 1e-13
    # linear in the kept set
    a, b = slice(0, 5), slice(5, None)
    ok &= _rel(m.rowsparse_dw(dy[a], x, keep[a]) + m.rowsparse_dw(dy[b], x, keep[b]), dw) <= 1e-13
    ok &= _rel(m.rowsparse_dx(dy[a], w, keep[a], 30) + m.rowsparse_dx(dy[b], w, keep[b], 30), dx) <= 1e-13
    # every row kept, in order: the dense backward of Y = X W^T
    full = np.arange(30)
    dyf = np.random.default_rng(seed + 7).standard_normal((30, 8))
    ok &= _rel(m.rowsparse_dw(dyf, x, full), np.einsum("ro,ri->oi", dyf, x)) <= 1e-13
    ok &= _rel(m.rowsparse_dx(dyf, w, full, 30), np.einsum("ro,oi->ri", dyf, w)) <= 1e-13
    return bool(ok)


@pytest.mark.parametrize("seed", [0, 1])
def test_invariants(seed):
    assert _pin_invariants(seed)


def test_input_dtypes_convert_exactly():
    # bf16 torch tensors enter the oracle exactly (no rounding on the way in)
    x = torch.randn(20, 16, generator=torch.Generator().manual_seed(0)).to(torch.bfloat16)
    dy = torch.randn(5, 8, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    keep = np.array([3, 17, 0, 9, 11])
    ref = dy.double().numpy().T @ x.double().numpy()[keep]
    assert np.array_equal(rs.rowsparse_dw(dy, x, keep), ref)


@pytest.mark.parametrize("name", ["dw_rows", "dw_transposed", "dx_rows", "dx_transposed"])
def test_pins_catch_planted_mistakes(name):
    m = mutants.py_mutant(name)
    # a transposed W only type-checks when W is square
    shapes = [s for s in SHAPES if s[2] == s[3] or name != "dx_transposed"]
    caught = (not all(_pin_autograd(s, 0, m) for s in shapes)
              or not _pin_brute(3, m) or not _pin_invariants(0, m))
    assert caught, mutants.PY_MUTANTS[name][0]
