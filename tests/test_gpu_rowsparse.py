"""Row-sparse projection backward (cfa_rowsparse_dw / _dx) vs the fp64 oracle.

Tolerances, from the arithmetic: the inputs are bf16, so every product is
exact in fp32 and the only error of an fp32 output is the fp32 accumulation
(typically ~sqrt(K) * 2^-24, far below 1e-5 for K <= 16k): fp32 outputs are
checked at Frobenius-relative 1e-5.  A bf16 output adds its own rounding (at
most 2^-9 relative per element): checked at Frobenius-relative 4e-3 and
normwise-max 8e-3.  Keep indices are integers: the rows written must be
exactly the kept ones.
"""
import os

import numpy as np
import pytest
import torch

from oracle import rowsparse as rs

pytestmark = pytest.mark.gpu

TOL_F32 = 1e-5
TOL_BF16 = 4e-3
TOL_BF16_MAX = 8e-3
SENTINEL = 7.0


def _rel(got, ref):
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


def _maxrel(got, ref):
    return float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-300))


def _inputs(n_rows, n_keep, d_in, d_out, seed, sort=True):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(n_rows, d_in, generator=g).to(torch.bfloat16)
    w = (torch.randn(d_out, d_in, generator=g) * d_in ** -0.5).to(torch.bfloat16)
    dy = torch.randn(n_keep, d_out, generator=g).to(torch.bfloat16)
    keep = torch.randperm(n_rows, generator=g)[:n_keep]
    if sort:
        keep = keep.sort().values
    return x, w, dy, keep.to(torch.int32)


SHAPES = [  # n_rows, n_keep, in, out
    (300, 64, 128, 128),        # one tile, one stage
    (1000, 200, 200, 136),      # ragged everywhere (tails of every dimension)
    (5000, 1, 256, 384),        # a single kept row
    (700, 700, 64, 8),          # every row kept; narrow out
    (8192, 4096, 128, 128),     # one output tile, long contraction: split K (dW)
    (4096, 256, 4096, 512),     # dX: few M tiles, long K: split K
    (2000, 513, 1024, 1024),    # many tiles, ragged K
]


def _ids(shapes):
    return ["x".join(map(str, s)) for s in shapes]


@pytest.mark.parametrize("shape", SHAPES, ids=_ids(SHAPES))
@pytest.mark.parametrize("sort", [True, False], ids=["sorted", "shuffled"])
def test_dw_f32(shape, sort):
    from frozen_prefix_chunk_gb300 import rowsparse as R
    import frozen_prefix_chunk_gb300 as cfa
    x, w, dy, keep = _inputs(*shape, seed=sum(shape), sort=sort)
    out, ws = R.dw(dy.cuda(), x.cuda(), keep.cuda())
    assert cfa.read_status(ws) == 0
    ref = rs.rowsparse_dw(dy, x, keep.numpy())
    e = _rel(out.double().cpu().numpy(), ref)
    print(shape, "dW f32", e)
    assert e <= TOL_F32


@pytest.mark.parametrize("shape", SHAPES, ids=_ids(SHAPES))
def test_dx(shape):
    from frozen_prefix_chunk_gb300 import rowsparse as R
    import frozen_prefix_chunk_gb300 as cfa
    x, w, dy, keep = _inputs(*shape, seed=sum(shape) + 1, sort=False)
    dx = torch.full((shape[0], shape[2]), SENTINEL, dtype=torch.bfloat16, device="cuda")
    dx, ws = R.dx(dy.cuda(), w.cuda(), keep.cuda(), dx)
    assert cfa.read_status(ws) == 0
    got = dx.double().cpu().numpy()
    kept = np.zeros(shape[0], dtype=bool)
    kept[keep.numpy()] = True
    assert np.all(got[~kept] == SENTINEL)          # rows not kept: untouched
    ref = rs.rowsparse_dx(dy, w, keep.numpy(), shape[0])
    e, m = _rel(got[kept], ref[kept]), _maxrel(got[kept], ref[kept])
    print(shape, "dX", e, m)
    assert e <= TOL_BF16 and m <= TOL_BF16_MAX


def test_dw_bf16_and_accumulate():
    from frozen_prefix_chunk_gb300 import rowsparse as R
    x, w, dy, keep = _inputs(3000, 300, 512, 256, seed=5)
    ref = rs.rowsparse_dw(dy, x, keep.numpy())
    g = torch.Generator().manual_seed(9)
    base32 = torch.randn(256, 512, generator=g)
    # fp32 accumulate: dW += dy^T x[keep]
    acc = base32.clone().cuda()
    R.dw(dy.cuda(), x.cuda(), keep.cuda(), out=acc, accumulate=True)
    assert _rel(acc.double().cpu().numpy(), base32.double().numpy() + ref) <= TOL_F32
    # bf16 output, overwrite and accumulate
    out, _ = R.dw(dy.cuda(), x.cuda(), keep.cuda(), dtype=torch.bfloat16)
    got = out.double().cpu().numpy()
    assert _rel(got, ref) <= TOL_BF16 and _maxrel(got, ref) <= TOL_BF16_MAX
    base16 = base32.to(torch.bfloat16)
    acc16 = base16.clone().cuda()
    R.dw(dy.cuda(), x.cuda(), keep.cuda(), out=acc16, accumulate=True)
    want = base16.double().numpy() + ref
    got = acc16.double().cpu().numpy()
    assert _rel(got, want) <= TOL_BF16 and _maxrel(got, want) <= TOL_BF16_MAX


def test_no_kept_rows():
    from frozen_prefix_chunk_gb300 import rowsparse as R
    x = torch.randn(100, 64).to(torch.bfloat16).cuda()
    w = torch.randn(32, 64).to(torch.bfloat16).cuda()
    dy = torch.zeros(0, 32, dtype=torch.bfloat16, device="cuda")
    keep = torch.zeros(0, dtype=torch.int32, device="cuda")
    out = torch.full((32, 64), 3.0, device="cuda")
    R.dw(dy, x, keep, out=out)
    assert torch.all(out == 0)
    out.fill_(3.0)
    R.dw(dy, x, keep, out=out, accumulate=True)
    assert torch.all(out == 3.0)
    dx = torch.full((100, 64), SENTINEL, dtype=torch.bfloat16, device="cuda")
    R.dx(dy, w, keep, dx)
    assert torch.all(dx == SENTINEL)


def test_split_k_is_deterministic():
    from frozen_prefix_chunk_gb300 import rowsparse as R
    x, w, dy, keep = _inputs(8192, 4096, 128, 128, seed=2)
    a, _ = R.dw(dy.cuda(), x.cuda(), keep.cuda())
    b, _ = R.dw(dy.cuda(), x.cuda(), keep.cuda())
    assert torch.equal(a, b)
    x, w, dy, keep = _inputs(4096, 256, 4096, 512, seed=3)
    d1 = torch.zeros(4096, 4096, dtype=torch.bfloat16, device="cuda")
    d2 = torch.zeros_like(d1)
    R.dx(dy.cuda(), w.cuda(), keep.cuda(), d1)
    R.dx(dy.cuda(), w.cuda(), keep.cuda(), d2)
    assert torch.equal(d1, d2)


def test_keep_index_outside_x_is_reported_and_skipped():
    from frozen_prefix_chunk_gb300 import rowsparse as R
    import frozen_prefix_chunk_gb300 as cfa
    x, w, dy, keep = _inputs(500, 40, 128, 64, seed=4)
    bad = keep.clone()
    bad[7] = 500          # one past the last row
    bad[20] = -3
    # dW: the bad rows read as zero rows of X
    out, ws = R.dw(dy.cuda(), x.cuda(), bad.cuda())
    assert cfa.read_status(ws) == -1
    ok = np.ones(40, dtype=bool)
    ok[[7, 20]] = False
    ref = rs.rowsparse_dw(dy[ok], x, keep.numpy()[ok])
    assert _rel(out.double().cpu().numpy(), ref) <= TOL_F32
    # dX: the bad rows are skipped, the others written
    dx = torch.full((500, 128), SENTINEL, dtype=torch.bfloat16, device="cuda")
    dx, ws = R.dx(dy.cuda(), w.cuda(), bad.cuda(), dx)
    assert cfa.read_status(ws) == -1
    got = dx.double().cpu().numpy()
    ref = rs.rowsparse_dx(dy[ok], w, keep.numpy()[ok], 500)
    good = keep.numpy()[ok]
    assert _rel(got[good], ref[good]) <= TOL_BF16
    rest = np.ones(500, dtype=bool)
    rest[good] = False
    assert np.all(got[rest] == SENTINEL)
    # the next call on the same workspace starts clean
    _, ws = R.dw(dy.cuda(), x.cuda(), keep.cuda(), ws=ws)
    assert cfa.read_status(ws) == 0


def test_keep_index_chunks_matches_the_packed_layout():
    from frozen_prefix_chunk_gb300 import rowsparse as R
    lp = [5, 0, 700, 128, 33]
    lc = [37, 100, 0, 256, 1]
    cu_p = np.concatenate([[0], np.cumsum(lp)]).astype(np.int32)
    cu_c = np.concatenate([[0], np.cumsum(lc)]).astype(np.int32)
    keep = R.keep_index_chunks(torch.from_numpy(cu_p).cuda(), torch.from_numpy(cu_c).cuda(),
                               int(cu_c[-1])).cpu().numpy()
    want, start = [], 0
    for p, c in zip(lp, lc):       # packed windows: Lp prefix rows, then Lc chunk rows
        want += list(range(start + p, start + p + c))
        start += p + c
    assert np.array_equal(keep, np.array(want, dtype=np.int32))


def test_q_projection_backward_from_the_attention_dq():
    # the attention backward's dQ [total_lc, hq, d] is the q projection's
    # dY_keep as it is; the kept rows come from cfa_keep_index_chunks
    import frozen_prefix_chunk_gb300 as cfa
    from frozen_prefix_chunk_gb300 import rowsparse as R
    import synth
    from tests import gpu_util as gu
    wl = synth.custom(hq=8, hkv=2, head_dim=128, lp=[300, 0, 129], lc=[77, 128, 200], seed=3)
    inp = synth.make_inputs(wl)
    d = gu.to_device(inp)
    args = gu.make_args(d)
    o, lse, _ = cfa.forward(args, d["q"])
    delta = cfa.backward_preprocess(args, o, d["dout"])
    dq, _, _, _ = cfa.backward(args, d["dout"], lse, delta)
    n_full = sum(wl.lp) + sum(wl.lc)
    hidden = 512
    g = torch.Generator().manual_seed(11)
    xh = torch.randn(n_full, hidden, generator=g).to(torch.bfloat16)     # layer input rows
    wq = (torch.randn(wl.hq * 128, hidden, generator=g) * hidden ** -0.5).to(torch.bfloat16)
    keep = R.keep_index_chunks(d["cu_seqlens_prefix"], d["cu_seqlens_chunk"], sum(wl.lc))
    dy = dq.view(sum(wl.lc), wl.hq * 128)
    dwq, _ = R.dw(dy, xh.cuda(), keep)
    dxh = torch.zeros(n_full, hidden, dtype=torch.bfloat16, device="cuda")
    R.dx(dy, wq.cuda(), keep, dxh)
    k = keep.cpu().numpy()
    dyc = dy.cpu()
    assert _rel(dwq.double().cpu().numpy(), rs.rowsparse_dw(dyc, xh, k)) <= TOL_F32
    ref = rs.rowsparse_dx(dyc, wq, k, n_full)
    got = dxh.double().cpu().numpy()
    assert _rel(got, ref) <= TOL_BF16
    ctx = np.ones(n_full, dtype=bool)
    ctx[k] = False
    assert np.all(got[ctx] == 0)   # context rows get no gradient


def test_qwen3_8b_projection_shapes_at_full_size():
    # the Qwen3-8B layer's q and down projections over the 16k window with its
    # 256 chunk rows kept, in the launch configuration the benchmark uses
    from frozen_prefix_chunk_gb300 import rowsparse as R
    n_rows, n_keep = 16384, 256
    g = torch.Generator().manual_seed(21)
    keep = (torch.arange(n_keep, dtype=torch.int32) + (n_rows - n_keep))
    for d_in, d_out in ((4096, 4096), (12288, 4096)):
        x = torch.randn(n_rows, d_in, generator=g).to(torch.bfloat16)
        w = (torch.randn(d_out, d_in, generator=g) * d_in ** -0.5).to(torch.bfloat16)
        dy = torch.randn(n_keep, d_out, generator=g).to(torch.bfloat16)
        out, _ = R.dw(dy.cuda(), x.cuda(), keep.cuda())
        ref = rs.rowsparse_dw(dy, x, keep.numpy())
        assert _rel(out.double().cpu().numpy(), ref) <= TOL_F32
        dx = torch.zeros(n_rows, d_in, dtype=torch.bfloat16, device="cuda")
        R.dx(dy.cuda(), w.cuda(), keep.cuda(), dx)
        got = dx[n_rows - n_keep:].double().cpu().numpy()
        ref = rs.rowsparse_dx(dy, w, keep.numpy(), n_rows)[n_rows - n_keep:]
        assert _rel(got, ref) <= TOL_BF16 and _maxrel(got, ref) <= TOL_BF16_MAX
        assert torch.count_nonzero(dx[: n_rows - n_keep]) == 0


def _dx_with(env_cluster, dy, w, keep, n_rows, d_in):
    from frozen_prefix_chunk_gb300 import rowsparse as R
    import frozen_prefix_chunk_gb300 as cfa
    old = os.environ.get("CFA_RS_CLUSTER")
    os.environ["CFA_RS_CLUSTER"] = env_cluster
    try:
        dx = torch.full((n_rows, d_in), SENTINEL, dtype=torch.bfloat16, device="cuda")
        dx, ws = R.dx(dy, w, keep, dx)
        torch.cuda.synchronize()
        return dx, cfa.read_status(ws), ws
    finally:
        if old is None:
            del os.environ["CFA_RS_CLUSTER"]
        else:
            os.environ["CFA_RS_CLUSTER"] = old


@pytest.mark.parametrize("shape", [(4096, 256, 4096, 512), (3000, 200, 8192, 1024)],
                         ids=["m256", "m200"])
def test_dx_split_k_cluster_path_equals_global_path(shape):
    """dX split K runs as one cluster per tile (the splits exchange their
    partials through L2 and each sums a share of the rows) where the splits
    fit; the sums are the same, in the same order, as the global-memory path's:
    bitwise equal outputs.  Four splits per tile (m256) and two (m200)."""
    x, w, dy, keep = _inputs(*shape, seed=sum(shape) + 7, sort=False)
    n_rows, n_keep, d_in, d_out = shape
    a, st_a, _ = _dx_with("1", dy.cuda(), w.cuda(), keep.cuda(), n_rows, d_in)
    b, st_b, _ = _dx_with("0", dy.cuda(), w.cuda(), keep.cuda(), n_rows, d_in)
    assert st_a == 0 and st_b == 0
    assert torch.equal(a, b)
    got = a.double().cpu().numpy()
    ref = rs.rowsparse_dx(dy, w, keep.numpy(), n_rows)
    kept = np.zeros(n_rows, dtype=bool)
    kept[keep.numpy()] = True
    assert np.all(got[~kept] == SENTINEL)
    assert _rel(got[kept], ref[kept]) <= TOL_BF16 and _maxrel(got[kept], ref[kept]) <= TOL_BF16_MAX


def test_dx_cluster_path_reports_a_bad_index_and_the_next_call_starts_clean():
    x, w, dy, keep = _inputs(500, 40, 8192, 512, seed=11)
    bad = keep.clone()
    bad[5] = 500
    bad[33] = -1
    dx, st, ws = _dx_with("1", dy.cuda(), w.cuda(), bad.cuda(), 500, 8192)
    assert st == -1
    ok = np.ones(40, dtype=bool)
    ok[[5, 33]] = False
    good = keep.numpy()[ok]
    got = dx.double().cpu().numpy()
    ref = rs.rowsparse_dx(dy[ok], w, good, 500)
    assert _rel(got[good], ref[good]) <= TOL_BF16
    rest = np.ones(500, dtype=bool)
    rest[good] = False
    assert np.all(got[rest] == SENTINEL)
    from frozen_prefix_chunk_gb300 import rowsparse as R
    import frozen_prefix_chunk_gb300 as cfa
    d2 = torch.zeros(500, 8192, dtype=torch.bfloat16, device="cuda")
    R.dx(dy.cuda(), w.cuda(), keep.cuda(), d2, ws=ws)
    assert cfa.read_status(ws) == 0
