"""The window walk (frozen_prefix_chunk_gb300.walk.WindowWalk) vs the oracle.

Each chunk of a walked window must match the oracle run on that chunk with
the cache before it as the frozen prefix -- for a q8_0 cache, the oracle's
own encoding of the earlier chunks, dequantised.  With a bf16 cache the
forward and dQ of every chunk also equal one call over all chunks at once
(every chunk row sees the same keys either way); dK/dV do not, since the
walk stops gradients at the cache.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

HQ, HKV, D = 8, 2, 128
SCALE = 128 ** -0.5


def _window(lp0, chunks, seed):
    g = torch.Generator().manual_seed(seed)
    n = lp0 + sum(chunks)
    k = torch.randn(n, HKV, D, generator=g).to(torch.bfloat16)
    v = torch.randn(n, HKV, D, generator=g).to(torch.bfloat16)
    q = torch.randn(sum(chunks), HQ, D, generator=g).to(torch.bfloat16)
    do = torch.randn(sum(chunks), HQ, D, generator=g).to(torch.bfloat16)
    return k, v, q, do


def _oracle_chunk(kp, vp, q, k, v, do, prefix_dtype, horizon=0):
    w = synth.custom(hq=HQ, hkv=HKV, head_dim=D, lp=[kp.shape[0]], lc=[q.shape[0]],
                     prefix_dtype=prefix_dtype, softmax_scale=SCALE)
    inp = dict(q=q, k_prefix=kp, v_prefix=vp, k_chunk=k, v_chunk=v, dout=do,
               cu_seqlens_prefix=synth.cu_seqlens(w.lp), cu_seqlens_chunk=synth.cu_seqlens(w.lc),
               workload=w)
    return inp, oracle.run(inp, prefix_grad_rows=horizon > 0)


def _walk(cache_dtype, lp0, chunks, seed, horizon=0):
    from frozen_prefix_chunk_gb300 import PREFIX_Q8_0
    from frozen_prefix_chunk_gb300.walk import WindowWalk
    k, v, q, do = _window(lp0, chunks, seed)
    walk = WindowWalk(k[:lp0].cuda(), v[:lp0].cuda(), lp0 + sum(chunks), HQ, SCALE,
                      cache_dtype, horizon)
    outs = []
    c0 = 0
    for lc in chunks:
        r = lp0 + c0
        outs.append([t.cpu() for t in walk.step(q[c0:c0 + lc].cuda(), k[r:r + lc].cuda(),
                                                 v[r:r + lc].cuda(), do[c0:c0 + lc].cuda())])
        c0 += lc
    torch.cuda.synchronize()
    return (k, v, q, do), outs, walk


def _prefix_as_cached(k, n, cache_dtype):
    """The first n rows as the cache holds them (bf16, or q8_0 bytes)."""
    if cache_dtype == synth.PREFIX_Q8_0:
        bits = k[:n].contiguous().view(torch.int16).numpy().view(np.uint16)
        return torch.from_numpy(oracle.quantize_q8_0(bits))
    return k[:n]


@pytest.mark.parametrize("cache_dtype", [synth.PREFIX_BF16, synth.PREFIX_Q8_0])
def test_walk_chunks_match_the_oracle(cache_dtype):
    lp0, chunks = 700, [200, 256, 77, 128]
    (k, v, q, do), outs, walk = _walk(cache_dtype, lp0, chunks, seed=3)
    c0 = 0
    for i, lc in enumerate(chunks):
        n = lp0 + c0
        kp, vp = _prefix_as_cached(k, n, cache_dtype), _prefix_as_cached(v, n, cache_dtype)
        inp, ref = _oracle_chunk(kp, vp, q[c0:c0 + lc], k[n:n + lc], v[n:n + lc],
                                 do[c0:c0 + lc], cache_dtype)
        o, lse, dq, dk, dv = outs[i]
        err = gu.errors(dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv,
                             delta=torch.from_numpy(ref["delta"]).float()), ref, inp)
        print("chunk", i, err)
        gu.assert_within(err)
        c0 += lc
    # the cache holds the context and every chunk, in the cache's format
    total = lp0 + sum(chunks)
    assert walk.lp == total
    assert torch.equal(walk.k_cache.cpu(), _prefix_as_cached(k, total, cache_dtype))


def test_walk_forward_and_dq_equal_one_call_over_all_chunks():
    import frozen_prefix_chunk_gb300 as cfa
    lp0, chunks = 500, [128, 200, 96]
    (k, v, q, do), outs, _ = _walk(synth.PREFIX_BF16, lp0, chunks, seed=4)
    w = synth.custom(hq=HQ, hkv=HKV, head_dim=D, lp=[lp0], lc=[sum(chunks)], softmax_scale=SCALE)
    inp = dict(q=q, k_prefix=k[:lp0], v_prefix=v[:lp0], k_chunk=k[lp0:], v_chunk=v[lp0:], dout=do,
               cu_seqlens_prefix=synth.cu_seqlens(w.lp), cu_seqlens_chunk=synth.cu_seqlens(w.lc),
               workload=w)
    one = gu.run_cuda(inp)
    c0 = 0
    for i, lc in enumerate(chunks):
        o, lse, dq = outs[i][:3]
        ref_o = one["o"][c0:c0 + lc].double()
        assert (o.double() - ref_o).abs().max() / ref_o.abs().max() <= 1e-2
        assert (lse - one["lse"][:, c0:c0 + lc]).abs().max() <= 2e-2
        ref_dq = one["dq"][c0:c0 + lc].double()
        assert (dq.double() - ref_dq).norm() / ref_dq.norm() <= 2e-2
        c0 += lc


def test_walk_with_horizon_prefix_gradients():
    lp0, chunks, horizon = 600, [192, 100], 300
    (k, v, q, do), outs, _ = _walk(synth.PREFIX_BF16, lp0, chunks, seed=5, horizon=horizon)
    c0 = 0
    for i, lc in enumerate(chunks):
        n = lp0 + c0
        inp, ref = _oracle_chunk(k[:n], v[:n], q[c0:c0 + lc], k[n:n + lc], v[n:n + lc],
                                 do[c0:c0 + lc], synth.PREFIX_BF16, horizon)
        dkp, dvp = outs[i][5].double().numpy(), outs[i][6].double().numpy()
        rows = slice(n - min(horizon, n), n)
        for got, want in ((dkp, ref["dkp"]), (dvp, ref["dvp"])):
            g, r = got[rows], want[rows]
            assert np.linalg.norm(g - r) / np.linalg.norm(r) <= gu.TOL_GRAD
            assert np.all(got[:rows.start] == 0)       # outside the horizon: untouched zeros
        c0 += lc


def test_walk_q8_0_decoded_rows_equal_the_calls_own_decoding():
    # the walk's bf16 copy of a q8_0 cache gives bitwise the results of
    # passing the q8_0 cache to the calls, which decode it themselves
    import frozen_prefix_chunk_gb300 as cfa
    lp0, chunks = 300, [128, 70]
    (k, v, q, do), outs, walk = _walk(synth.PREFIX_Q8_0, lp0, chunks, seed=8)
    c0 = 0
    for i, lc in enumerate(chunks):
        n = lp0 + c0
        # the args hold raw pointers: every tensor they name stays referenced
        qq, dd = q[c0:c0 + lc].cuda(), do[c0:c0 + lc].cuda()
        kc, vc = k[n:n + lc].cuda(), v[n:n + lc].cuda()
        cu_p = torch.tensor([0, n], dtype=torch.int32, device="cuda")
        cu_c = torch.tensor([0, lc], dtype=torch.int32, device="cuda")
        a = cfa.make_args(qq, walk.k_cache[:n], walk.v_cache[:n], kc, vc, cu_p, cu_c, n, lc,
                          SCALE, cfa.PREFIX_Q8_0, hkv=HKV)
        o, lse, _ = cfa.forward(a, qq)
        delta = cfa.backward_preprocess(a, o, dd)
        dq, dk, dv, _ = cfa.backward(a, dd, lse, delta)
        for got, want in zip(outs[i], (o, lse, dq, dk, dv)):
            assert torch.equal(got, want.cpu())
        c0 += lc
