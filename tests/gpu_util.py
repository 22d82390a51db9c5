"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and
compare it with the fp64 oracle using the tolerances of the method:

* O: normwise-max relative error  max|O - O*| / max|O*|      <= 1e-2
* dQ, dK_chunk, dV_chunk: Frobenius relative error             <= 2e-2
* delta: normwise-max relative error  max|d - d*| / max|d*|    <= 1e-2
  (the GPU takes delta = dO . O from its stored bf16 O, the oracle from its
  fp64 O; the bf16 rounding of O, a relative 2^-9 per element, and the
  forward's own error, within the O tolerance, bound the difference)
* LSE: max absolute error (reported; checked loosely)
"""
import numpy as np
import torch

import frozen_prefix_chunk_gb300 as cfa

TOL_O = 1e-2
TOL_GRAD = 2e-2
TOL_LSE = 2e-2
TOL_DELTA = 1e-2


def to_device(inp, device="cuda"):
    out = dict(inp)
    for k in ("q", "k_prefix", "v_prefix", "k_chunk", "v_chunk", "dout",
              "cu_seqlens_prefix", "cu_seqlens_chunk"):
        out[k] = inp[k].to(device)
    return out


def make_args(dev_inp):
    w = dev_inp["workload"]
    return cfa.make_args(dev_inp["q"], dev_inp["k_prefix"] if sum(w.lp) else None,
                         dev_inp["v_prefix"] if sum(w.lp) else None, dev_inp["k_chunk"],
                         dev_inp["v_chunk"], dev_inp["cu_seqlens_prefix"],
                         dev_inp["cu_seqlens_chunk"], max(w.lp), max(w.lc), w.softmax_scale,
                         w.prefix_dtype, hkv=w.hkv, total_lp=sum(w.lp))


def run_cuda(inp, backward=True):
    """One fwd(+bwd) step on the GPU; returns CPU tensors."""
    d = to_device(inp)
    args = make_args(d)
    o, lse, ws_f = cfa.forward(args, d["q"])
    res = dict(o=o, lse=lse)
    if backward:
        delta = cfa.backward_preprocess(args, o, d["dout"])
        dq, dk, dv, ws_b = cfa.backward(args, d["dout"], lse, delta)
        res.update(delta=delta, dq=dq, dk=dk, dv=dv)
        assert cfa.read_status(ws_b) == 0
    assert cfa.read_status(ws_f) == 0
    torch.cuda.synchronize()
    return {k: v.cpu() for k, v in res.items()}


def _sel(a, rows):
    return a if rows is None else a[rows]


def errors(gpu, ref, inp, groups=None):
    """Errors of the CUDA outputs against the oracle over the rows the oracle
    computed (all rows, or those of the selected (window, kv head) groups)."""
    w = inp["workload"]
    g = w.hq // w.hkv
    cu_c = inp["cu_seqlens_chunk"].tolist()
    tc = cu_c[-1]
    mask_q = np.zeros((tc, w.hq), dtype=bool)
    mask_kv = np.zeros((tc, w.hkv), dtype=bool)
    if groups is None:
        groups = [(b, hk) for b in range(w.batch) for hk in range(w.hkv)]
    for b, hk in groups:
        mask_q[cu_c[b]:cu_c[b + 1], hk * g:(hk + 1) * g] = True
        mask_kv[cu_c[b]:cu_c[b + 1], hk] = True

    def rel_max(x, y, m):
        x, y = x[m], y[m]
        return float(np.abs(x - y).max() / max(np.abs(y).max(), 1e-30))

    def rel_fro(x, y, m):
        x, y = x[m], y[m]
        return float(np.linalg.norm(x - y) / max(np.linalg.norm(y), 1e-30))

    out = {}
    o = gpu["o"].double().numpy()
    out["o"] = rel_max(o, ref["o"], mask_q)
    lse = gpu["lse"].double().numpy().T      # [tc, hq]
    out["lse"] = float(np.abs(lse[mask_q] - ref["lse"].T[mask_q]).max())
    if "dq" in gpu:
        out["dq"] = rel_fro(gpu["dq"].double().numpy(), ref["dq"], mask_q)
        out["dk"] = rel_fro(gpu["dk"].double().numpy(), ref["dk"], mask_kv)
        out["dv"] = rel_fro(gpu["dv"].double().numpy(), ref["dv"], mask_kv)
    if "delta" in gpu:
        dl = gpu["delta"].double().numpy().T     # [tc, hq]
        rd = ref["delta"].T
        out["delta"] = float(np.abs(dl[mask_q] - rd[mask_q]).max() /
                             max(np.abs(rd[mask_q]).max(), 1e-30))
    return out


def assert_within(err):
    assert err["o"] <= TOL_O, err
    assert err["lse"] <= TOL_LSE, err
    for k in ("dq", "dk", "dv"):
        if k in err:
            assert err[k] <= TOL_GRAD, err
    if "delta" in err:
        assert err["delta"] <= TOL_DELTA, err
