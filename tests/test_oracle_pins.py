"""Pins for the fp64 oracle: checks against things other than itself.

* q8_0 dequant against hand-worked values (tests/golden/q8_0_dequant.txt).
* The hand-derived backward against central finite differences of the
  oracle's own forward.
* Forward and backward against full-window causal attention with the prefix
  detached, via torch fp64 autograd and scaled_dot_product_attention (the
  stop-gradient prefix of "Context-Frozen Training" / "train: walk the
  window" is exactly that).
* Lp = 0 against plain causal SDPA.
* Closed forms: Q = 0 gives uniform weights and LSE = ln(#visible keys);
  identical keys give dQ = 0; with Lp = 0 the chunk dV sums to the dO sum;
  identical heads in a group scale dK/dV by g.
* Prefix gradients for the horizon extension (the exact reverse pass):
  central finite differences wrt the prefix K/V, and full-window attention
  with the prefix NOT detached (torch fp64 autograd).
* Planted mistakes in the oracle (edited copies of its sources,
  tests/oracle_mutants.py) each fail at least one of the above.
"""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import synth
from tests import oracle_mutants as mutants

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "q8_0_dequant.txt")


# ---------------------------------------------------------------- helpers --

def _rand_group(lp, lc, g, d, seed, scale_q=1.0):
    rng = np.random.default_rng(seed)
    return dict(q=rng.standard_normal((lc, g, d)) * scale_q,
                kp=rng.standard_normal((lp, d)), vp=rng.standard_normal((lp, d)),
                kc=rng.standard_normal((lc, d)), vc=rng.standard_normal((lc, d)),
                dout=rng.standard_normal((lc, g, d)))


def _oracle(x, lp, lc, g, d, scale):
    return oracle.group(lp, lc, g, d, scale, x["q"], x["kp"], x["vp"], x["kc"], x["vc"],
                        x["dout"])


def _detached_reference(x, lp, lc, g, d, scale):
    """Full-window causal attention over Lp+Lc positions, prefix K/V detached;
    returns O, LSE and grads of <O_chunk, dO> wrt q, k_chunk, v_chunk."""
    q = torch.tensor(x["q"]).permute(1, 0, 2).contiguous().requires_grad_(True)  # [g, lc, d]
    kc = torch.tensor(x["kc"]).requires_grad_(True)
    vc = torch.tensor(x["vc"]).requires_grad_(True)
    kp = torch.tensor(x["kp"]).reshape(lp, d)
    vp = torch.tensor(x["vp"]).reshape(lp, d)
    k = torch.cat([kp.detach(), kc], 0)[None].expand(g, lp + lc, d)
    v = torch.cat([vp.detach(), vc], 0)[None].expand(g, lp + lc, d)
    qpos = torch.arange(lp, lp + lc)[:, None]
    kpos = torch.arange(lp + lc)[None, :]
    mask = kpos <= qpos                                   # causal over the full window
    o = F.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=scale)
    s = (q @ k.transpose(-1, -2)) * scale
    lse = torch.logsumexp(s.masked_fill(~mask, -math.inf), -1)          # [g, lc]
    dout = torch.tensor(x["dout"]).permute(1, 0, 2)
    (o * dout).sum().backward()
    return dict(o=o.detach().permute(1, 0, 2).numpy(), lse=lse.detach().numpy(),
                dq=q.grad.permute(1, 0, 2).numpy(), dk=kc.grad.numpy(), dv=vc.grad.numpy())


def _rel(a, b):
    a, b = np.asarray(a), np.asarray(b)
    den = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (den if den > 0 else 1.0)


# ------------------------------------------------------------ q8_0 golden --

def _golden_cases():
    cases = []
    for line in open(GOLDEN):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        sbits, code, f32bits, bfbits = line.split()
        cases.append((int(sbits, 16), int(code), int(f32bits, 16), int(bfbits, 16)))
    return cases


def test_golden_file_is_nonempty():
    assert len(_golden_cases()) >= 10


def test_dequant_q8_0_golden():
    assert _dequant_golden_ok()


def _dequant_golden_ok():
    cases = _golden_cases()
    blocks = np.zeros((len(cases), 34), dtype=np.uint8)
    for i, (sbits, code, _, _) in enumerate(cases):
        blocks[i, 0] = sbits & 0xFF
        blocks[i, 1] = sbits >> 8
        blocks[i, 2 + (i % 32)] = np.int8(code).view(np.uint8)   # vary the position
    f64, f32, bf = oracle.dequant_q8_0(blocks)
    ok = True
    for i, (sbits, code, f32bits, bfbits) in enumerate(cases):
        pos = i % 32
        got32 = int(np.float32(f32[i, pos]).view(np.uint32))
        ok &= got32 == f32bits
        ok &= int(bf[i, pos]) == bfbits
        ok &= float(np.float32(f64[i, pos])) == float(f32[i, pos])
        # every other code in the block is zero -> value is +-0
        others = np.delete(f32[i], pos)
        ok &= bool(np.all(others == 0))
    return bool(ok)


def test_dequant_matches_encoder_roundtrip_bound():
    # the encoder's codes times the fp16 scale land within half a step of x
    x = torch.randn(64, 128, generator=torch.Generator().manual_seed(3))
    b = synth.encode_q8_0(x)
    f64, _, _ = oracle.dequant_q8_0(b.numpy())
    amax = x.reshape(-1, 32).abs().max(1).values.numpy()
    err = np.abs(f64.reshape(-1, 32) - x.reshape(-1, 32).numpy().astype(np.float64))
    # half a quantisation step plus the fp16 rounding of the scale (<= 2^-11 rel)
    bound = amax / 127 * 0.5 + amax * 2.0 ** -11 + 1e-12
    assert np.all(err <= bound[:, None] * 1.0001)


# ------------------------------------------------------ finite differences --

def _loss(x, lp, lc, g, d, scale):
    r = oracle.group(lp, lc, g, d, scale, x["q"], x["kp"], x["vp"], x["kc"], x["vc"],
                     x["dout"], backward=False)
    return float(np.sum(r["o"] * x["dout"]))


def _fd_ok(lp, lc, g, d, seed, tol=1e-7):
    scale = 1.0 / math.sqrt(d)
    x = _rand_group(lp, lc, g, d, seed)
    r = _oracle(x, lp, lc, g, d, scale)
    h = 1e-6
    ok = True
    for name, grad in (("q", r["dq"]), ("kc", r["dk"]), ("vc", r["dv"])):
        fd = np.zeros_like(x[name])
        it = np.nditer(x[name], flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp = {k: v.copy() for k, v in x.items()}
            xm = {k: v.copy() for k, v in x.items()}
            xp[name][idx] += h
            xm[name][idx] -= h
            fd[idx] = (_loss(xp, lp, lc, g, d, scale) - _loss(xm, lp, lc, g, d, scale)) / (2 * h)
        ok &= _rel(grad, fd) <= tol
    return bool(ok)


@pytest.mark.parametrize("lp,lc,g,d", [(5, 4, 2, 8), (0, 4, 2, 8), (7, 3, 1, 4), (3, 1, 3, 8)])
def test_backward_matches_finite_differences(lp, lc, g, d):
    assert _fd_ok(lp, lc, g, d, seed=lp * 31 + lc)


def test_prefix_has_true_nonzero_gradient_that_is_truncated():
    # the stop-gradient is a truncation: the true derivative wrt the prefix is
    # not zero, and the oracle returns no prefix gradient at all
    lp, lc, g, d = 4, 3, 2, 8
    x = _rand_group(lp, lc, g, d, 11)
    scale = 1 / math.sqrt(d)
    h = 1e-6
    xp = {k: v.copy() for k, v in x.items()}
    xp["kp"][1, 2] += h
    xm = {k: v.copy() for k, v in x.items()}
    xm["kp"][1, 2] -= h
    fd = (_loss(xp, lp, lc, g, d, scale) - _loss(xm, lp, lc, g, d, scale)) / (2 * h)
    assert abs(fd) > 1e-6
    r = _oracle(x, lp, lc, g, d, scale)
    assert set(r) == {"o", "lse", "delta", "dq", "dk", "dv"}
    assert r["dk"].shape == (lc, d)          # chunk keys only


# ------------------------------------------- full window, prefix detached --

SHAPES_I3 = [(37, 19, 2, 16), (0, 9, 2, 8), (130, 5, 1, 32), (6, 17, 4, 8)]


def _detached_ok(lp, lc, g, d, seed, tol=1e-12):
    scale = 1.0 / math.sqrt(d) * 1.3
    x = _rand_group(lp, lc, g, d, seed)
    r = _oracle(x, lp, lc, g, d, scale)
    ref = _detached_reference(x, lp, lc, g, d, scale)
    errs = dict(o=_rel(r["o"], ref["o"]), lse=_rel(r["lse"], ref["lse"]),
                dq=_rel(r["dq"], ref["dq"]), dk=_rel(r["dk"], ref["dk"]),
                dv=_rel(r["dv"], ref["dv"]))
    return all(e <= tol for e in errs.values()), errs


@pytest.mark.parametrize("lp,lc,g,d", SHAPES_I3)
def test_matches_full_window_with_detached_prefix(lp, lc, g, d):
    ok, errs = _detached_ok(lp, lc, g, d, seed=lp + 7 * lc)
    assert ok, errs


def _packed_ok(orc=oracle):
    """Through the packed-batch glue (the oracle module `orc`): 2 windows,
    hkv=2, g=2, against the detached reference written with repeat_interleave
    for GQA."""
    w = synth.custom(hq=4, hkv=2, head_dim=16, lp=[11, 0], lc=[6, 5], dout_std=1.0, seed=5)
    inp = synth.make_inputs(w)
    r = orc.run(inp)
    g = w.hq // w.hkv
    ok = True
    cu_p = inp["cu_seqlens_prefix"].tolist()
    cu_c = inp["cu_seqlens_chunk"].tolist()
    for b in range(w.batch):
        lp, lc = w.lp[b], w.lc[b]
        q = inp["q"][cu_c[b]:cu_c[b + 1]].double().permute(1, 0, 2).contiguous().requires_grad_(True)
        kc = inp["k_chunk"][cu_c[b]:cu_c[b + 1]].double().permute(1, 0, 2).contiguous().requires_grad_(True)
        vc = inp["v_chunk"][cu_c[b]:cu_c[b + 1]].double().permute(1, 0, 2).contiguous().requires_grad_(True)
        kp = inp["k_prefix"][cu_p[b]:cu_p[b + 1]].double().permute(1, 0, 2)
        vp = inp["v_prefix"][cu_p[b]:cu_p[b + 1]].double().permute(1, 0, 2)
        k = torch.cat([kp, kc], 1).repeat_interleave(g, 0)
        v = torch.cat([vp, vc], 1).repeat_interleave(g, 0)
        mask = torch.arange(lp + lc)[None, :] <= torch.arange(lp, lp + lc)[:, None]
        o = F.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=w.softmax_scale)
        dout = inp["dout"][cu_c[b]:cu_c[b + 1]].double().permute(1, 0, 2)
        (o * dout).sum().backward()
        sl = slice(cu_c[b], cu_c[b + 1])
        ok &= _rel(r["o"][sl], o.detach().permute(1, 0, 2).numpy()) < 1e-12
        ok &= _rel(r["dq"][sl], q.grad.permute(1, 0, 2).numpy()) < 1e-12
        ok &= _rel(r["dk"][sl], kc.grad.permute(1, 0, 2).numpy()) < 1e-12
        ok &= _rel(r["dv"][sl], vc.grad.permute(1, 0, 2).numpy()) < 1e-12
    return bool(ok)


def test_packed_batch_gqa_matches_reference():
    assert _packed_ok()


# --------------------------------------------------------- Lp = 0, causal --

def test_no_prefix_is_plain_causal_attention():
    lc, g, d = 13, 2, 16
    x = _rand_group(0, lc, g, d, 2)
    scale = 0.25
    r = _oracle(x, 0, lc, g, d, scale)
    q = torch.tensor(x["q"]).permute(1, 0, 2)
    k = torch.tensor(x["kc"])[None].expand(g, lc, d)
    v = torch.tensor(x["vc"])[None].expand(g, lc, d)
    o = F.scaled_dot_product_attention(q, k, v, is_causal=True, scale=scale)
    assert _rel(r["o"], o.permute(1, 0, 2).numpy()) < 1e-12


# ------------------------------------------------------------ closed forms --

def _closed_forms_ok():
    ok = True
    lp, lc, g, d = 9, 6, 2, 8
    scale = 0.3
    # Q = 0: uniform weights over the visible keys
    x = _rand_group(lp, lc, g, d, 4)
    x["q"][:] = 0.0
    r = _oracle(x, lp, lc, g, d, scale)
    for t in range(lc):
        vis = np.concatenate([x["vp"], x["vc"][: t + 1]], 0)
        for h in range(g):
            ok &= np.allclose(r["o"][t, h], vis.mean(0), rtol=0, atol=1e-13)
            ok &= abs(r["lse"][h, t] - math.log(lp + t + 1)) < 1e-13
    # identical keys: softmax weights do not depend on q -> dQ = 0
    x = _rand_group(lp, lc, g, d, 5)
    x["kp"][:] = x["kc"][0]
    x["kc"][:] = x["kc"][0]
    r = _oracle(x, lp, lc, g, d, scale)
    ok &= np.abs(r["dq"]).max() < 1e-12
    # Lp = 0: column sums of P are the chunk dV; their total is sum of dO
    x = _rand_group(0, lc, g, d, 6)
    r = _oracle(x, 0, lc, g, d, scale)
    ok &= np.allclose(r["dv"].sum(0), x["dout"].sum((0, 1)), rtol=0, atol=1e-12)
    # identical query heads and dO within a group: dK, dV are g times one head's
    x = _rand_group(lp, lc, 1, d, 7)
    r1 = _oracle(x, lp, lc, 1, d, scale)
    x3 = dict(x)
    x3["q"] = np.repeat(x["q"], 3, axis=1)
    x3["dout"] = np.repeat(x["dout"], 3, axis=1)
    r3 = _oracle(x3, lp, lc, 3, d, scale)
    ok &= np.allclose(r3["dk"], 3 * r1["dk"], rtol=1e-12, atol=1e-13)
    ok &= np.allclose(r3["dv"], 3 * r1["dv"], rtol=1e-12, atol=1e-13)
    return bool(ok)


def test_closed_forms():
    assert _closed_forms_ok()


# ---------------------------------------------------------- planted mistakes --

ATTN_MUTANTS = list(range(1, 11))


def _all_attention_pins_pass():
    ok = _fd_ok(5, 4, 2, 8, seed=1)
    for lp, lc, g, d in SHAPES_I3[:2] + SHAPES_I3[3:]:
        ok &= _detached_ok(lp, lc, g, d, seed=3)[0]
    ok &= _closed_forms_ok()
    return bool(ok)


def test_pins_pass_on_the_oracle():
    assert _all_attention_pins_pass()


@pytest.mark.parametrize("n", ATTN_MUTANTS)
def test_pins_catch_planted_attention_mistake(n):
    with mutants.c_mutant(n):
        assert not _all_attention_pins_pass(), mutants.C_MUTANTS[n][0]


@pytest.mark.parametrize("n", [11, 12])
def test_pins_catch_planted_dequant_mistake(n):
    with mutants.c_mutant(n):
        assert not _dequant_golden_ok(), mutants.C_MUTANTS[n][0]


def test_pins_catch_transposed_head_map():
    assert not _packed_ok(mutants.py_mutant("head_map")), mutants.PY_MUTANTS["head_map"][0]


# ------------------------------------------- prefix gradients (horizon H) --

def _prefix_grad(x, lp, lc, g, d, scale):
    r = _oracle(x, lp, lc, g, d, scale)
    return oracle.prefix_grad(lp, lc, g, d, scale, x["q"], x["kp"], x["vp"], x["dout"],
                              r["lse"], r["delta"])


def _prefix_fd_ok(lp, lc, g, d, seed, tol=1e-7):
    scale = 1.0 / math.sqrt(d)
    x = _rand_group(lp, lc, g, d, seed)
    dkp, dvp = _prefix_grad(x, lp, lc, g, d, scale)
    h = 1e-6
    ok = True
    for name, grad in (("kp", dkp), ("vp", dvp)):
        fd = np.zeros_like(x[name])
        it = np.nditer(x[name], flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp = {k: v.copy() for k, v in x.items()}
            xm = {k: v.copy() for k, v in x.items()}
            xp[name][idx] += h
            xm[name][idx] -= h
            fd[idx] = (_loss(xp, lp, lc, g, d, scale) - _loss(xm, lp, lc, g, d, scale)) / (2 * h)
        ok &= _rel(grad, fd) <= tol
    return bool(ok)


@pytest.mark.parametrize("lp,lc,g,d", [(5, 4, 2, 8), (7, 3, 1, 4), (3, 1, 3, 8)])
def test_prefix_gradient_matches_finite_differences(lp, lc, g, d):
    assert _prefix_fd_ok(lp, lc, g, d, seed=lp * 17 + lc)


def _full_window_prefix_grads(x, lp, lc, g, d, scale):
    """Full-window causal attention with the prefix K/V trainable: grads of
    <O_chunk, dO> wrt the prefix keys and values."""
    q = torch.tensor(x["q"]).permute(1, 0, 2).contiguous()
    kp = torch.tensor(x["kp"]).requires_grad_(True)
    vp = torch.tensor(x["vp"]).requires_grad_(True)
    k = torch.cat([kp, torch.tensor(x["kc"])], 0)[None].expand(g, lp + lc, d)
    v = torch.cat([vp, torch.tensor(x["vc"])], 0)[None].expand(g, lp + lc, d)
    mask = torch.arange(lp + lc)[None, :] <= torch.arange(lp, lp + lc)[:, None]
    o = F.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=scale)
    (o * torch.tensor(x["dout"]).permute(1, 0, 2)).sum().backward()
    return kp.grad.numpy(), vp.grad.numpy()


def _prefix_full_window_ok(lp, lc, g, d, seed, tol=1e-12):
    scale = 1.0 / math.sqrt(d) * 1.3
    x = _rand_group(lp, lc, g, d, seed)
    dkp, dvp = _prefix_grad(x, lp, lc, g, d, scale)
    rk, rv = _full_window_prefix_grads(x, lp, lc, g, d, scale)
    return _rel(dkp, rk) <= tol and _rel(dvp, rv) <= tol


@pytest.mark.parametrize("lp,lc,g,d", [(37, 19, 2, 16), (130, 5, 1, 32), (6, 17, 4, 8)])
def test_prefix_gradient_matches_full_window_autograd(lp, lc, g, d):
    assert _prefix_full_window_ok(lp, lc, g, d, seed=lp + 3 * lc)


def test_truncated_prefix_derivative_is_the_horizon_gradient():
    # the derivative the stop-gradient drops is exactly what prefix_grad returns
    lp, lc, g, d = 4, 3, 2, 8
    x = _rand_group(lp, lc, g, d, 11)
    scale = 1 / math.sqrt(d)
    h = 1e-6
    xp = {k: v.copy() for k, v in x.items()}
    xp["kp"][1, 2] += h
    xm = {k: v.copy() for k, v in x.items()}
    xm["kp"][1, 2] -= h
    fd = (_loss(xp, lp, lc, g, d, scale) - _loss(xm, lp, lc, g, d, scale)) / (2 * h)
    dkp, _ = _prefix_grad(x, lp, lc, g, d, scale)
    assert abs(dkp[1, 2] - fd) <= 1e-7 * max(1.0, abs(fd))


@pytest.mark.parametrize("n", [13, 14])
def test_pins_catch_planted_prefix_gradient_mistake(n):
    with mutants.c_mutant(n):
        ok = _prefix_fd_ok(5, 4, 2, 8, seed=2)
        ok &= _prefix_full_window_ok(6, 17, 4, 8, seed=5)
    assert not ok, mutants.C_MUTANTS[n][0]


def test_every_planted_mistake_is_tested():
    # each mutant of the oracle's sources has a pin test above or in the
    # encoder / row-sparse pin files
    assert sorted(mutants.C_MUTANTS) == list(range(1, 17))
    assert set(mutants.PY_MUTANTS) == {"head_map", "dw_rows", "dw_transposed", "dx_rows",
                                       "dx_transposed"}
