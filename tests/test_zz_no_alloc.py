"""cfa_forward_noalloc, the forward for callers that cannot allocate.

Some callers have no way to allocate device memory -- a trainer running next
to an inference server that reserved the GPU's memory up front, or a C
program whose device memory comes only from someone else's pool -- so they
cannot provide cfa_forward's workspace.  cfa_forward_noalloc keeps the split
partials in a fixed scratch array inside the library instead.  These tests
call it through the C ABI and check, on two calls in a row with different
inputs (the shared scratch keeps the previous call's contents), that its
output is bitwise that of cfa_forward on the same inputs and matches the fp64
oracle within the forward's tolerance; that its device status word reads 0,
and reports a device-side wait that ran out; and that an oversized request is
refused.

The file is named so that pytest collects it last.
"""
import ctypes

import pytest
import torch

import oracle
import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _forward_both(seed):
    import frozen_prefix_chunk_gb300 as cfa

    # Lp=1536, Lc=512, Hq=16, Hkv=8: the forward is split along the keys, so
    # the scratch array really holds partials
    w = synth.workload("qwen3_1p7b", seed=seed)
    inp = synth.make_inputs(w)
    d = gu.to_device(inp)
    args = gu.make_args(d)
    need = cfa.workspace_size(args, cfa.WS_FORWARD)
    assert 256 < need <= cfa.lib().cfa_noalloc_scratch_bytes()
    o_ref, lse_ref, _ = cfa.forward(args, d["q"])
    o = torch.empty_like(o_ref)
    lse = torch.empty_like(lse_ref)
    cfa.forward_noalloc(args, o, lse)
    assert cfa.noalloc_read_status() == 0
    torch.cuda.synchronize()
    return inp, o_ref, lse_ref, o, lse


def _compare(inp, o_ref, lse_ref, o, lse):
    # the same kernels on the same inputs: the same bits as cfa_forward
    assert torch.equal(o, o_ref)
    assert torch.equal(lse, lse_ref)
    # and the oracle's values, element by element, within the tolerance
    ref = oracle.run(inp)
    err = gu.errors({"o": o.cpu(), "lse": lse.cpu()}, ref, inp)
    gu.assert_within(err)


def test_noalloc_forward_matches_forward_and_oracle_twice():
    import frozen_prefix_chunk_gb300 as cfa

    cfa.lib(build_if_missing=True)
    first = _forward_both(seed=0)
    _compare(*first)
    second = _forward_both(seed=1)
    _compare(*second)
    # the second call saw different inputs, so its output differs from the first
    assert not torch.equal(first[3], second[3])


def test_noalloc_forward_reports_a_device_timeout(monkeypatch):
    import frozen_prefix_chunk_gb300 as cfa

    cfa.lib(build_if_missing=True)
    inp = synth.make_inputs(synth.custom(hq=8, hkv=2, head_dim=128, lp=[2000], lc=[256], seed=2))
    d = gu.to_device(inp)
    args = gu.make_args(d)
    o = torch.empty_like(d["q"])
    lse = torch.empty(8, 256, dtype=torch.float32, device="cuda")
    # every forward kernel's MMA warp first waits on a barrier nothing
    # arrives on; the 2 ms bounded wait runs out and the kernel unwinds
    monkeypatch.setenv("CFA_WAIT_LIMIT_NS", "2000000")
    monkeypatch.setenv("CFA_DEBUG_WAIT_NEVER", "1")
    cfa.forward_noalloc(args, o, lse)
    assert cfa.noalloc_read_status() == -5
    monkeypatch.delenv("CFA_DEBUG_WAIT_NEVER")
    monkeypatch.delenv("CFA_WAIT_LIMIT_NS")
    # the next call clears the status word and computes the forward
    cfa.forward_noalloc(args, o, lse)
    assert cfa.noalloc_read_status() == 0
    o_ref, lse_ref, _ = cfa.forward(args, d["q"])
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)


def test_noalloc_forward_refuses_requests_beyond_its_scratch():
    import frozen_prefix_chunk_gb300 as cfa

    cfa.lib(build_if_missing=True)
    # a q8_0 prefix is expanded to bf16 in the workspace, so a long one needs
    # more than the fixed array; take the first shape that does on this GPU
    limit = cfa.lib().cfa_noalloc_scratch_bytes()
    for lp in (20000, 60000, 120000):
        w = synth.custom(hq=32, hkv=8, head_dim=128, lp=[lp], lc=[256],
                         prefix_dtype=synth.PREFIX_Q8_0, seed=0)
        d = gu.to_device(synth.make_inputs(w))
        args = gu.make_args(d)
        if cfa.workspace_size(args, cfa.WS_FORWARD) > limit:
            break
        del d
    else:
        pytest.fail("no test shape needs more than the fixed scratch")
    o = torch.empty_like(d["q"])
    lse = torch.empty(w.hq, sum(w.lc), dtype=torch.float32, device="cuda")
    st = cfa.lib().cfa_forward_noalloc(ctypes.byref(args), ctypes.c_void_p(o.data_ptr()),
                                       ctypes.c_void_p(lse.data_ptr()), None)
    assert st == -7, st
