"""Failure detection without faulting the GPU.

Every device-side wait in the kernels is bounded by wall time.  The test hook
CFA_DEBUG_WAIT_NEVER=1 makes each attention kernel's MMA thread wait on a
barrier that nothing arrives on; with a 2 ms limit that wait runs out, the
CTA records CFA_ERR_DEVICE_TIMEOUT in the workspace status word, every role
drains the copies and MMAs it issued, TMEM is freed and the kernel returns.
The host reads the status with cfa_read_status, and the context stays usable
for the next call.
"""
import os

import pytest
import torch

import oracle
import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _run(inp):
    import frozen_prefix_chunk_gb300 as cfa

    d = gu.to_device(inp)
    args = gu.make_args(d)
    o, lse, ws_f = cfa.forward(args, d["q"])
    st_f = cfa.read_status(ws_f)
    delta = cfa.backward_preprocess(args, o, d["dout"])
    dq, dk, dv, ws_b = cfa.backward(args, d["dout"], lse, delta)
    st_b = cfa.read_status(ws_b)
    torch.cuda.synchronize()
    return st_f, st_b


def test_wait_timeout_is_reported_and_context_survives(monkeypatch):
    inp = synth.make_inputs(synth.custom(hq=8, hkv=2, head_dim=128, lp=[2000], lc=[256], seed=2))
    monkeypatch.setenv("CFA_WAIT_LIMIT_NS", "2000000")
    monkeypatch.setenv("CFA_DEBUG_WAIT_NEVER", "1")
    st_f, st_b = _run(inp)
    assert st_f == -5 and st_b == -5, (st_f, st_b)
    monkeypatch.delenv("CFA_DEBUG_WAIT_NEVER")
    monkeypatch.delenv("CFA_WAIT_LIMIT_NS")
    # the next call clears the status word and computes correctly
    st_f, st_b = _run(inp)
    assert st_f == 0 and st_b == 0
    gpu = gu.run_cuda(inp)
    err = gu.errors(gpu, oracle.run(inp), inp)
    gu.assert_within(err)
