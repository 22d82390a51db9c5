"""Walking one window chunk by chunk over a growing KV cache.

"train: walk the window" ("What it is") trains a long window in chunks: each
chunk's queries attend to the cached keys and values of everything before it
-- read as stop-gradient constants -- plus the chunk's own keys causally, and
after the chunk its keys and values are written to the cache (the fork keeps
the cache at F16 or q8_0) so that the next chunk sees them.  ``WindowWalk``
is that loop around the library's calls: per chunk one forward, backward
preprocess and backward with the cache as the frozen prefix, then the cache
write (a copy for a bf16 cache, ``cfa_quantize_q8_0`` for a q8_0 one).

The chunk's Q/K/V and the incoming dO come from the model and its loss, so
they are the caller's inputs; the walk owns the cache and the workspaces
(allocated once, for the cache capacity).  Everything runs asynchronously on
the current stream; nothing is read back to the host.
"""
from __future__ import annotations

import torch

from . import (PREFIX_BF16, PREFIX_Q8_0, backward, backward_horizon, backward_preprocess,
               forward, make_args, quantize_q8_0, workspace_size, WS_BACKWARD, WS_FORWARD)


class WindowWalk:
    def __init__(self, context_k: torch.Tensor, context_v: torch.Tensor, capacity: int,
                 hq: int, softmax_scale: float, cache_dtype: int = PREFIX_BF16,
                 horizon: int = 0):
        """``context_k/v``: bf16 [Lp0, hkv, d] keys/values of the window's
        context; ``capacity``: cache rows (context plus every chunk to come);
        ``horizon``: prefix rows before each chunk that receive dK/dV (0 = the
        stop-gradient walk)."""
        assert context_k.dtype == torch.bfloat16 and context_k.shape == context_v.shape
        lp0, hkv, d = context_k.shape
        assert capacity >= lp0 and cache_dtype in (PREFIX_BF16, PREFIX_Q8_0)
        self.dev = context_k.device
        self.hq, self.hkv, self.d = hq, hkv, d
        self.scale = float(softmax_scale)
        self.cache_dtype = cache_dtype
        self.horizon = int(horizon)
        self.capacity = capacity
        if cache_dtype == PREFIX_Q8_0:
            shape = (capacity, hkv, d // 32 * 34)
            self.k_cache = torch.zeros(shape, dtype=torch.uint8, device=self.dev)
            self.v_cache = torch.zeros(shape, dtype=torch.uint8, device=self.dev)
        else:
            self.k_cache = torch.zeros(capacity, hkv, d, dtype=torch.bfloat16, device=self.dev)
            self.v_cache = torch.zeros_like(self.k_cache)
        self.lp = 0
        self._append(context_k, context_v)
        self._ws = {}

    def _append(self, k: torch.Tensor, v: torch.Tensor):
        """Cache write: rows [lp, lp + n) get the chunk's keys and values."""
        n = k.shape[0]
        assert self.lp + n <= self.capacity, "cache capacity exceeded"
        if self.cache_dtype == PREFIX_Q8_0:
            quantize_q8_0(k.contiguous(), out=self.k_cache[self.lp:self.lp + n])
            quantize_q8_0(v.contiguous(), out=self.v_cache[self.lp:self.lp + n])
        else:
            self.k_cache[self.lp:self.lp + n].copy_(k)
            self.v_cache[self.lp:self.lp + n].copy_(v)
        self.lp += n

    def _workspace(self, args, which):
        # sizes grow with the prefix: keep the largest seen
        need = workspace_size(args, which)
        ws = self._ws.get(which)
        if ws is None or ws.numel() < need:
            ws = torch.empty(need, dtype=torch.uint8, device=self.dev)
            self._ws[which] = ws
        return ws

    def step(self, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, dout: torch.Tensor):
        """One chunk: q, dout [Lc, hq, d], k, v [Lc, hkv, d] (bf16).  Returns
        (O, LSE, dQ, dK_chunk, dV_chunk[, dK_prefix, dV_prefix]) -- the
        prefix gradients (rows [lp - horizon, lp) of the cache before this
        chunk) only with a horizon -- then appends k, v to the cache."""
        lc = q.shape[0]
        lp = self.lp
        cu_p = torch.tensor([0, lp], dtype=torch.int32, device=self.dev)
        cu_c = torch.tensor([0, lc], dtype=torch.int32, device=self.dev)
        kp = self.k_cache[:lp] if lp else None
        vp = self.v_cache[:lp] if lp else None
        a = make_args(q, kp, vp, k, v, cu_p, cu_c, lp, lc, self.scale, self.cache_dtype,
                      hkv=self.hkv, total_lp=lp)
        o, lse, _ = forward(a, q, ws=self._workspace(a, WS_FORWARD))
        delta = backward_preprocess(a, o, dout)
        wsb = self._workspace(a, WS_BACKWARD)
        if self.horizon:
            dq, dk, dv, dkp, dvp, _ = backward_horizon(a, self.horizon, dout, lse, delta, ws=wsb)
            out = (o, lse, dq, dk, dv, dkp, dvp)
        else:
            dq, dk, dv, _ = backward(a, dout, lse, delta, ws=wsb)
            out = (o, lse, dq, dk, dv)
        self._append(k, v)
        return out
