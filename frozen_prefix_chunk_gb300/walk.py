"""Walking one window chunk by chunk over a growing KV cache.

"train: walk the window" ("What it is") trains a long window in chunks: each
chunk's queries attend to the cached keys and values of everything before it
-- read as stop-gradient constants -- plus the chunk's own keys causally, and
after the chunk its keys and values are written to the cache (the fork keeps
the cache at F16 or q8_0) so that the next chunk sees them.  ``WindowWalk``
is that loop around the library's calls: per chunk one forward, backward
preprocess and backward with the cache as the frozen prefix, then the cache
write (a copy for a bf16 cache, ``cfa_quantize_q8_0`` for a q8_0 one).

A q8_0 cache also keeps its rows decoded to bf16 (``cfa_dequant_q8_0`` of
each appended chunk, once): every call of a chunk would otherwise decode the
whole cache into its workspace again, twice per chunk (forward and backward),
and those workspace rows take the same memory as the decoded copy.  The
decoding is the one the calls do themselves, so the results are bitwise the
same.

The chunk's Q/K/V and the incoming dO come from the model and its loss, so
they are the caller's inputs; the walk owns the cache and the workspaces
(grown to the largest chunk seen).  Everything runs asynchronously on the
current stream; nothing is read back to the host and nothing waits for it.
"""
from __future__ import annotations

import torch

from . import (PREFIX_BF16, PREFIX_Q8_0, backward, backward_horizon, backward_preprocess,
               dequant_q8_0, forward, make_args, quantize_q8_0, workspace_size, WS_BACKWARD,
               WS_FORWARD)


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
        # the bf16 rows the calls read: the cache itself, or its decoded copy
        self.k_rows = torch.zeros(capacity, hkv, d, dtype=torch.bfloat16, device=self.dev)
        self.v_rows = torch.zeros_like(self.k_rows)
        if cache_dtype == PREFIX_Q8_0:
            shape = (capacity, hkv, d // 32 * 34)
            self.k_cache = torch.zeros(shape, dtype=torch.uint8, device=self.dev)
            self.v_cache = torch.zeros(shape, dtype=torch.uint8, device=self.dev)
        else:
            self.k_cache, self.v_cache = self.k_rows, self.v_rows
        self.lp = 0
        self._append(context_k, context_v)
        self._ws = {}
        # cu_seqlens of the one window, rewritten on the device every step:
        # a host tensor copied over would block the host on the stream
        self._cu = torch.zeros(2, 2, dtype=torch.int32, device=self.dev)

    def rewind(self, rows: int):
        """Forget every cache row from ``rows`` on (e.g. to walk the window
        again from its context)."""
        assert 0 <= rows <= self.lp
        self.lp = rows

    def _append(self, k: torch.Tensor, v: torch.Tensor):
        """Cache write: rows [lp, lp + n) get the chunk's keys and values."""
        n = k.shape[0]
        assert self.lp + n <= self.capacity, "cache capacity exceeded"
        if self.cache_dtype == PREFIX_Q8_0:
            rows = slice(self.lp, self.lp + n)
            for x, blocks, dec in ((k, self.k_cache, self.k_rows), (v, self.v_cache, self.v_rows)):
                quantize_q8_0(x.contiguous(), out=blocks[rows])
                dequant_q8_0(blocks[rows], out_bf16=dec[rows], want_f32=False)
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
        cu_p, cu_c = self._cu[0], self._cu[1]
        cu_p[1].fill_(lp)
        cu_c[1].fill_(lc)
        kp = self.k_rows[:lp] if lp else None
        vp = self.v_rows[:lp] if lp else None
        a = make_args(q, kp, vp, k, v, cu_p, cu_c, lp, lc, self.scale, PREFIX_BF16,
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
