"""frozen_prefix_chunk_gb300 -- Python binding of the cfa C-ABI library.

Frozen-prefix chunk attention for GB300 (sm_103a): a trainable chunk of Lc
query rows attends to a stop-gradient KV prefix of Lp cached rows plus its
own causal keys; the backward returns dQ and the chunk's dK/dV only (the
query-split backward).  See ``include/cfa.h`` for the contract.

This module only marshals arguments: it takes torch CUDA tensors (PyTorch is
used for device memory and streams), fills the ``cfa_args`` struct and calls
the library on the current CUDA stream.  Every step of the computation runs in
the library's own kernels; there is no fallback -- if ``libcfa.so`` is missing
the calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

__all__ = ["CfaError", "Args", "lib", "workspace_size", "forward", "backward_preprocess",
           "backward", "backward_dq", "backward_dkdv", "dequant_q8_0", "read_status", "PREFIX_BF16", "PREFIX_Q8_0",
           "PREFIX_F16", "backward_horizon", "quantize_q8_0"]

PREFIX_BF16 = 0
PREFIX_Q8_0 = 1
PREFIX_F16 = 2
WS_FORWARD = 0
WS_BACKWARD = 1

_lib = None
_lock = threading.Lock()


class CfaError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} ({status})")
        self.status = status


class Args(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k_prefix", ctypes.c_void_p),
                ("v_prefix", ctypes.c_void_p), ("k_chunk", ctypes.c_void_p),
                ("v_chunk", ctypes.c_void_p), ("cu_seqlens_prefix", ctypes.c_void_p),
                ("cu_seqlens_chunk", ctypes.c_void_p), ("batch", ctypes.c_int32),
                ("max_lp", ctypes.c_int32), ("max_lc", ctypes.c_int32),
                ("total_lp", ctypes.c_int32), ("total_lc", ctypes.c_int32),
                ("hq", ctypes.c_int32), ("hkv", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("prefix_dtype", ctypes.c_int32), ("softmax_scale", ctypes.c_float)]


def lib(build_if_missing: bool = False):
    """The loaded libcfa.so.  Raises when it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB_PATH
            if build_if_missing and _build.is_stale():
                _build.build()
            if not os.path.exists(path):
                raise RuntimeError(f"cfa CUDA library not built ({path}); run "
                                   "frozen_prefix_chunk_gb300.build.build()")
            L = ctypes.CDLL(path)
            vp, sz = ctypes.c_void_p, ctypes.c_size_t
            ap = ctypes.POINTER(Args)
            L.cfa_workspace_size.argtypes = [ap, ctypes.c_int]
            L.cfa_workspace_size.restype = sz
            L.cfa_forward.argtypes = [ap, vp, vp, vp, sz, vp]
            L.cfa_backward_preprocess.argtypes = [ap, vp, vp, vp, vp]
            L.cfa_backward.argtypes = [ap, vp, vp, vp, vp, vp, vp, vp, sz, vp]
            L.cfa_backward_horizon.argtypes = [ap, ctypes.c_int, vp, vp, vp, vp, vp, vp, vp, vp,
                                               vp, sz, vp]
            L.cfa_backward_dq.argtypes = [ap, vp, vp, vp, vp, vp, sz, vp]
            L.cfa_backward_dkdv.argtypes = [ap, vp, vp, vp, vp, vp, vp, sz, vp]
            L.cfa_dequant_q8_0.argtypes = [vp, ctypes.c_longlong, vp, vp, vp]
            L.cfa_quantize_q8_0.argtypes = [vp, ctypes.c_longlong, vp, vp]
            L.cfa_read_status.argtypes = [vp, vp]
            L.cfa_forward_noalloc.argtypes = [ap, vp, vp, vp]
            L.cfa_forward_noalloc.restype = ctypes.c_int
            L.cfa_noalloc_scratch_bytes.argtypes = []
            L.cfa_noalloc_scratch_bytes.restype = sz
            L.cfa_noalloc_read_status.argtypes = [vp]
            L.cfa_noalloc_read_status.restype = ctypes.c_int
            L.cfa_status_string.argtypes = [ctypes.c_int]
            L.cfa_status_string.restype = ctypes.c_char_p
            for f in ("cfa_forward", "cfa_backward_preprocess", "cfa_backward",
                      "cfa_backward_dq", "cfa_backward_dkdv",
                      "cfa_dequant_q8_0", "cfa_read_status", "cfa_version"):
                getattr(L, f).restype = ctypes.c_int
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().cfa_status_string(status).decode()


def _check(status: int, what: str):
    if status != 0:
        raise CfaError(status, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def make_args(q, k_prefix, v_prefix, k_chunk, v_chunk, cu_seqlens_prefix, cu_seqlens_chunk,
              max_lp, max_lc, softmax_scale, prefix_dtype=PREFIX_BF16, hkv=None,
              total_lp=None) -> Args:
    """Fill cfa_args from tensors.  ``max_lp``/``max_lc`` are host ints (no
    device read).  For a q8_0 prefix, k/v_prefix are uint8
    [total_lp, hkv, d/32*34]; for an fp16 prefix, float16 [total_lp, hkv, d].
    The result holds raw device pointers, not the tensors: keep every tensor
    passed here referenced for as long as calls made with it may run."""
    total_lc, hq, d = q.shape
    if hkv is None:
        hkv = k_chunk.shape[1]
    if total_lp is None:
        total_lp = k_prefix.shape[0] if k_prefix is not None else 0
    a = Args()
    a.q, a.k_prefix, a.v_prefix = _ptr(q), _ptr(k_prefix), _ptr(v_prefix)
    a.k_chunk, a.v_chunk = _ptr(k_chunk), _ptr(v_chunk)
    a.cu_seqlens_prefix, a.cu_seqlens_chunk = _ptr(cu_seqlens_prefix), _ptr(cu_seqlens_chunk)
    a.batch = cu_seqlens_chunk.numel() - 1
    a.max_lp, a.max_lc = int(max_lp), int(max_lc)
    a.total_lp, a.total_lc = int(total_lp), int(total_lc)
    a.hq, a.hkv, a.head_dim = int(hq), int(hkv), int(d)
    a.prefix_dtype = int(prefix_dtype)
    a.softmax_scale = float(softmax_scale)
    return a


def workspace_size(args: Args, which: int) -> int:
    return int(lib().cfa_workspace_size(ctypes.byref(args), which))


def _workspace(args: Args, which: int, device) -> torch.Tensor:
    n = workspace_size(args, which)
    if n == 0:
        raise CfaError(-1, "cfa_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device)


def forward(args: Args, q: torch.Tensor, o=None, lse=None, ws=None, stream=None):
    """cfa_forward.  Returns (O bf16 [total_lc, hq, d], LSE fp32 [hq, total_lc], ws)."""
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(args.hq, args.total_lc, dtype=torch.float32, device=q.device)
    if ws is None:
        ws = _workspace(args, WS_FORWARD, q.device)
    _check(lib().cfa_forward(ctypes.byref(args), _ptr(o), _ptr(lse), _ptr(ws), ws.numel(),
                             _stream(stream)), "cfa_forward")
    return o, lse, ws


def forward_noalloc(args: Args, o: torch.Tensor, lse: torch.Tensor, stream=None):
    """cfa_forward_noalloc: the forward for callers that cannot allocate; its
    split partials live in the library's fixed device scratch array instead
    of a caller workspace.  o and lse are caller-provided; nothing is
    allocated.  Calls overlapping on the GPU race on the shared scratch."""
    _check(lib().cfa_forward_noalloc(ctypes.byref(args), _ptr(o), _ptr(lse), _stream(stream)),
           "cfa_forward_noalloc")
    return o, lse


def noalloc_read_status(stream=None) -> int:
    """cfa_noalloc_read_status: synchronises the stream and returns the device
    status word of the last cfa_forward_noalloc call on this device."""
    return int(lib().cfa_noalloc_read_status(_stream(stream)))


def backward_preprocess(args: Args, o, dout, delta=None, stream=None):
    """cfa_backward_preprocess.  Returns delta fp32 [hq, total_lc]."""
    if delta is None:
        delta = torch.empty(args.hq, args.total_lc, dtype=torch.float32, device=o.device)
    _check(lib().cfa_backward_preprocess(ctypes.byref(args), _ptr(o), _ptr(dout), _ptr(delta),
                                         _stream(stream)), "cfa_backward_preprocess")
    return delta


def backward(args: Args, dout, lse, delta, dq=None, dk=None, dv=None, ws=None, stream=None):
    """cfa_backward.  Returns (dQ, dK_chunk, dV_chunk, ws), all bf16."""
    dev = dout.device
    if dq is None:
        dq = torch.empty_like(dout)
    shape_kv = (args.total_lc, args.hkv, args.head_dim)
    if dk is None:
        dk = torch.empty(shape_kv, dtype=torch.bfloat16, device=dev)
    if dv is None:
        dv = torch.empty(shape_kv, dtype=torch.bfloat16, device=dev)
    if ws is None:
        ws = _workspace(args, WS_BACKWARD, dev)
    _check(lib().cfa_backward(ctypes.byref(args), _ptr(dout), _ptr(lse), _ptr(delta), _ptr(dq),
                              _ptr(dk), _ptr(dv), _ptr(ws), ws.numel(), _stream(stream)),
           "cfa_backward")
    return dq, dk, dv, ws


def backward_horizon(args: Args, horizon: int, dout, lse, delta, dq=None, dk=None, dv=None,
                     dkp=None, dvp=None, ws=None, stream=None):
    """cfa_backward_horizon: cfa_backward plus dK/dV of the last ``horizon``
    prefix rows of every window.  Returns (dQ, dK_chunk, dV_chunk, dK_prefix,
    dV_prefix, ws); prefix rows outside the horizon are left as given (zeros
    when the buffers are allocated here)."""
    dev = dout.device
    if dq is None:
        dq = torch.empty_like(dout)
    shape_kv = (args.total_lc, args.hkv, args.head_dim)
    shape_p = (args.total_lp, args.hkv, args.head_dim)
    if dk is None:
        dk = torch.empty(shape_kv, dtype=torch.bfloat16, device=dev)
    if dv is None:
        dv = torch.empty(shape_kv, dtype=torch.bfloat16, device=dev)
    if dkp is None:
        dkp = torch.zeros(shape_p, dtype=torch.bfloat16, device=dev)
    if dvp is None:
        dvp = torch.zeros(shape_p, dtype=torch.bfloat16, device=dev)
    if ws is None:
        ws = _workspace(args, WS_BACKWARD, dev)
    _check(lib().cfa_backward_horizon(ctypes.byref(args), int(horizon), _ptr(dout), _ptr(lse),
                                      _ptr(delta), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dkp),
                                      _ptr(dvp), _ptr(ws), ws.numel(), _stream(stream)),
           "cfa_backward_horizon")
    return dq, dk, dv, dkp, dvp, ws


def backward_dq(args: Args, dout, lse, delta, dq, ws, stream=None):
    """cfa_backward_dq: the dQ half of the backward (dq preallocated)."""
    _check(lib().cfa_backward_dq(ctypes.byref(args), _ptr(dout), _ptr(lse), _ptr(delta),
                                 _ptr(dq), _ptr(ws), ws.numel(), _stream(stream)),
           "cfa_backward_dq")
    return dq


def backward_dkdv(args: Args, dout, lse, delta, dk, dv, ws, stream=None):
    """cfa_backward_dkdv: the chunk dK/dV half of the backward."""
    _check(lib().cfa_backward_dkdv(ctypes.byref(args), _ptr(dout), _ptr(lse), _ptr(delta),
                                   _ptr(dk), _ptr(dv), _ptr(ws), ws.numel(), _stream(stream)),
           "cfa_backward_dkdv")
    return dk, dv


def dequant_q8_0(blocks: torch.Tensor, stream=None, out_bf16=None, want_f32=True):
    """cfa_dequant_q8_0 on uint8 blocks (last dim a multiple of 34).
    Returns (fp32 values or None, bf16 values) with last dim = 32 per block;
    out_bf16 may be given (preallocated), and want_f32=False skips the fp32
    output."""
    assert blocks.dtype == torch.uint8 and blocks.shape[-1] % 34 == 0
    nb = blocks.numel() // 34
    shape = tuple(blocks.shape[:-1]) + (blocks.shape[-1] // 34 * 32,)
    f32 = torch.empty(shape, dtype=torch.float32, device=blocks.device) if want_f32 else None
    bf = out_bf16 if out_bf16 is not None else torch.empty(shape, dtype=torch.bfloat16,
                                                           device=blocks.device)
    assert bf.dtype == torch.bfloat16 and bf.numel() == nb * 32 and bf.is_contiguous()
    _check(lib().cfa_dequant_q8_0(_ptr(blocks), nb, _ptr(f32) if f32 is not None else None,
                                  _ptr(bf), _stream(stream)), "cfa_dequant_q8_0")
    return f32, bf


def quantize_q8_0(x: torch.Tensor, out=None, stream=None):
    """cfa_quantize_q8_0 on bf16 values (last dim a multiple of 32).  Returns
    uint8 blocks with the last dim replaced by 34 per block; ``out`` may be a
    preallocated uint8 tensor (or a view into a cache) of that many bytes."""
    assert x.dtype == torch.bfloat16 and x.shape[-1] % 32 == 0 and x.is_contiguous()
    nb = x.numel() // 32
    if out is None:
        out = torch.empty(tuple(x.shape[:-1]) + (x.shape[-1] // 32 * 34,), dtype=torch.uint8,
                          device=x.device)
    assert out.dtype == torch.uint8 and out.numel() == nb * 34
    _check(lib().cfa_quantize_q8_0(_ptr(x), nb, _ptr(out), _stream(stream)), "cfa_quantize_q8_0")
    return out


def read_status(ws: torch.Tensor, stream=None) -> int:
    """Synchronises the stream and returns the device status word (0 = ok)."""
    return int(lib().cfa_read_status(_ptr(ws), _stream(stream)))
