"""Row-sparse projection backward: binding of the cfa_rowsparse_* calls.

"POC: stop-gradient through context tokens" (prime-rl), "Mechanism": for a
linear layer Y = X W^T whose incoming gradient is zero on every row but the
kept ones, the backward runs on the kept rows only:

    dW          = dY_keep^T X[keep]
    dX[keep[i]] = dY_keep[i] W        (other rows of dX: zero, untouched here)

``dY_keep`` is compact (row i belongs to row ``keep[i]``).  The frozen-prefix
attention backward hands the q projection exactly that: its dQ
[total_lc, hq, d] is dY_keep [total_lc, hq * d] as it is, and
``keep_index_chunks`` gives the rows of the packed full sequence that the
chunk rows occupy.  Argument marshalling only; the library's kernels do the
work, on the current CUDA stream.
"""
from __future__ import annotations

import ctypes

import torch

from . import CfaError, _check, _ptr, _stream, lib as _lib

__all__ = ["RowSparseArgs", "rowsparse_args", "workspace_size", "dw", "dx",
           "keep_index_chunks", "RS_DW", "RS_DX"]

RS_DW, RS_DX = 0, 1
_GRAD_F32, _GRAD_BF16 = 0, 1


class RowSparseArgs(ctypes.Structure):
    _fields_ = [("dy", ctypes.c_void_p), ("x", ctypes.c_void_p), ("w", ctypes.c_void_p),
                ("keep_idx", ctypes.c_void_p), ("n_keep", ctypes.c_int32),
                ("n_rows", ctypes.c_int32), ("in_features", ctypes.c_int32),
                ("out_features", ctypes.c_int32)]


_registered = False


def _L():
    global _registered
    L = _lib()
    if not _registered:
        vp, sz = ctypes.c_void_p, ctypes.c_size_t
        ap = ctypes.POINTER(RowSparseArgs)
        L.cfa_rowsparse_workspace_size.argtypes = [ap, ctypes.c_int]
        L.cfa_rowsparse_workspace_size.restype = sz
        L.cfa_rowsparse_dw.argtypes = [ap, vp, ctypes.c_int, ctypes.c_int, vp, sz, vp]
        L.cfa_rowsparse_dw.restype = ctypes.c_int
        L.cfa_rowsparse_dx.argtypes = [ap, vp, vp, sz, vp]
        L.cfa_rowsparse_dx.restype = ctypes.c_int
        L.cfa_keep_index_chunks.argtypes = [vp, vp, ctypes.c_int, ctypes.c_int, vp, vp]
        L.cfa_keep_index_chunks.restype = ctypes.c_int
        _registered = True
    return L


def rowsparse_args(dy: torch.Tensor, keep: torch.Tensor, x: torch.Tensor = None,
                   w: torch.Tensor = None, n_rows: int = None,
                   in_features: int = None) -> RowSparseArgs:
    """dy bf16 [n_keep, out]; keep int32 [n_keep]; x bf16 [n_rows, in] (for
    dW); w bf16 [out, in] (for dX).  The result holds raw device pointers:
    keep the tensors referenced while calls made with it may run."""
    a = RowSparseArgs()
    a.dy, a.x, a.w, a.keep_idx = _ptr(dy), _ptr(x), _ptr(w), _ptr(keep)
    a.n_keep = dy.shape[0]
    a.out_features = dy.shape[1]
    if in_features is None:
        in_features = x.shape[1] if x is not None else w.shape[1]
    a.in_features = int(in_features)
    if n_rows is None:
        n_rows = x.shape[0] if x is not None else 0
    a.n_rows = int(n_rows)
    return a


def workspace_size(args: RowSparseArgs, which: int) -> int:
    return int(_L().cfa_rowsparse_workspace_size(ctypes.byref(args), which))


def _ws(args, which, device, ws):
    need = workspace_size(args, which)
    if need == 0:
        raise CfaError(-1, "cfa_rowsparse_workspace_size")
    if ws is None or ws.numel() < need:
        ws = torch.empty(need, dtype=torch.uint8, device=device)
    return ws


def dw(dy: torch.Tensor, x: torch.Tensor, keep: torch.Tensor, out: torch.Tensor = None,
       dtype=torch.float32, accumulate: bool = False, ws=None, stream=None):
    """cfa_rowsparse_dw: dW [out, in] = (or +=) dy^T x[keep].  Returns (dW, ws)."""
    assert dy.dtype == torch.bfloat16 and x.dtype == torch.bfloat16 and keep.dtype == torch.int32
    assert dy.is_contiguous() and x.is_contiguous() and keep.is_contiguous()
    if out is None:
        out = torch.empty(dy.shape[1], x.shape[1], dtype=dtype, device=x.device)
    assert out.dtype in (torch.float32, torch.bfloat16) and out.is_contiguous()
    a = rowsparse_args(dy, keep, x=x)
    ws = _ws(a, RS_DW, x.device, ws)
    _check(_L().cfa_rowsparse_dw(ctypes.byref(a), _ptr(out),
                                 _GRAD_F32 if out.dtype == torch.float32 else _GRAD_BF16,
                                 1 if accumulate else 0, _ptr(ws), ws.numel(), _stream(stream)),
           "cfa_rowsparse_dw")
    return out, ws


def dx(dy: torch.Tensor, w: torch.Tensor, keep: torch.Tensor, out: torch.Tensor, ws=None,
       stream=None):
    """cfa_rowsparse_dx: rows keep[i] of ``out`` (bf16 [n_rows, in]) = dy[i] w.
    Rows that are not kept are left as they are.  Returns (out, ws)."""
    assert dy.dtype == torch.bfloat16 and w.dtype == torch.bfloat16 and keep.dtype == torch.int32
    assert out.dtype == torch.bfloat16 and out.is_contiguous() and w.is_contiguous()
    a = rowsparse_args(dy, keep, w=w, n_rows=out.shape[0])
    ws = _ws(a, RS_DX, w.device, ws)
    _check(_L().cfa_rowsparse_dx(ctypes.byref(a), _ptr(out), _ptr(ws), ws.numel(),
                                 _stream(stream)), "cfa_rowsparse_dx")
    return out, ws


def keep_index_chunks(cu_seqlens_prefix: torch.Tensor, cu_seqlens_chunk: torch.Tensor,
                      total_lc: int, out: torch.Tensor = None, stream=None) -> torch.Tensor:
    """Rows of the packed full sequence (windows of Lp_b + Lc_b rows) that the
    chunk rows occupy: int32 [total_lc]."""
    if out is None:
        out = torch.empty(total_lc, dtype=torch.int32, device=cu_seqlens_chunk.device)
    _check(_L().cfa_keep_index_chunks(_ptr(cu_seqlens_prefix), _ptr(cu_seqlens_chunk),
                                      cu_seqlens_chunk.numel() - 1, int(total_lc), _ptr(out),
                                      _stream(stream)), "cfa_keep_index_chunks")
    return out
