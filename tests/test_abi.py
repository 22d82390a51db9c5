"""The C-ABI library builds, loads and exports every symbol include/cfa.h
declares; host-side argument checks answer without a GPU."""
import ctypes
import math
import os
import re
import subprocess

import pytest

import frozen_prefix_chunk_gb300 as cfa
from frozen_prefix_chunk_gb300 import build as cfa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "cfa.h")


@pytest.fixture(scope="module")
def L():
    cfa_build.build()
    return cfa.lib()


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"\b(cfa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ("cfa_forward", "cfa_backward_preprocess", "cfa_backward", "cfa_workspace_size",
              "cfa_dequant_q8_0", "cfa_read_status", "cfa_status_string", "cfa_version"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    out = subprocess.run(["nm", "-D", "--defined-only", cfa_build.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (cfa_[a-z0-9_]+)", out))
    for n in _declared():
        assert n in exported, n
        assert hasattr(L, n)


def test_status_strings_and_version(L):
    assert cfa.status_string(0) == "ok"
    assert "timed out" in cfa.status_string(-5)
    assert L.cfa_version() >> 16 == 1


def _args(**kw):
    a = cfa.Args()
    a.q = a.k_chunk = a.v_chunk = a.k_prefix = a.v_prefix = 4096
    a.cu_seqlens_prefix = a.cu_seqlens_chunk = 8192
    a.batch, a.max_lp, a.max_lc, a.total_lp, a.total_lc = 1, 16, 8, 16, 8
    a.hq, a.hkv, a.head_dim, a.prefix_dtype, a.softmax_scale = 4, 2, 128, 0, 0.125
    for k, v in kw.items():
        setattr(a, k, v)
    return a


BAD = [
    (dict(hq=5, hkv=2), -1),            # hq % hkv
    (dict(hkv=0), -1),
    (dict(batch=0), -1),
    (dict(head_dim=96), -2),            # unsupported head_dim
    (dict(hq=256, hkv=1), -2),          # group wider than a tile
    (dict(hq=65536 * 2, hkv=2048), -2),  # more query heads than a grid dimension holds
    (dict(prefix_dtype=7), -1),
    (dict(softmax_scale=0.0), -1),
    (dict(softmax_scale=math.inf), -1),
    (dict(max_lc=9), -1),               # max beyond total
    (dict(q=4104), -1),                 # misaligned (8 B)
    (dict(k_prefix=None), -1),          # prefix rows without a pointer
    (dict(cu_seqlens_chunk=None), -1),
    (dict(total_lp=-1), -1),
]


@pytest.mark.parametrize("kw,status", BAD, ids=[str(i) for i in range(len(BAD))])
def test_forward_rejects_bad_arguments_on_the_host(L, kw, status):
    a = _args(**kw)
    assert L.cfa_forward(ctypes.byref(a), 4096, 4096, 4096, 1 << 20, None) == status
    assert L.cfa_backward(ctypes.byref(a), 4096, 4096, 4096, 4096, 4096, 4096, 4096, 1 << 20,
                          None) == status
    assert L.cfa_workspace_size(ctypes.byref(a), 0) == 0
    # the entry point without a workspace reports the same status, before it
    # looks up its fixed scratch (nothing touches the device)
    assert L.cfa_forward_noalloc(ctypes.byref(a), 4096, 4096, None) == status


def test_null_args_and_dequant_checks(L):
    assert L.cfa_forward(None, None, None, None, 0, None) == -1
    assert L.cfa_dequant_q8_0(None, 4, 4096, None, None) == -1
    assert L.cfa_dequant_q8_0(4096, -1, 4096, None, None) == -1
    assert L.cfa_dequant_q8_0(4097, 4, 4096, None, None) == -1    # odd block address
    assert L.cfa_dequant_q8_0(4096, 0, None, None, None) == 0      # nothing to do
    assert L.cfa_read_status(None, None) == -1


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(cfa_build, "LIB_PATH", str(tmp_path / "nope.so"))
    monkeypatch.setattr(cfa, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        cfa.lib()


def test_backward_horizon_rejects_bad_arguments_on_the_host(L):
    a = _args()
    f = L.cfa_backward_horizon
    # negative horizon
    assert f(ctypes.byref(a), -1, 4096, 4096, 4096, 4096, 4096, 4096, 4096, 4096, 4096,
             1 << 20, None) == -1
    # a horizon needs both prefix gradient buffers, 16-byte aligned
    assert f(ctypes.byref(a), 4, 4096, 4096, 4096, 4096, 4096, 4096, None, 4096, 4096,
             1 << 20, None) == -1
    assert f(ctypes.byref(a), 4, 4096, 4096, 4096, 4096, 4096, 4096, 4096, 4104, 4096,
             1 << 20, None) == -1


def _rs_args(**kw):
    from frozen_prefix_chunk_gb300.rowsparse import RowSparseArgs
    a = RowSparseArgs()
    a.dy, a.x, a.w, a.keep_idx = 4096, 8192, 12288, 16384
    a.n_keep, a.n_rows, a.in_features, a.out_features = 16, 64, 128, 256
    for k, v in kw.items():
        setattr(a, k, v)
    return a


RS_BAD = [
    dict(in_features=12),        # rows not a multiple of 16 bytes
    dict(out_features=100),
    dict(in_features=0),
    dict(n_keep=-1),
    dict(n_rows=-5),
    dict(dy=None),               # kept rows without a gradient
    dict(dy=4100),               # misaligned
    dict(keep_idx=None),
    dict(keep_idx=16386),        # int32 indices need 4-byte alignment
]


@pytest.mark.parametrize("kw", RS_BAD, ids=[str(i) for i in range(len(RS_BAD))])
def test_rowsparse_rejects_bad_arguments_on_the_host(L, kw):
    from frozen_prefix_chunk_gb300 import rowsparse as R
    R._L()
    a = _rs_args(**kw)
    assert L.cfa_rowsparse_dw(ctypes.byref(a), 4096, 0, 0, 4096, 1 << 20, None) == -1
    assert L.cfa_rowsparse_dx(ctypes.byref(a), 4096, 4096, 1 << 20, None) == -1
    assert L.cfa_rowsparse_workspace_size(ctypes.byref(a), 0) == 0


def test_rowsparse_output_checks_on_the_host(L):
    from frozen_prefix_chunk_gb300 import rowsparse as R
    R._L()
    a = _rs_args()
    f = L.cfa_rowsparse_dw
    assert f(ctypes.byref(a), 4096, 2, 0, 4096, 1 << 20, None) == -1     # unknown dW type
    assert f(ctypes.byref(a), None, 0, 0, 4096, 1 << 20, None) == -1     # no output
    assert f(ctypes.byref(a), 4104, 0, 0, 4096, 1 << 20, None) == -1     # misaligned output
    b = _rs_args(x=None)
    assert f(ctypes.byref(b), 4096, 0, 0, 4096, 1 << 20, None) == -1     # dW needs x
    c = _rs_args(w=None)
    assert L.cfa_rowsparse_dx(ctypes.byref(c), 4096, 4096, 1 << 20, None) == -1  # dX needs w
    assert L.cfa_rowsparse_workspace_size(ctypes.byref(a), 7) == 0       # unknown selector
    assert L.cfa_keep_index_chunks(4096, 4096, 0, 4, 4096, None) == -1   # no windows
    assert L.cfa_keep_index_chunks(None, 4096, 1, 4, 4096, None) == -1
    assert L.cfa_keep_index_chunks(4096, 4096, 1, 0, 4096, None) == 0    # nothing to do
