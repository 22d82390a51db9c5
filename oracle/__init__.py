"""fp64 CPU oracle for frozen-prefix chunk attention (ctypes glue).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg use it; the library under
``frozen_prefix_chunk_gb300`` never imports it, and this module never imports
that package.  The arithmetic lives in ``cfa_oracle.c`` (plain loops, fp64);
this file only builds it, slices the packed inputs per (window, KV head) and
converts bf16 to fp64 (exact).

Parity is pinned by the CPU tests in ``tests/test_oracle_pins.py``: central
finite differences, full-window attention with the prefix detached (torch
fp64 autograd), Lp = 0 against causal SDPA, closed forms, and hand-worked q8_0
dequant values in ``tests/golden``.  The sources hold the plain definition
only: the tests plant mistakes in edited copies of them
(``tests/oracle_mutants.py``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "cfa_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libcfa_oracle.so")
_lib = None
_lock = threading.Lock()

_dp = ctypes.POINTER(ctypes.c_double)


def compile_library(src: str, out: str) -> str:
    """Compile a C source of the oracle's form with gcc (-O3, OpenMP) into
    the shared library `out` (written atomically).  Returns `out`."""
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O3", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                           "-o", tmp, src, "-lm"])
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle.  Returns the .so path."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    return compile_library(_SRC, _LIB_PATH)


def load(path: str):
    """The oracle's entry points in the compiled library at `path`."""
    lb = ctypes.CDLL(path)
    lb.cfa_oracle_group.restype = ctypes.c_int
    lb.cfa_oracle_group.argtypes = [
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
        _dp, _dp, _dp, _dp, _dp, _dp,
        _dp, _dp, _dp, _dp, _dp, _dp]
    lb.cfa_oracle_dequant_q8_0.restype = None
    lb.cfa_oracle_dequant_q8_0.argtypes = [
        ctypes.c_void_p, ctypes.c_long, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    lb.cfa_oracle_threads.restype = ctypes.c_int
    lb.cfa_oracle_quantize_q8_0.restype = None
    lb.cfa_oracle_quantize_q8_0.argtypes = [ctypes.c_void_p, ctypes.c_long, ctypes.c_void_p]
    lb.cfa_oracle_group_prefix_grad.restype = None
    lb.cfa_oracle_group_prefix_grad.argtypes = [
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
        _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp]
    return lb


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load(build())
    return _lib


def threads() -> int:
    return lib().cfa_oracle_threads()


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_dp) if a is not None else None


def dequant_q8_0(blocks):
    """q8_0 bytes (any shape, last dim a multiple of 34) -> (f64, f32, bf16 bits).
    Each output has the shape of ``blocks`` with the last dim replaced by the
    number of values (32 per block)."""
    b = np.ascontiguousarray(np.asarray(blocks, dtype=np.uint8))
    assert b.shape[-1] % 34 == 0
    nb = b.size // 34
    shape = b.shape[:-1] + (b.shape[-1] // 34 * 32,)
    f64 = np.empty(shape, dtype=np.float64)
    f32 = np.empty(shape, dtype=np.float32)
    bf = np.empty(shape, dtype=np.uint16)
    lib().cfa_oracle_dequant_q8_0(b.ctypes.data, nb, f64.ctypes.data, f32.ctypes.data,
                                  bf.ctypes.data)
    return f64, f32, bf


def quantize_q8_0(x_bf16_bits) -> np.ndarray:
    """bf16 bit patterns (uint16, last dim a multiple of 32) -> q8_0 bytes with
    the last dim replaced by 34 per block."""
    x = np.ascontiguousarray(np.asarray(x_bf16_bits, dtype=np.uint16))
    assert x.shape[-1] % 32 == 0
    nb = x.size // 32
    out = np.empty(x.shape[:-1] + (x.shape[-1] // 32 * 34,), dtype=np.uint8)
    lib().cfa_oracle_quantize_q8_0(x.ctypes.data, nb, out.ctypes.data)
    return out


def _f64(x) -> np.ndarray:
    if isinstance(x, torch.Tensor):
        return np.ascontiguousarray(x.to(torch.float64).numpy())
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def group(lp, lc, g, d, scale, q, kp, vp, kc, vc, dout, backward=True):
    """Run the oracle on one (window, KV head) group given fp64 arrays:
    q, dout [lc, g, d]; kp, vp [lp, d]; kc, vc [lc, d].
    Returns dict o, lse [g, lc], delta [g, lc], dq, dk, dv."""
    q, kp, vp, kc, vc, dout = (_f64(a) for a in (q, kp, vp, kc, vc, dout))
    o = np.zeros((lc, g, d))
    lse = np.zeros((g, lc))
    delta = np.zeros((g, lc))
    dq = np.zeros((lc, g, d)) if backward else None
    dk = np.zeros((lc, d)) if backward else None
    dv = np.zeros((lc, d)) if backward else None
    # empty arrays still need a valid pointer
    kp = kp if kp.size else np.zeros(1)
    vp = vp if vp.size else np.zeros(1)
    rc = lib().cfa_oracle_group(lp, lc, g, d, float(scale), _ptr(q), _ptr(kp), _ptr(vp),
                                _ptr(kc), _ptr(vc), _ptr(dout), _ptr(o), _ptr(lse),
                                _ptr(delta), _ptr(dq), _ptr(dk), _ptr(dv))
    if rc != 0:
        raise MemoryError("oracle allocation failed")
    return dict(o=o, lse=lse, delta=delta, dq=dq, dk=dk, dv=dv)


def prefix_grad(lp, lc, g, d, scale, q, kp, vp, dout, lse, delta):
    """Exact dK, dV [lp, d] of the prefix rows of one (window, KV head) group,
    given fp64 arrays q, dout [lc, g, d]; kp, vp [lp, d]; lse, delta [g, lc]
    (from ``group``)."""
    q, kp, vp, dout, lse, delta = (_f64(a) for a in (q, kp, vp, dout, lse, delta))
    dkp = np.zeros((lp, d))
    dvp = np.zeros((lp, d))
    if lp == 0 or lc == 0:
        return dkp, dvp
    lib().cfa_oracle_group_prefix_grad(lp, lc, g, d, float(scale), _ptr(q), _ptr(kp), _ptr(vp),
                                       _ptr(dout), _ptr(lse), _ptr(delta), _ptr(dkp),
                                       _ptr(dvp))
    return dkp, dvp


def _prefix_rows(x: torch.Tensor, p0: int, p1: int, hk: int, d: int, q8: bool) -> np.ndarray:
    if q8:
        blocks = x[p0:p1, hk].numpy()                        # [lp, d/32*34]
        f64, _, _ = dequant_q8_0(blocks)
        return f64.reshape(p1 - p0, d)
    return _f64(x[p0:p1, hk])                                # bf16 or fp16: exact in fp64


def run(inputs: dict, groups=None, backward=True, prefix_grad_rows: bool = False) -> dict:
    """Oracle outputs for packed inputs from ``synth.make_inputs``.

    ``groups``: iterable of (window, kv_head) pairs to compute (default: all).
    Entries of the outputs outside those groups are NaN.  KV head hk serves
    the query heads h with h // g == hk.
    Returns O [tc, hq, d], LSE [hq, tc], delta [hq, tc], dQ [tc, hq, d],
    dK_c / dV_c [tc, hkv, d] (float64 numpy); with ``prefix_grad_rows`` also
    dK_p / dV_p [tp, hkv, d] (``dkp``, ``dvp``) for every prefix row.
    """
    w = inputs["workload"]
    hq, hkv, d = w.hq, w.hkv, w.head_dim
    g = hq // hkv
    cu_p = inputs["cu_seqlens_prefix"].tolist()
    cu_c = inputs["cu_seqlens_chunk"].tolist()
    tc = cu_c[-1]
    q8 = w.prefix_dtype == 1
    out = dict(o=np.full((tc, hq, d), np.nan), lse=np.full((hq, tc), np.nan),
               delta=np.full((hq, tc), np.nan), dq=np.full((tc, hq, d), np.nan),
               dk=np.full((tc, hkv, d), np.nan), dv=np.full((tc, hkv, d), np.nan))
    if prefix_grad_rows:
        tp = cu_p[-1]
        out["dkp"] = np.full((tp, hkv, d), np.nan)
        out["dvp"] = np.full((tp, hkv, d), np.nan)
    if groups is None:
        groups = [(b, hk) for b in range(w.batch) for hk in range(hkv)]
    for b, hk in groups:
        p0, p1, c0, c1 = cu_p[b], cu_p[b + 1], cu_c[b], cu_c[b + 1]
        lp, lc = p1 - p0, c1 - c0
        if lc == 0:
            if prefix_grad_rows:
                # no chunk row attends to this prefix: its gradient is the empty sum
                out["dkp"][p0:p1, hk] = 0.0
                out["dvp"][p0:p1, hk] = 0.0
            continue
        heads = list(range(hk * g, (hk + 1) * g))
        qg = inputs["q"][c0:c1, heads]
        dog = inputs["dout"][c0:c1, heads]
        kp = _prefix_rows(inputs["k_prefix"], p0, p1, hk, d, q8)
        vp = _prefix_rows(inputs["v_prefix"], p0, p1, hk, d, q8)
        r = group(lp, lc, g, d, w.softmax_scale, qg, kp, vp, inputs["k_chunk"][c0:c1, hk],
                  inputs["v_chunk"][c0:c1, hk], dog, backward=backward)
        out["o"][c0:c1, heads] = r["o"]
        out["lse"][heads, c0:c1] = r["lse"]
        out["delta"][heads, c0:c1] = r["delta"]
        if backward:
            out["dq"][c0:c1, heads] = r["dq"]
            out["dk"][c0:c1, hk] = r["dk"]
            out["dv"][c0:c1, hk] = r["dv"]
        if prefix_grad_rows:
            dkp, dvp = prefix_grad(lp, lc, g, d, w.softmax_scale, qg, kp, vp, dog, r["lse"],
                                   r["delta"])
            out["dkp"][p0:p1, hk] = dkp
            out["dvp"][p0:p1, hk] = dvp
    return out
