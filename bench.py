#!/usr/bin/env python
"""Benchmark: frozen-prefix chunk attention fwd+bwd on GB300.

One step = cfa_forward + cfa_backward_preprocess + cfa_backward (as its two
halves, cfa_backward_dq and cfa_backward_dkdv) over one batch of synthetic
input resident in HBM.  Prints ONE JSON line (rank 0).

Metric: useful TFLOP/s of fwd+bwd.  Useful FLOPs per query head, with
Np = sum Lc*Lp and Nc = sum Lc(Lc+1)/2 (masked halves and the prefix dK/dV
the method never computes are not counted):
    forward  4 d (Np + Nc)          backward  6 d Np + 10 d Nc
Roofline of the step: t_roof = max(F / bf16 peak, algorithmic bytes / HBM
bandwidth), fraction = t_roof / t_measured.

Timing: W warm-up steps, then K steps, each bracketed by CUDA events on the
launching stream; L2 is flushed before every timed step, outside the events:
a 256 MiB write, then a 256 MiB read that writes those dirty lines back, so
the step starts with none of its inputs in L2 and no write-back of the flush
buffer left to do (--flush write keeps only the write).  Under torchrun every rank runs its own replica of the
workload (weak scaling, no collective on the data path); value = all ranks'
FLOPs / max over ranks of the time.

--impl reference times the fp64 CPU oracle instead (the deliberately slow
baseline arm), on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import synth  # noqa: E402

METRIC = "frozen-prefix chunk attention fwd+bwd TFLOP/s and % of GB300 roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20


# ------------------------------------------------------------- accounting --

def useful_flops(w, horizon=0) -> dict:
    np_pairs = sum(c * p for c, p in zip(w.lc, w.lp))
    nc_pairs = sum(c * (c + 1) // 2 for c in w.lc)
    # pairs (chunk row, prefix key in the horizon): their dK and dV
    nh_pairs = sum(c * min(horizon, p) for c, p in zip(w.lc, w.lp))
    d, h = w.head_dim, w.hq
    fwd = 4 * d * (np_pairs + nc_pairs) * h
    bwd = (6 * d * np_pairs + 4 * d * nh_pairs + 10 * d * nc_pairs) * h
    # the dQ kernel's own contraction work: S, dP and dQ over every visible pair
    dq_kernel = 6 * d * (np_pairs + nc_pairs) * h
    return dict(fwd=fwd, bwd=bwd, total=fwd + bwd, dq_kernel=dq_kernel, dkdv_kernel=bwd - dq_kernel)


def algorithmic_bytes(w, horizon=0) -> dict:
    """Bytes each pass must move at least once (split partials excluded)."""
    d, tp, tc = w.head_dim, sum(w.lp), sum(w.lc)
    th = sum(min(horizon, p) for p in w.lp)          # prefix rows in the horizon
    pref = 34 / 32 if w.prefix_dtype == synth.PREFIX_Q8_0 else 2.0
    qb = tc * w.hq * d * 2
    kvp = 2 * tp * w.hkv * d * pref
    kvc = 2 * tc * w.hkv * d * 2
    lse = tc * w.hq * 4
    fwd = qb + kvp + kvc + qb + lse                  # read q, k, v; write O, LSE
    pre = 2 * qb + lse                                # read O, dO; write delta
    dq_kernel = 2 * qb + 2 * lse + kvp + kvc + qb     # read q, dO, lse, delta, k, v; write dQ
    bwd = dq_kernel + 2 * qb + 2 * lse + kvc + kvc    # + dK/dV half: q, dO, lse, delta, kc/vc, dK/dV
    bwd += 2 * th * w.hkv * d * 2                     # + dK/dV of the horizon's prefix rows
    return dict(fwd=fwd, pre=pre, bwd=bwd, dq_kernel=dq_kernel, total=fwd + pre + bwd)


def slowest_rank_ms(tot_ms: float, world: int, device) -> float:
    """The timed region's length on the slowest rank.  Every rank times its
    own replica between barriers; the job takes as long as the slowest one
    (a MAX all-reduce, the only collective, outside the data path)."""
    if world <= 1:
        return tot_ms
    import torch.distributed as dist
    t = torch.tensor([tot_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world: int, flops_per_rank: float, ms_per_step: float) -> float:
    """Whole-job useful TFLOP/s: every rank's FLOPs over the slowest rank's time."""
    return world * flops_per_rank / (ms_per_step * 1e-3) / 1e12


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# the sources the dQ kernel (the roofline object's kernel) is built from
DQ_KERNEL_SOURCES = ("cfa_bwd.cu", "cfa_kernels.cuh", "cfa_ptx.cuh", "cfa_sched.cuh")


def kernel_source_sha() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "frozen_prefix_chunk_gb300", "csrc")
    for f in DQ_KERNEL_SOURCES:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch of the dQ kernel from the committed ncu summary,
    or None when the kernels changed since that capture."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    rec = d.get(workload)
    if not rec or rec.get("csrc_sha") != kernel_source_sha():
        return None
    return rec.get("dram_bytes_per_launch")


# ----------------------------------------------------------------- clocks --

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(device_index), "-lms", "100"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.flush()
        self.f.seek(0)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.f.read().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.f.name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "power_w_max": max(power), "samples": len(sm), "reasons": sorted(reasons)}


# --------------------------------------------------------------- oracle arm --

def _group_inputs(inp, b, hk, lc_sub):
    """The first lc_sub chunk rows of window b, KV head hk, as a one-window
    one-head-group workload (rows before lc_sub see exactly the same keys)."""
    w = inp["workload"]
    g = w.hq // w.hkv
    cu_p = inp["cu_seqlens_prefix"].tolist()
    cu_c = inp["cu_seqlens_chunk"].tolist()
    c0, p0, p1 = cu_c[b], cu_p[b], cu_p[b + 1]
    sub = synth.custom(hq=g, hkv=1, head_dim=w.head_dim, lp=[p1 - p0], lc=[lc_sub],
                       prefix_dtype=w.prefix_dtype, softmax_scale=w.softmax_scale,
                       name=w.name)
    heads = slice(hk * g, (hk + 1) * g)
    rows = slice(c0, c0 + lc_sub)
    return dict(q=inp["q"][rows, heads].contiguous(),
                k_prefix=inp["k_prefix"][p0:p1, hk:hk + 1].contiguous(),
                v_prefix=inp["v_prefix"][p0:p1, hk:hk + 1].contiguous(),
                k_chunk=inp["k_chunk"][rows, hk:hk + 1].contiguous(),
                v_chunk=inp["v_chunk"][rows, hk:hk + 1].contiguous(),
                dout=inp["dout"][rows, heads].contiguous(),
                cu_seqlens_prefix=synth.cu_seqlens([p1 - p0]),
                cu_seqlens_chunk=synth.cu_seqlens([lc_sub]), workload=sub)


def oracle_sample(inp, budget_s, group=(0, 0)):
    """Time the oracle, as it stands, on a bounded sample: the first rows of
    one (window, KV head) group, as many as fit in about budget_s (calibrated
    on two rows).  Returns (seconds, useful FLOPs of the sample, text)."""
    import oracle

    oracle.build()
    w = inp["workload"]
    b, hk = group
    lc = w.lc[b]
    probe = _group_inputs(inp, b, hk, min(lc, 2))
    t0 = time.perf_counter()
    oracle.run(probe)
    per_row = (time.perf_counter() - t0) / min(lc, 2)
    lc_sub = max(1, min(lc, int(budget_s / max(per_row, 1e-9))))
    sub = _group_inputs(inp, b, hk, lc_sub)
    t0 = time.perf_counter()
    oracle.run(sub)
    dt = time.perf_counter() - t0
    f = useful_flops(sub["workload"])["total"]
    desc = (f"oracle fwd+bwd of chunk rows 0..{lc_sub - 1} of window {b}, kv head {hk} of "
            f"{w.name} ({w.hq // w.hkv} query heads, Lp={w.lp[b]}, Lc={lc_sub} of {lc})")
    return dt, f, desc


def run_reference(args, w, rank):
    if rank != 0:
        return
    import oracle

    inp = synth.make_inputs(w)
    oracle.build()
    budget = min(20.0, 150.0 / max(1, args.steps + args.warmup))
    times, f, desc = [], 0, ""
    for i in range(args.warmup + args.steps):
        dt, f, desc = oracle_sample(inp, budget, group=(i % w.batch, i % w.hkv))
        if i >= args.warmup:
            times.append((dt, f))
    sec = sum(t for t, _ in times)
    value = sum(x for _, x in times) / sec / 1e12
    ms = sec / len(times) * 1e3
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(w, "n/a (CPU)"),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.threads(),
                             "kind": "oracle", "sample": desc + " (one group per step)"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def config_of(w, l2, horizon=0):
    return {"workload": w.name, "batch": w.batch, "hq": w.hq, "hkv": w.hkv, "horizon": horizon,
            "head_dim": w.head_dim, "lp": w.lp, "lc": w.lc,
            "prefix": ("q8_0 (dequantised to bf16 once per step, read by both passes)"
                       if w.prefix_dtype == synth.PREFIX_Q8_0 else "bf16"),
            "softmax_scale": w.softmax_scale, "l2": l2, "parallelism": "replicas"}


# ---------------------------------------------------------------- GPU arm --

def run_walk(args, w):
    """--walk C: the workload's first window walked chunk by chunk (chunks of
    C rows over its Lc chunk rows, each attending to the context plus the
    chunks before it in a growing cache), against one call over all the chunk
    rows and, up to 32k rows, one full-window call (no frozen context)."""
    import frozen_prefix_chunk_gb300 as cfa
    from frozen_prefix_chunk_gb300.walk import WindowWalk
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    cfa.lib(build_if_missing=True)
    lp0, lcw, C = w.lp[0], w.lc[0], args.walk
    if not 0 < C <= lcw:
        raise SystemExit(f"--walk: chunk rows must be in [1, {lcw}] (the window's chunk rows)")
    n_chunks = lcw // C
    lcw = n_chunks * C
    g = torch.Generator().manual_seed(0)
    def rnd(*shape, std=1.0):
        return (torch.randn(*shape, generator=g) * std).to(torch.bfloat16).to(dev)
    k, v = rnd(lp0 + lcw, w.hkv, w.head_dim), rnd(lp0 + lcw, w.hkv, w.head_dim)
    q, do = rnd(lcw, w.hq, w.head_dim), rnd(lcw, w.hq, w.head_dim, std=w.dout_std)
    cache = cfa.PREFIX_Q8_0 if w.prefix_dtype == synth.PREFIX_Q8_0 else cfa.PREFIX_BF16
    walk = WindowWalk(k[:lp0], v[:lp0], lp0 + lcw, w.hq, w.softmax_scale, cache)
    flush = L2Flush(dev, args.flush)

    def walk_once():
        walk.rewind(lp0)
        for c in range(n_chunks):
            r, t = lp0 + c * C, c * C
            walk.step(q[t:t + C], k[r:r + C], v[r:r + C], do[t:t + C])

    def one_call(lp, kk, vv, qq, dd, pref, kpv=None):
        kp, vp = (kpv if kpv is not None else (kk[:lp], vv[:lp])) if lp else (None, None)
        cu_p = torch.tensor([0, lp], dtype=torch.int32, device=dev)
        cu_c = torch.tensor([0, qq.shape[0]], dtype=torch.int32, device=dev)
        a = cfa.make_args(qq, kp, vp, kk[lp:], vv[lp:], cu_p, cu_c, lp, qq.shape[0],
                          w.softmax_scale, pref, hkv=w.hkv, total_lp=lp)
        o, lse, wsf = cfa.forward(a, qq)
        delta = cfa.backward_preprocess(a, o, dd)
        dq, dk, dv, wsb = cfa.backward(a, dd, lse, delta)
        # `a` holds raw pointers: every tensor it points to must stay alive
        # (cu_p / cu_c freed here would be reused by the next small allocation)
        keep = (cu_p, cu_c, kp, vp, kk, vv, qq, dd)
        def run():
            assert keep
            cfa.forward(a, qq, o, lse, wsf)
            cfa.backward_preprocess(a, o, dd, delta)
            cfa.backward(a, dd, lse, delta, dq, dk, dv, wsb)
        return run

    def timed(fn, steps):
        for _ in range(args.warmup):
            flush()
            fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(steps):
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            ts.append((e0, e1))
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in ts)

    steps = max(3, min(args.steps, 200))
    sampler = ClockSampler(0)
    walk_ms = timed(walk_once, steps)
    # the same walk replayed from a CUDA graph: no host work between chunks
    walk_once()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        walk_once()
    graph_ms = timed(graph.replay, steps)
    # one call over all chunk rows, the context frozen (in the cache's format)
    kpv = None
    if cache == cfa.PREFIX_Q8_0:
        kpv = (walk.k_rows[:lp0], walk.v_rows[:lp0])
    single_ms = timed(one_call(lp0, k, v, q, do, cfa.PREFIX_BF16, kpv), steps)
    full_ms = None
    if lp0 + lcw <= 32768:
        qf = torch.cat([rnd(lp0, w.hq, w.head_dim), q])
        dof = torch.cat([rnd(lp0, w.hq, w.head_dim, std=w.dout_std), do])
        full_ms = timed(one_call(0, k, v, qf, dof, cfa.PREFIX_BF16), max(3, steps // 4))
    clocks = sampler.stop()
    d, h = w.head_dim, w.hq
    fl = 0
    for c in range(n_chunks):
        lp_c = lp0 + c * C
        np_, nc_ = C * lp_c, C * (C + 1) // 2
        fl += (4 * d * (np_ + nc_) + 6 * d * np_ + 10 * d * nc_) * h
    line = {"metric": "window walk: fwd+bwd of every chunk over a growing KV cache, useful TFLOP/s",
            "value": fl / (walk_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "n_gpus": 1,
            "value_graph": fl / (graph_ms * 1e-3) / 1e12,
            "steps": steps, "warmup": args.warmup, "ms_per_step": walk_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) q/k/v)",
            "config": {"workload": w.name, "context": lp0, "chunk": C, "n_chunks": n_chunks,
                       "cache": "q8_0" if cache == cfa.PREFIX_Q8_0 else "bf16",
                       "l2": flush.describe()},
            "walk_ms": walk_ms, "walk_graph_ms": graph_ms, "single_call_ms": single_ms,
            "full_window_ms": full_ms, "full_window_rows": lp0 + lcw,
            "gpu_launches": None, "clocks": clocks}
    print(json.dumps(line), flush=True)


class L2Flush:
    """Evicts L2 before a timed step.  "write": a 256 MiB write (the lines it
    leaves are dirty, and their write-back to HBM then runs during the timed
    step); "write+read": the same write followed by a 256 MiB read of another
    buffer, which forces that write-back before the step and leaves only clean
    lines behind."""

    def __init__(self, dev, mode="write+read"):
        self.mode = mode
        self.buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.rbuf = (torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
                     if mode == "write+read" else None)
        self.out = torch.zeros((), dtype=torch.int64, device=dev)

    def __call__(self):
        self.buf.zero_()
        if self.rbuf is not None:
            # read every line; the result goes to a kept buffer, so a flush
            # allocates nothing
            torch.sum(self.rbuf, dim=0, dtype=torch.int64, out=self.out)

    def describe(self):
        return {"write": "flushed before every timed step (256 MiB write)",
                "write+read": "flushed before every timed step (256 MiB write, then a 256 MiB "
                              "read that writes the dirty lines back before the step)"}[self.mode]


# MLP width of the Qwen3 layer each workload stands in for (hidden = hq * d)
INTERMEDIATE = {"tiny": 512, "qwen3_1p7b": 6144}
DEFAULT_INTERMEDIATE = 12288   # Qwen3-8B


def rowsparse_gemms(w):
    """The row-sparse projections of the layer ("POC: stop-gradient through
    context tokens", "Mechanism": q/o and the dense MLP): (name, in, out)."""
    hidden = w.hq * w.head_dim
    inter = INTERMEDIATE.get(w.name, DEFAULT_INTERMEDIATE)
    return [("q", hidden, hidden), ("o", hidden, hidden), ("gate", hidden, inter),
            ("up", hidden, inter), ("down", inter, hidden)]


def run_rowsparse(args, w):
    """--rowsparse: the layer's row-sparse projection backward over the
    workload's kept rows (its chunk rows; the context rows get no gradient):
    per projection dW = dY_keep^T X[keep] (fp32) and dX[keep] = dY_keep W
    (bf16).  One step = the ten GEMMs on one stream."""
    import frozen_prefix_chunk_gb300 as cfa
    from frozen_prefix_chunk_gb300 import rowsparse as R
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    cfa.lib(build_if_missing=True)
    n_rows = sum(w.lp) + sum(w.lc)
    n_keep = sum(w.lc)
    cu_p = synth.cu_seqlens(w.lp).to(dev)
    cu_c = synth.cu_seqlens(w.lc).to(dev)
    keep = R.keep_index_chunks(cu_p, cu_c, n_keep)
    g = torch.Generator(device=dev).manual_seed(0)
    gemms = []
    xs = {}
    for name, d_in, d_out in rowsparse_gemms(w):
        # q/gate/up read the normed hidden states, o the attention output,
        # down the MLP activation: one [n_rows, in] input per distinct source
        src = {"q": "attn_in", "o": "attn_out", "gate": "mlp_in", "up": "mlp_in",
               "down": "mlp_act"}[name]
        if src not in xs:
            xs[src] = torch.randn(n_rows, d_in, device=dev, generator=g).to(torch.bfloat16)
        wt = (torch.randn(d_out, d_in, device=dev, generator=g) * d_in ** -0.5).to(torch.bfloat16)
        dy = torch.randn(n_keep, d_out, device=dev, generator=g).to(torch.bfloat16)
        dw = torch.empty(d_out, d_in, dtype=torch.float32, device=dev)
        dx = torch.zeros(n_rows, d_in, dtype=torch.bfloat16, device=dev)
        gemms.append(dict(name=name, d_in=d_in, d_out=d_out, x=xs[src], w=wt, dy=dy, dw=dw,
                          dx=dx, ws_w=None, ws_x=None))
    for G in gemms:
        _, G["ws_w"] = R.dw(G["dy"], G["x"], keep, out=G["dw"])
        _, G["ws_x"] = R.dx(G["dy"], G["w"], keep, G["dx"])
    for G in gemms:
        assert cfa.read_status(G["ws_w"]) == 0 and cfa.read_status(G["ws_x"]) == 0

    def step():
        for G in gemms:
            R.dw(G["dy"], G["x"], keep, out=G["dw"], ws=G["ws_w"])
            R.dx(G["dy"], G["w"], keep, G["dx"], ws=G["ws_x"])

    flush = L2Flush(dev, args.flush)
    peaks, peak_src = load_peaks()
    pk_t, pk_b = peaks["bf16_tflops"], peaks["hbm_gbs"]

    def timed(fn, steps):
        for _ in range(max(3, args.warmup)):
            flush()
            fn()
        torch.cuda.synchronize()
        ev = []
        for _ in range(steps):
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            ev.append((e0, e1))
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in ev)

    steps = max(3, min(args.steps, 300))
    sampler = ClockSampler(0)
    ms = timed(step, steps)
    per = []
    t_roof = 0.0
    fl_total = 0
    for G in gemms:
        for kind in ("dW", "dX"):
            fl = 2 * n_keep * G["d_in"] * G["d_out"]
            if kind == "dW":
                by = 2 * n_keep * (G["d_out"] + G["d_in"]) + 4 * G["d_in"] * G["d_out"]
                fn = lambda G=G: R.dw(G["dy"], G["x"], keep, out=G["dw"], ws=G["ws_w"])
            else:
                by = 2 * n_keep * (G["d_out"] + G["d_in"]) + 2 * G["d_in"] * G["d_out"]
                fn = lambda G=G: R.dx(G["dy"], G["w"], keep, G["dx"], ws=G["ws_x"])
            t_ms = timed(fn, max(3, steps // 4))
            roof = max(fl / (pk_t * 1e12), by / (pk_b * 1e9)) * 1e3
            t_roof += roof
            fl_total += fl
            per.append({"gemm": f"{G['name']}.{kind}", "ms": t_ms,
                        "tflops": fl / (t_ms * 1e-3) / 1e12, "gbs": by / (t_ms * 1e-3) / 1e9,
                        "bound": "tensor" if fl / (pk_t * 1e12) > by / (pk_b * 1e9) else "hbm",
                        "frac": roof / t_ms})
    # what the row-sparse backward replaces: the dense full-row backward
    # (cuBLAS through torch), dW over all n_rows and dX for every row
    dense = []
    for G in gemms:
        dyf = torch.zeros(n_rows, G["d_out"], dtype=torch.bfloat16, device=dev)
        dyf[keep.long()] = G["dy"]
        dense.append((dyf, G))

    def dense_step():
        for dyf, G in dense:
            torch.mm(dyf.t(), G["x"])
            torch.mm(dyf, G["w"])

    dense_ms = timed(dense_step, max(3, steps // 10))
    clocks = sampler.stop()
    dom = max(per, key=lambda r: r["ms"])
    line = {"metric": "row-sparse projection backward (q, o, gate, up, down: dW and dX over the kept rows), TFLOP/s",
            "value": fl_total / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "n_gpus": 1,
            "steps": steps, "warmup": max(3, args.warmup), "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) X and dY, W scaled by in^-1/2)",
            "config": {"workload": w.name, "n_rows": n_rows, "n_keep": n_keep,
                       "hidden": w.hq * w.head_dim,
                       "intermediate": INTERMEDIATE.get(w.name, DEFAULT_INTERMEDIATE),
                       "dW": "fp32", "dX": "bf16", "l2": flush.describe()},
            "roofline": {"bound": "sum over the ten GEMMs of max(flops/peak, bytes/bw)",
                         "t_roof_ms": t_roof, "frac": t_roof / ms, "peak_tflops": pk_t,
                         "peak_gbs": pk_b, "peak_source": peak_src},
            "dominant": dom, "per_gemm": per,
            "dense_full_rows_ms": dense_ms, "speedup_vs_dense": dense_ms / ms,
            "gpu_launches": 10 * steps, "clocks": clocks}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="cfa", choices=["cfa", "reference"])
    ap.add_argument("--workload", default="qwen3_8b", choices=list(synth.WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--flush", default="write+read", choices=["write", "write+read"],
                    help="how L2 is evicted before each timed step")
    ap.add_argument("--rowsparse", action="store_true",
                    help="time the layer's row-sparse projection backward instead")
    ap.add_argument("--walk", type=int, default=0,
                    help="chunk rows: walk the workload's window chunk by chunk instead")
    ap.add_argument("--horizon", type=int, default=0,
                    help="prefix rows per window that get dK/dV (cfa_backward_horizon)")
    args = ap.parse_args()
    assert args.warmup >= 3 or args.impl == "reference", "at least 3 warm-up steps"

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    w = synth.workload(args.workload, seed=0)

    if args.impl == "reference":
        run_reference(args, w, rank)
        return
    if args.walk:
        run_walk(args, w)
        return
    if args.rowsparse:
        run_rowsparse(args, w)
        return

    import torch.distributed as dist
    import frozen_prefix_chunk_gb300 as cfa

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    cfa.lib(build_if_missing=True)

    # every rank has its own replica of the workload
    w = synth.workload(args.workload, seed=rank)
    host = synth.make_inputs(w)
    names = ("q", "k_prefix", "v_prefix", "k_chunk", "v_chunk", "dout",
             "cu_seqlens_prefix", "cu_seqlens_chunk")
    d = {k: host[k].to(dev) for k in names}
    a = cfa.make_args(d["q"], d["k_prefix"], d["v_prefix"], d["k_chunk"], d["v_chunk"],
                      d["cu_seqlens_prefix"], d["cu_seqlens_chunk"], max(w.lp), max(w.lc),
                      w.softmax_scale, w.prefix_dtype, hkv=w.hkv, total_lp=sum(w.lp))
    q8 = w.prefix_dtype == synth.PREFIX_Q8_0
    if q8:
        # The prefix is frozen, so one step dequantises it once (one
        # cfa_dequant_q8_0 launch per tensor) and both passes read the bf16
        # copy; handing the q8_0 prefix to cfa_forward and cfa_backward
        # instead would dequantise it inside each of them.
        kp16 = torch.empty(sum(w.lp), w.hkv, w.head_dim, dtype=torch.bfloat16, device=dev)
        vp16 = torch.empty_like(kp16)
        a = cfa.make_args(d["q"], kp16, vp16, d["k_chunk"], d["v_chunk"],
                          d["cu_seqlens_prefix"], d["cu_seqlens_chunk"], max(w.lp), max(w.lc),
                          w.softmax_scale, synth.PREFIX_BF16, hkv=w.hkv, total_lp=sum(w.lp))
    tc = sum(w.lc)
    o = torch.empty_like(d["q"])
    lse = torch.empty(w.hq, tc, dtype=torch.float32, device=dev)
    delta = torch.empty_like(lse)
    dq = torch.empty_like(d["q"])
    dk = torch.empty(tc, w.hkv, w.head_dim, dtype=torch.bfloat16, device=dev)
    dv = torch.empty_like(dk)
    ws_f = torch.empty(cfa.workspace_size(a, cfa.WS_FORWARD), dtype=torch.uint8, device=dev)
    ws_b = torch.empty(cfa.workspace_size(a, cfa.WS_BACKWARD), dtype=torch.uint8, device=dev)
    flush = L2Flush(dev, args.flush)
    dkp = dvp = None
    if args.horizon:
        dkp = torch.zeros(sum(w.lp), w.hkv, w.head_dim, dtype=torch.bfloat16, device=dev)
        dvp = torch.zeros_like(dkp)
    stream = torch.cuda.current_stream()
    # kernels launched per step: forward (+ split combine), delta, dQ (+ split
    # reduce), dK/dV; a workspace beyond its 256-byte header holds partials
    launches_per_step = (1 + (ws_f.numel() > 256)) + 1 + (1 + (ws_b.numel() > 256)) + 1 + 2 * q8

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        if q8:
            cfa.dequant_q8_0(d["k_prefix"], out_bf16=kp16, want_f32=False)
            cfa.dequant_q8_0(d["v_prefix"], out_bf16=vp16, want_f32=False)
        cfa.forward(a, d["q"], o, lse, ws_f)
        if ev:
            ev[1].record(stream)
        cfa.backward_preprocess(a, o, d["dout"], delta)
        if ev:
            ev[2].record(stream)
        # dQ on this stream; the library runs dK/dV beside it on a few SMs of
        # a second stream and joins it back before returning
        if args.horizon:
            cfa.backward_horizon(a, args.horizon, d["dout"], lse, delta, dq, dk, dv, dkp, dvp,
                                 ws_b)
        else:
            cfa.backward(a, d["dout"], lse, delta, dq, dk, dv, ws_b)
        if ev:
            ev[3].record(stream)

    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize()
    for ws in (ws_f, ws_b):
        st = cfa.read_status(ws)
        assert st == 0, f"device status {st}"

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    t_wall = time.perf_counter()
    for k in range(args.steps):
        flush()
        step(evs[k])
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    clocks = sampler.stop()
    if world > 1:
        dist.barrier()
    for ws in (ws_f, ws_b):
        assert cfa.read_status(ws) == 0

    step_ms = [e[0].elapsed_time(e[3]) for e in evs]
    fwd_ms = [e[0].elapsed_time(e[1]) for e in evs]
    bwd_ms = [e[2].elapsed_time(e[3]) for e in evs]
    tot_ms = slowest_rank_ms(sum(step_ms), world, dev)
    ms_per_step = tot_ms / args.steps

    flops = useful_flops(w, args.horizon)
    byts = algorithmic_bytes(w, args.horizon)
    value = job_tflops(world, flops["total"], ms_per_step)

    peaks, peak_src = load_peaks()
    bf16_peak = peaks["bf16_tflops"]
    hbm_peak = peaks["hbm_gbs"]
    # The dQ kernel (+ its split reduce) is the step's largest kernel.  It is
    # timed by the events around cfa_backward on its own stream: that span is
    # the dQ launch, or longer if the dK/dV kernel beside it (on a second
    # stream, its FLOPs not counted here) finished later.
    bwd_mean = statistics.mean(bwd_ms)
    achieved = flops["dq_kernel"] / (bwd_mean * 1e-3) / 1e12
    roofline = {"bound": "tensor", "achieved": achieved, "peak": bf16_peak, "unit": "TFLOP/s",
                "frac": achieved / bf16_peak, "traffic": recorded_traffic(w.name),
                "kernel": "bwd_dq_kernel + split reduce (timed as the cfa_backward span; "
                          "dK/dV runs beside it on a second stream)",
                "peak_source": f"bf16_tflops burst, {peak_src}",
                "algorithmic_flops_per_launch": flops["dq_kernel"], "ms_per_launch": bwd_mean}
    t_roof = max(flops["total"] / (bf16_peak * 1e12), byts["total"] / (hbm_peak * 1e9))
    step_roof = {"t_roof_ms": t_roof * 1e3, "frac": t_roof / (ms_per_step * 1e-3),
                 "fwd_ms": statistics.mean(fwd_ms), "bwd_ms": bwd_mean,
                 "bwd_tflops": (flops["dq_kernel"] + flops["dkdv_kernel"]) / (bwd_mean * 1e-3) / 1e12,
                 "fwd_tflops": flops["fwd"] / (statistics.mean(fwd_ms) * 1e-3) / 1e12,
                 "useful_gflop": flops["total"] / 1e9, "algorithmic_mb": byts["total"] / 1e6,
                 "peaks": f"bf16 {bf16_peak} TFLOP/s, HBM {hbm_peak} GB/s ({peak_src})"}

    # ---- end to end through the public API, host buffers, copies timed
    pin = {k: host[k].pin_memory() for k in names}
    outs = [o, lse, dq, dk, dv] + ([dkp, dvp] if args.horizon else [])
    outs_h = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
    h2d = sum(t.numel() * t.element_size() for t in pin.values())
    d2h = sum(t.numel() * t.element_size() for t in outs_h)
    e2e_ms = []
    for k in range(args.e2e_steps + 2):
        flush()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for n in names:
            d[n].copy_(pin[n], non_blocking=True)
        step()
        for src, dst in zip(outs, outs_h):
            dst.copy_(src, non_blocking=True)
        e1.record(stream)
        e1.synchronize()
        if k >= 2:
            e2e_ms.append(e0.elapsed_time(e1))
    e2e_val = job_tflops(world, flops["total"], statistics.mean(e2e_ms))

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        dt, f, desc = oracle_sample(host, 15.0, (0, 0))
        cpu = {"value": f / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.threads(),
               "kind": "oracle", "sample": desc, "seconds": dt}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16", "data": "synthetic (seeded N(0,1) q/k/v, N(0,0.1) dO)",
                "config": config_of(w, flush.describe(),
                                    args.horizon),
                "roofline": roofline, "step_roofline": step_roof,
                "cpu_baseline": cpu,
                "e2e": {"value": e2e_val, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                        "d2h_bytes_per_step": d2h, "ms_per_step": statistics.mean(e2e_ms)},
                "gpu_launches": launches_per_step * args.steps,
                "clocks": clocks, "wall_s_timed": t_wall}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
