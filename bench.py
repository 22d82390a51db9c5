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
buffer left to do (--flush write keeps only the write).  Under torchrun every
rank runs its own replica of the workload, with the same shapes (weak scaling,
no collective on the data path); value = all ranks' FLOPs (a SUM all-reduce)
over the slowest rank's time (a MAX all-reduce).

The headline workload is the 63k-token window with its q8_0 prefix handed to
the library as it is; the other configurations the roofline target names
(the Qwen3-8B layer and the varlen batch) are timed in the same run, each
long enough for the clock sampler to see it under load, and reported under
"extra" with their own step roofline and dominant-kernel roofline.

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
                 "-i", str(device_index), "-lms", "50"], stdout=self.f,
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

def _group_inputs(inp, b, hk, lc_sub, nh=1):
    """The first lc_sub chunk rows of window b, KV heads hk .. hk + nh - 1
    (and their query heads), as a one-window workload (rows before lc_sub see
    exactly the same keys)."""
    w = inp["workload"]
    g = w.hq // w.hkv
    cu_p = inp["cu_seqlens_prefix"].tolist()
    cu_c = inp["cu_seqlens_chunk"].tolist()
    c0, p0, p1 = cu_c[b], cu_p[b], cu_p[b + 1]
    sub = synth.custom(hq=g * nh, hkv=nh, head_dim=w.head_dim, lp=[p1 - p0], lc=[lc_sub],
                       prefix_dtype=w.prefix_dtype, softmax_scale=w.softmax_scale,
                       name=w.name)
    heads = slice(hk * g, (hk + nh) * g)
    rows = slice(c0, c0 + lc_sub)
    return dict(q=inp["q"][rows, heads].contiguous(),
                k_prefix=inp["k_prefix"][p0:p1, hk:hk + nh].contiguous(),
                v_prefix=inp["v_prefix"][p0:p1, hk:hk + nh].contiguous(),
                k_chunk=inp["k_chunk"][rows, hk:hk + nh].contiguous(),
                v_chunk=inp["v_chunk"][rows, hk:hk + nh].contiguous(),
                dout=inp["dout"][rows, heads].contiguous(),
                cu_seqlens_prefix=synth.cu_seqlens([p1 - p0]),
                cu_seqlens_chunk=synth.cu_seqlens([lc_sub]), workload=sub)


def oracle_sample(inp, budget_s, group=(0, 0)):
    """Time the oracle, as it stands, on a bounded sample of about budget_s:
    the first rows of the (window, KV head) group, or, when the whole group
    takes less, all chunk rows of that window's KV heads from hk on, as many
    as fit (calibrated on the group's first 32 rows, enough to keep the
    oracle's threads busy).  Returns (seconds, useful FLOPs of the sample,
    text)."""
    import oracle

    oracle.build()
    w = inp["workload"]
    b, hk = group
    lc = w.lc[b]
    n_probe = min(lc, 32)
    probe = _group_inputs(inp, b, hk, n_probe)
    t0 = time.perf_counter()
    oracle.run(probe)
    per_row = (time.perf_counter() - t0) / n_probe
    rows = budget_s / max(per_row, 1e-9)
    if rows <= lc:
        lc_sub, nh = max(1, int(rows)), 1
    else:
        lc_sub, nh = lc, max(1, min(w.hkv - hk, int(rows / lc)))
    sub = _group_inputs(inp, b, hk, lc_sub, nh)
    t0 = time.perf_counter()
    oracle.run(sub)
    dt = time.perf_counter() - t0
    f = useful_flops(sub["workload"])["total"]
    heads = f"kv head {hk}" if nh == 1 else f"kv heads {hk}..{hk + nh - 1}"
    desc = (f"oracle fwd+bwd of chunk rows 0..{lc_sub - 1} of window {b}, {heads} of "
            f"{w.name} ({w.hq // w.hkv} query heads each, Lp={w.lp[b]}, Lc={lc_sub} of {lc})")
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
                             "kind": "oracle",
                             "sample": desc + " (the last step's; each step samples from the "
                                              "next (window, KV head) group on)"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def config_of(w, l2, horizon=0, q8="product"):
    if w.prefix_dtype != synth.PREFIX_Q8_0:
        prefix = "bf16"
    elif q8 == "export":
        prefix = "q8_0 (expanded to bf16 once per step by cfa_dequant_q8_0, read by both passes)"
    else:
        prefix = "q8_0 (handed to cfa_forward / cfa_backward as it is)"
    return {"workload": w.name, "batch": w.batch, "hq": w.hq, "hkv": w.hkv, "horizon": horizon,
            "head_dim": w.head_dim, "lp": w.lp, "lc": w.lc, "prefix": prefix,
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


# ------------------------------------------------------- the attention step --

# the configurations the >= 60 %-of-roofline target names
TARGETS = ("qwen3_8b", "window_63k_q8", "varlen8")
# launches of the library per step: forward, split merge, delta, dQ, dQ reduce, dK/dV
LAUNCHES_ATTN = 6


class AttnStep:
    """One workload resident in HBM and its fwd+bwd step through the C ABI.

    The step is cfa_forward, cfa_backward_preprocess and cfa_backward (dQ on
    the caller's stream, dK/dV beside it on the library's second stream,
    joined back), or cfa_backward_horizon with a horizon.  A q8_0 prefix is
    handed to the library as it is ("product", the path a caller with a q8_0
    cache takes); q8 = "export" instead expands it once per step through
    cfa_dequant_q8_0 into bf16 buffers that both passes read."""

    def __init__(self, w, dev, horizon=0, q8="product"):
        import frozen_prefix_chunk_gb300 as cfa
        self.cfa, self.w, self.dev, self.horizon = cfa, w, dev, horizon
        self.host = synth.make_inputs(w)
        names = ("q", "k_prefix", "v_prefix", "k_chunk", "v_chunk", "dout",
                 "cu_seqlens_prefix", "cu_seqlens_chunk")
        self.names = names
        self.q8 = q8 if w.prefix_dtype == synth.PREFIX_Q8_0 else None
        if self.q8 == "export":
            self.kp16 = torch.empty(sum(w.lp), w.hkv, w.head_dim, dtype=torch.bfloat16, device=dev)
            self.vp16 = torch.empty_like(self.kp16)
        self.io = self.make_io({k: self.host[k].to(dev) for k in names})
        self.d = self.io["d"]
        self.a = self.io["a"]
        self.ws_f = torch.empty(cfa.workspace_size(self.a, cfa.WS_FORWARD), dtype=torch.uint8,
                                device=dev)
        self.ws_b = torch.empty(cfa.workspace_size(self.a, cfa.WS_BACKWARD), dtype=torch.uint8,
                                device=dev)
        self.stream = torch.cuda.current_stream()
        # library launches per step: the six attention kernels, plus the
        # prefix expansion (q8_0 / fp16) inside each pass or the two exports
        self.launches = LAUNCHES_ATTN + (2 if self.q8 else 0)
        self.flops = useful_flops(w, horizon)
        self.bytes = algorithmic_bytes(w, horizon)

    def make_io(self, d):
        """The arguments and output buffers of a step over the device inputs
        `d` (tensors shaped like the host inputs).  Steps over different
        input sets share the workspaces (and, for q8 = "export", the bf16
        prefix buffers), so they must run one after the other on one stream."""
        cfa, w, dev = self.cfa, self.w, self.dev
        pref = w.prefix_dtype
        kp, vp = d["k_prefix"], d["v_prefix"]
        if self.q8 == "export":
            kp, vp, pref = self.kp16, self.vp16, synth.PREFIX_BF16
        a = cfa.make_args(d["q"], kp, vp, d["k_chunk"], d["v_chunk"], d["cu_seqlens_prefix"],
                          d["cu_seqlens_chunk"], max(w.lp), max(w.lc), w.softmax_scale, pref,
                          hkv=w.hkv, total_lp=sum(w.lp))
        tc = sum(w.lc)
        io = dict(d=d, a=a, o=torch.empty_like(d["q"]),
                  lse=torch.empty(w.hq, tc, dtype=torch.float32, device=dev),
                  dq=torch.empty_like(d["q"]),
                  dk=torch.empty(tc, w.hkv, w.head_dim, dtype=torch.bfloat16, device=dev),
                  dkp=None, dvp=None)
        io["delta"] = torch.empty_like(io["lse"])
        io["dv"] = torch.empty_like(io["dk"])
        if self.horizon:
            io["dkp"] = torch.zeros(sum(w.lp), w.hkv, w.head_dim, dtype=torch.bfloat16, device=dev)
            io["dvp"] = torch.zeros_like(io["dkp"])
        return io

    # the first input set's outputs
    o = property(lambda self: self.io["o"])
    lse = property(lambda self: self.io["lse"])
    delta = property(lambda self: self.io["delta"])
    dq = property(lambda self: self.io["dq"])
    dk = property(lambda self: self.io["dk"])
    dv = property(lambda self: self.io["dv"])
    dkp = property(lambda self: self.io["dkp"])
    dvp = property(lambda self: self.io["dvp"])

    def step(self, ev=None, io=None):
        cfa, s = self.cfa, self.stream
        io = io or self.io
        d, a = io["d"], io["a"]
        if ev:
            ev[0].record(s)
        if self.q8 == "export":
            cfa.dequant_q8_0(d["k_prefix"], out_bf16=self.kp16, want_f32=False)
            cfa.dequant_q8_0(d["v_prefix"], out_bf16=self.vp16, want_f32=False)
        cfa.forward(a, d["q"], io["o"], io["lse"], self.ws_f)
        if ev:
            ev[1].record(s)
        cfa.backward_preprocess(a, io["o"], d["dout"], io["delta"])
        if ev:
            ev[2].record(s)
        if self.horizon:
            cfa.backward_horizon(a, self.horizon, d["dout"], io["lse"], io["delta"], io["dq"],
                                 io["dk"], io["dv"], io["dkp"], io["dvp"], self.ws_b)
        else:
            cfa.backward(a, d["dout"], io["lse"], io["delta"], io["dq"], io["dk"], io["dv"],
                         self.ws_b)
        if ev:
            ev[3].record(s)

    def capture(self, io=None):
        """Capture one step (the same C-ABI calls, on a side stream) into a
        CUDA graph; replay() then launches the whole step at once.  The
        library's calls are capture-safe: no host synchronisation, no
        allocation, its second stream forked and joined with events.  With
        `io` (an input / output set from make_io) the graph is returned for
        that set instead."""
        s = torch.cuda.Stream(device=self.dev)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self.step(io=io)  # first call on this stream: outside the capture
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s, capture_error_mode="relaxed"):
            self.step(io=io)
        torch.cuda.synchronize()
        if io is not None:
            return graph
        self.graph = graph

    def replay(self, ev=None):
        s = self.stream
        if ev:
            ev[0].record(s)
        self.graph.replay()
        if ev:
            ev[3].record(s)

    def check_status(self):
        for ws in (self.ws_f, self.ws_b):
            st = self.cfa.read_status(ws)
            assert st == 0, f"device status {st}"

    def outputs(self, io=None):
        io = io or self.io
        outs = [io["o"], io["lse"], io["dq"], io["dk"], io["dv"]]
        return outs + ([io["dkp"], io["dvp"]] if self.horizon else [])


def e2e_pipelined(case, pin, outs_h, steps, flush, dev):
    """Milliseconds per step of `steps` steps through the public API with host
    inputs and outputs (each step one replay of its C-ABI calls captured as a
    CUDA graph, as in the timed steps), pipelined the way a training loop
    streams its data:
    step k's inputs are copied in from pinned host memory on one copy stream
    while step k-1 runs, and its outputs copied out to pinned host memory on
    another while step k+1 runs.  Two sets of device inputs and outputs
    alternate; a set is refilled only after the step that used it is done and
    its outputs have been read.  L2 is flushed once before the first step.
    One pair of events spans everything: the first input copy to the last
    output copy."""
    s = case.stream
    ios = [case.io, case.make_io({k: torch.empty_like(v) for k, v in case.d.items()})]
    # each set's step captured once, as the timed steps are (the same C-ABI calls)
    for io in ios:
        for n in case.names:
            io["d"][n].copy_(pin[n])
    graphs = [case.capture(io) for io in ios]
    h2d_s, d2h_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    in_ready = [torch.cuda.Event() for _ in range(2)]
    computed = [torch.cuda.Event() for _ in range(2)]
    out_read = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]
    flush()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(h2d_s)
    for k in range(steps):
        b = k % 2
        io = ios[b]
        if used[b]:
            h2d_s.wait_event(computed[b])
        with torch.cuda.stream(h2d_s):
            for n in case.names:
                io["d"][n].copy_(pin[n], non_blocking=True)
        in_ready[b].record(h2d_s)
        s.wait_event(in_ready[b])
        if used[b]:
            s.wait_event(out_read[b])
        graphs[b].replay()
        computed[b].record(s)
        d2h_s.wait_event(computed[b])
        with torch.cuda.stream(d2h_s):
            for src, dst in zip(case.outputs(io), outs_h):
                dst.copy_(src, non_blocking=True)
        out_read[b].record(d2h_s)
        used[b] = True
    s.wait_stream(d2h_s)
    s.wait_stream(h2d_s)
    e1.record(s)
    e1.synchronize()
    case.check_status()
    return e0.elapsed_time(e1) / steps


def time_steps(case, steps, warmup, flush, world, dev, sampler_index=None, launch="graph"):
    """W untimed warm-up steps, then exactly `steps` steps, each bracketed by
    CUDA events on the launching stream, L2 flushed before each outside the
    events; barrier + synchronize on both sides.  launch = "graph": the step
    is captured once as a CUDA graph and each timed step is one replay (the
    forward / backward split then comes from a short run of stream-launched
    steps before the timed region, which is also reported); "stream": each
    timed step launches the calls one by one.  Returns per-step lists of the
    step, forward and backward times (ms), the slowest rank's total, the
    clock record, the wall time of the timed loop and the stream-launched
    step times."""
    import torch.distributed as dist
    for _ in range(warmup):
        flush()
        case.step()
    torch.cuda.synchronize()
    case.check_status()

    def stream_run(n):
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n)]
        for k in range(n):
            flush()
            case.step(evs[k])
        torch.cuda.synchronize()
        return evs

    split = None
    if launch == "graph":
        split = stream_run(min(steps, 50))
        case.capture()
        for _ in range(3):
            flush()
            case.replay()
        torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(sampler_index) if sampler_index is not None else None
    t_wall = time.perf_counter()
    for k in range(steps):
        flush()
        if launch == "graph":
            case.replay(evs[k])
        else:
            case.step(evs[k])
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    clocks = sampler.stop() if sampler else None
    if world > 1:
        dist.barrier()
    case.check_status()
    step_ms = [e[0].elapsed_time(e[3]) for e in evs]
    sp = split if split is not None else evs
    fwd_ms = [e[0].elapsed_time(e[1]) for e in sp]
    bwd_ms = [e[2].elapsed_time(e[3]) for e in sp]
    stream_ms = [e[0].elapsed_time(e[3]) for e in sp]
    tot_ms = slowest_rank_ms(sum(step_ms), world, dev)
    return dict(step_ms=step_ms, fwd_ms=fwd_ms, bwd_ms=bwd_ms, tot_ms=tot_ms, clocks=clocks,
                wall_s=t_wall, stream_ms=stream_ms, launch=launch)


def summarise(case, t, steps, world, dev, peaks, peak_src):
    """Value, step roofline and the dominant kernel's roofline of one timed run."""
    w, flops, byts = case.w, case.flops, case.bytes
    ms_per_step = t["tot_ms"] / steps
    value = job_tflops_sum(flops["total"], ms_per_step, world, dev)
    bf16_peak, hbm_peak = peaks["bf16_tflops"], peaks["hbm_gbs"]
    fwd_mean, bwd_mean = statistics.mean(t["fwd_ms"]), statistics.mean(t["bwd_ms"])
    # The dQ kernel (+ its split reduce) is the step's largest kernel.  It is
    # timed by the events around cfa_backward on its own stream: that span is
    # the dQ launch, or longer if the dK/dV kernel beside it (on a second
    # stream, its FLOPs not counted here) finished later, or if the call first
    # expands a q8_0 prefix into its workspace.
    achieved = flops["dq_kernel"] / (bwd_mean * 1e-3) / 1e12
    roofline = {"bound": "tensor", "achieved": achieved, "peak": bf16_peak, "unit": "TFLOP/s",
                "frac": achieved / bf16_peak, "traffic": recorded_traffic(w.name),
                "kernel": "bwd_dq_kernel + split reduce (timed as the cfa_backward span, a lower "
                          "bound: dK/dV runs beside it on a second stream"
                          + (", and the span includes the call's q8_0 expansion" if case.q8 ==
                             "product" else "") + ")",
                "peak_source": f"bf16_tflops burst, {peak_src}",
                "algorithmic_flops_per_launch": flops["dq_kernel"], "ms_per_launch": bwd_mean}
    t_roof = max(flops["total"] / (bf16_peak * 1e12), byts["total"] / (hbm_peak * 1e9))
    step_roof = {"t_roof_ms": t_roof * 1e3, "frac": t_roof / (ms_per_step * 1e-3),
                 "fwd_ms": fwd_mean, "bwd_ms": bwd_mean,
                 "bwd_tflops": (flops["dq_kernel"] + flops["dkdv_kernel"]) / (bwd_mean * 1e-3) / 1e12,
                 "fwd_tflops": flops["fwd"] / (fwd_mean * 1e-3) / 1e12,
                 "useful_gflop": flops["total"] / 1e9, "algorithmic_mb": byts["total"] / 1e6,
                 "peaks": f"bf16 {bf16_peak} TFLOP/s, HBM {hbm_peak} GB/s ({peak_src})",
                 "launch": t["launch"]}
    if t["launch"] == "graph":
        # the same step with the calls launched one by one on the stream
        st_ms = statistics.mean(t["stream_ms"])
        step_roof["stream_launch"] = {"ms_per_step": st_ms, "frac": t_roof / (st_ms * 1e-3),
                                      "steps": len(t["stream_ms"])}
    return ms_per_step, value, roofline, step_roof


def job_tflops_sum(flops_rank: float, ms_per_step: float, world: int, device) -> float:
    """Whole-job useful TFLOP/s: the FLOPs of all ranks (a SUM all-reduce, so
    replicas of different sizes are counted as they are) over the slowest
    rank's time per step."""
    total = flops_rank
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([float(flops_rank)], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.SUM)
        total = float(t.item())
    return total / (ms_per_step * 1e-3) / 1e12


def extra_steps(case, flush, want_s=0.3, lo=20, hi=4000):
    """Steps for an extra workload's timed region: about `want_s` seconds, so
    the clock sampler sees it under load (estimated from three steps)."""
    for _ in range(2):
        flush()
        case.step()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(3):
        flush()
        case.step()
    torch.cuda.synchronize()
    per = (time.perf_counter() - t0) / 3
    return max(lo, min(hi, int(want_s / max(per, 1e-6))))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="cfa", choices=["cfa", "reference"])
    ap.add_argument("--workload", default="window_63k_q8", choices=list(synth.WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="time the headline workload only (not the other target configs)")
    ap.add_argument("--q8", default="product", choices=["product", "export"],
                    help="q8_0 prefix: handed to the library as it is, or expanded once per "
                         "step through cfa_dequant_q8_0 and read as bf16")
    ap.add_argument("--launch", default="graph", choices=["graph", "stream"],
                    help="each timed step: one replay of the step captured as a CUDA graph "
                         "(through the same C-ABI calls), or the calls launched one by one")
    ap.add_argument("--flush", default="write+read", choices=["write", "write+read"],
                    help="how L2 is evicted before each timed step")
    ap.add_argument("--rowsparse", action="store_true",
                    help="time the layer's row-sparse projection backward instead")
    ap.add_argument("--walk", type=int, default=0,
                    help="chunk rows: walk the workload's window chunk by chunk instead")
    ap.add_argument("--horizon", type=int, default=0,
                    help="prefix rows per window that get dK/dV (cfa_backward_horizon)")
    ap.add_argument("--lp", type=int, default=0,
                    help="override every window's prefix length (smaller cases of the same "
                         "kernels, for profiler captures)")
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
    flush = L2Flush(dev, args.flush)
    peaks, peak_src = load_peaks()

    # Every rank has its own replica of the workload: the same shapes (the
    # varlen window lengths drawn with seed 0), values seeded by the rank.
    def make_case(name, horizon=0):
        wl = synth.workload(name, seed=rank, shape_seed=0)
        if args.lp:
            wl.lp = [args.lp] * wl.batch
            wl.shape_seed = -1   # lengths no longer those the seed draws
        return AttnStep(wl, dev, horizon, args.q8)

    # ---- the other target configurations, each timed on its own, long
    # enough for the clock sampler to see it under load
    extras = {}
    if not args.no_extras and not args.horizon:
        for name in TARGETS:
            if name == args.workload:
                continue
            case = make_case(name)
            n = extra_steps(case, flush)
            if world > 1:
                t = torch.tensor([n], dtype=torch.int64, device=dev)
                dist.all_reduce(t, op=dist.ReduceOp.MAX)
                n = int(t.item())
            t = time_steps(case, n, args.warmup, flush, world, dev, sampler_index=local,
                           launch=args.launch)
            ms, val, roof, sroof = summarise(case, t, n, world, dev, peaks, peak_src)
            extras[name] = {"value": val, "unit": "TFLOP/s", "ms_per_step": ms, "steps": n,
                            "step_roofline": sroof, "roofline": roof,
                            "config": config_of(case.w, flush.describe(), 0, case.q8),
                            "gpu_launches": case.launches * n, "clocks": t["clocks"]}
            del case
            torch.cuda.empty_cache()

    # ---- the headline workload: exactly K timed steps
    case = make_case(args.workload, args.horizon)
    t = time_steps(case, args.steps, args.warmup, flush, world, dev, sampler_index=local,
                   launch=args.launch)
    ms_per_step, value, roofline, step_roof = summarise(case, t, args.steps, world, dev, peaks,
                                                        peak_src)

    # ---- end to end through the public API, host buffers, copies timed
    host, d, stream = case.host, case.d, case.stream
    pin = {k: host[k].pin_memory() for k in case.names}
    outs = case.outputs()
    outs_h = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs]
    h2d = sum(v.numel() * v.element_size() for v in pin.values())
    d2h = sum(v.numel() * v.element_size() for v in outs_h)
    # one step at a time (copy in, step, copy out; L2 flushed before each)
    serial_ms = []
    for k in range(args.e2e_steps + 2):
        flush()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for n in case.names:
            d[n].copy_(pin[n], non_blocking=True)
        case.step()
        for src, dst in zip(outs, outs_h):
            dst.copy_(src, non_blocking=True)
        e1.record(stream)
        e1.synchronize()
        if k >= 2:
            serial_ms.append(e0.elapsed_time(e1))
    # as a training loop streams its inputs: every step's copies, overlapped
    e2e_pipe_ms = e2e_pipelined(case, pin, outs_h, 2, flush, dev)
    e2e_pipe_ms = e2e_pipelined(case, pin, outs_h, args.e2e_steps, flush, dev)
    e2e_val = job_tflops_sum(case.flops["total"], e2e_pipe_ms, world, dev)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        dt, f, desc = oracle_sample(host, 15.0, (0, 0))
        cpu = {"value": f / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.threads(),
               "kind": "oracle", "sample": desc, "seconds": dt}

    if rank == 0:
        fracs = {args.workload: step_roof["frac"]}
        fracs.update({k: v["step_roofline"]["frac"] for k, v in extras.items()})
        line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16", "data": "synthetic (seeded N(0,1) q/k/v, N(0,0.1) dO)",
                "config": config_of(case.w, flush.describe(), args.horizon, case.q8),
                "roofline": roofline, "step_roofline": step_roof,
                "cpu_baseline": cpu,
                "e2e": {"value": e2e_val, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                        "d2h_bytes_per_step": d2h, "ms_per_step": e2e_pipe_ms,
                        "steps": args.e2e_steps,
                        "overlap": "pipelined: each step's inputs copied in from pinned host "
                                   "memory on a copy stream while the previous step runs, its "
                                   "outputs copied out on another while the next one runs "
                                   "(two input / output sets alternate); one event pair spans "
                                   "all steps, every copy inside it",
                        "serial_ms_per_step": statistics.mean(serial_ms),
                        "serial_value": job_tflops_sum(case.flops["total"],
                                                       statistics.mean(serial_ms), world, dev)},
                "gpu_launches": case.launches * args.steps,
                "launch": ("cuda_graph (one step captured through the C-ABI calls, one replay "
                           "per timed step; step_roofline.stream_launch has the same step "
                           "launched call by call)" if args.launch == "graph" else "stream"),
                "clocks": t["clocks"], "wall_s_timed": t["wall_s"],
                "target_step_fracs": fracs, "extra": extras}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
