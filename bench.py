#!/usr/bin/env python3
"""Throughput of the row-wise LayerNorm / RMSNorm forward on GB300.

One step = one forward call over the benchmark workload (RMSNorm fp32,
B=8 T=1024 C=4096: M=8192 rows of N=4096), inputs resident in HBM. Several
input/output sets are rotated so that no call finds its operands in L2, and
the calls are issued as CUDA-graph replays so that the device time per call
is not hidden behind host launch overhead.
The line printed reports achieved HBM GB/s of algorithmic bytes (read x,
write y, read the parameters, write 8 B/row of statistics for LayerNorm),
its fraction of the measured copy bandwidth, µs per call, the end-to-end
figure with host buffers, and the CPU oracle timed on the host cores.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl libnorm|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import glob
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_BYTES = 126 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
CLOCK_FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20000)
    p.add_argument("--warmup", type=int, default=50)
    p.add_argument("--impl", default="libnorm", choices=["libnorm", "reference"])
    p.add_argument("--workload", default=None)
    p.add_argument("--rows", type=int, default=None,
                   help="run the workload with this many rows instead of its own (a small case for profiling)")
    p.add_argument("--e2e-steps", type=int, default=30)
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--no-table", action="store_true", help="skip the per-workload table")
    return p.parse_args()


# ------------------------------------------------------------------ helpers

# The sources the forward kernels compile from: an ncu traffic figure below
# stays valid while these are unchanged.
FWD_KERNEL_SOURCES = ("norm_kernels.cuh", "norm_device.cuh", "norm_args.h")


def strip_comments(src: str) -> str:
    """C/C++ source without its comments and with runs of whitespace
    collapsed (string and character literals kept as written), so that the
    hash below follows the code and not its commentary."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            out.append(" ")
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash() -> str:
    """Hash of the forward kernel sources' code (comments and layout
    ignored): a traffic figure taken at one hash holds for any source with
    the same code."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "row_wise_normalization_ln_gb300", "csrc")
    for f in FWD_KERNEL_SOURCES:
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update(f.encode())
            h.update(strip_comments(fh.read()).encode())
    return h.hexdigest()[:16]


def measured_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# dram__bytes_read.sum + dram__bytes_write.sum of one launch, from the ncu
# capture summarised in profiles/ (workload -> (kernel source hash at capture,
# bytes per launch, summary file)).
NCU_TRAFFIC = {
    "rms_f32_8192x4096": ("6827a1cb9770479f", 206_823_936, "profiles/norm_fwd_cta_rms_f32_8192x4096.md"),
    "ln_bf16_4096x8192_outliers": ("6827a1cb9770479f", 86_684_928, "profiles/norm_fwd_cta_ln_bf16_4096x8192.md"),
    "rms_bf16_65536x2048": ("6827a1cb9770479f", 480_300_800, "profiles/norm_fwd_cta_rms_bf16_65536x2048.md"),
    "ln_f32_2048x65536": ("6827a1cb9770479f", 1_034_413_568, "profiles/norm_fwd_cta_ln_f32_2048x65536.md"),
    "ln_f32_8192x5000": ("6827a1cb9770479f", 269_315_328, "profiles/norm_fwd_cta_ln_f32_8192x5000.md"),
    "ln_f32_128x1024": ("6827a1cb9770479f", 544_512, "profiles/norm_fwd_cta_ln_f32_128x1024.md"),
    "fp8_ln_bf16_4096x8192_outliers": ("6827a1cb9770479f", 71_389_184, "profiles/norm_fwd_cta_fp8_ln_bf16_4096x8192.md"),
}


def ncu_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu capture, or None when the
    kernel sources changed since it was taken."""
    t = NCU_TRAFFIC.get(workload)
    return t[1] if t and t[0] == kernel_source_hash() else None


def kernel_name(w, plan) -> str:
    kind = "group" if plan["mapping"] == 0 else "cta"
    t = "float" if w.dtype == "f32" else "__nv_bfloat16"
    op = ("ADD+" if w.add else "") + ("LN" if w.op == "ln" else "RMS") + ("+E4M3" if w.fp8 else "")
    if w.bwd:
        return f"norm_bwd_cta<{t},{plan['vec_elems']},{plan['per_thread']},{op}>"
    return f"norm_fwd_{kind}<{t},{plan['vec_elems']},{plan['per_thread']},{op}>"


def op_name(w) -> str:
    return ("add+" if w.add else "") + w.op + ("_bwd" if w.bwd else "") + ("_fp8" if w.fp8 else "")


def metric_name(w) -> str:
    return f"LN/RMSNorm {'bwd' if w.bwd else 'fwd'} achieved HBM GB/s"


def plan_for(rn, w, num_sms):
    if w.bwd:
        return rn.make_bwd_plan(w.M, w.N, w.torch_dtype, w.op == "ln", True, num_sms)
    return rn.make_plan(w.M, w.N, w.torch_dtype, True, num_sms, add=w.add)


class ClockSampler:
    """nvidia-smi samples (200 ms) while the timed region runs."""

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.path = os.path.join("/tmp", f"libnorm_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        time.sleep(0.25)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.fh.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                if self.uuid and self.uuid not in parts[0]:
                    continue
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        reasons = set()
        for r in rows:
            for name, col in (("hw_slowdown", 5), ("hw_thermal_slowdown", 6), ("sw_thermal_slowdown", 7),
                              ("sw_power_cap", 8)):
                if r[col].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": num(rows[0][2]),
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max((num(r[3]) or 0.0) for r in rows)}


# ------------------------------------------------------------------ the GPU arm

def make_sets(w, inp, n_sets, device):
    import torch
    if w.bwd:
        return make_bwd_sets(w, inp, n_sets, device)
    sets = []
    for _ in range(n_sets):
        s = {"x": inp["x"].to(device),
             "y": torch.empty(w.M, w.N, dtype=torch.uint8 if w.fp8 else w.torch_dtype, device=device)}
        if w.add:
            s["r"] = inp["r"].to(device)
            s["h"] = torch.empty(w.M, w.N, dtype=w.torch_dtype, device=device)
        if w.op == "ln":
            s["mean"] = torch.empty(w.M, dtype=torch.float32, device=device)
            s["rstd"] = torch.empty(w.M, dtype=torch.float32, device=device)
        sets.append(s)
    params = {k: v.to(device) for k, v in inp.items() if k not in ("x", "r")}
    if w.fp8:
        params["scale"] = torch.tensor([w.qscale], dtype=torch.float32, device=device)
    return sets, params


def make_bwd_sets(w, inp, n_sets, device):
    """Backward sets: dy, x, dx per set (LayerNorm: the statistics of x from
    ln_fwd, computed once here, outside the timed region); the column
    gradients and the workspace are shared by the sets (calls are
    serialised on one stream)."""
    import torch
    import row_wise_normalization_ln_gb300 as rn
    params = {k: v.to(device) for k, v in inp.items() if k not in ("x", "dy")}
    sets = []
    for _ in range(n_sets):
        s = {"x": inp["x"].to(device), "dy": inp["dy"].to(device), "dx": torch.empty(w.M, w.N, dtype=w.torch_dtype,
                                                                                     device=device)}
        if w.op == "ln":
            _, s["mean"], s["rstd"] = rn.ln_fwd(s["x"], params["gamma"], params["beta"], w.eps, out=s["dx"])
        sets.append(s)
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    plan = rn.make_bwd_plan(w.M, w.N, w.torch_dtype, w.op == "ln", True, sms)
    nb = rn.bwd_workspace_bytes(plan, w.N, w.op == "ln")
    params["ws"] = torch.empty(max(nb, 16) // 4, dtype=torch.float32, device=device)
    params["dg"] = torch.empty(w.N, dtype=torch.float32, device=device)
    params["db"] = torch.empty(w.N, dtype=torch.float32, device=device)
    return sets, params


def step_fn(w, rn, params):
    if w.bwd and w.op == "ln":
        g, ws, dg, db = params["gamma"], params["ws"], params["dg"], params["db"]

        def f(s):
            rn.ln_bwd(s["dy"], s["x"], g, s["mean"], s["rstd"], dx=s["dx"], dgamma=dg, dbeta=db, workspace=ws)
    elif w.bwd:
        wt, ws, dg = params["w"], params["ws"], params["dg"]

        def f(s):
            rn.rms_bwd(s["dy"], s["x"], wt, w.eps, dx=s["dx"], dw=dg, workspace=ws)
    elif w.fp8 and w.op == "ln":
        g, b, sc = params["gamma"], params["beta"], params["scale"]

        def f(s):
            rn.ln_fwd_fp8(s["x"], g, b, sc, w.eps, residual=s.get("r"), h_out=s.get("h"), out=s["y"],
                          mean=s["mean"], rstd=s["rstd"])
    elif w.fp8:
        wt, sc = params["w"], params["scale"]

        def f(s):
            rn.rms_fwd_fp8(s["x"], wt, sc, w.eps, residual=s.get("r"), h_out=s.get("h"), out=s["y"])
    elif w.add and w.op == "ln":
        g, b = params["gamma"], params["beta"]

        def f(s):
            rn.ln_fwd_add(s["x"], s["r"], g, b, w.eps, h_out=s["h"], out=s["y"], mean=s["mean"], rstd=s["rstd"])
    elif w.add:
        wt = params["w"]

        def f(s):
            rn.rms_fwd_add(s["x"], s["r"], wt, w.eps, h_out=s["h"], out=s["y"])
    elif w.op == "ln":
        g, b = params["gamma"], params["beta"]

        def f(s):
            rn.ln_fwd(s["x"], g, b, w.eps, out=s["y"], mean=s["mean"], rstd=s["rstd"])
    else:
        wt = params["w"]

        def f(s):
            rn.rms_fwd(s["x"], wt, w.eps, out=s["y"])
    return f


def time_same_bytes_copy(w, inp, device, steps=600, per_graph=60):
    """Device time of torch's copy of one buffer into another, each as large
    as half the call's [M, N] traffic (x; x and r for the fused add; 1.5 [M, N]
    for the backward, which moves dy, x and dx): the algorithmic bytes minus
    parameters and statistics, over rotating sets larger than L2: what a
    plain copy of this size achieves. Timed both as graph replays and as
    plain launches, the faster kept: captured in a graph, torch's copy of
    512 MB or more becomes a memcpy node that runs at about half the copy
    bandwidth of the same copy launched directly."""
    import torch
    n = w.M * w.N * w.row_bytes // 2
    sets = [(torch.empty(n, dtype=torch.uint8, device=device), torch.empty(n, dtype=torch.uint8, device=device))
            for _ in range(n_sets_for(w))]
    for src, _ in sets:
        src.fill_(1.0)
    for src, dst in sets[:3]:
        dst.copy_(src)
    side = torch.cuda.Stream(device)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            for i in range(per_graph):
                src, dst = sets[i % len(sets)]
                dst.copy_(src)
    g.replay()
    torch.cuda.synchronize(device)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(steps // per_graph):
        g.replay()
    t1.record()
    torch.cuda.synchronize(device)
    graph_ms = t0.elapsed_time(t1) / (steps // per_graph * per_graph)
    plain = min(steps, 200)
    t0.record()
    for i in range(plain):
        src, dst = sets[i % len(sets)]
        dst.copy_(src)
    t1.record()
    torch.cuda.synchronize(device)
    plain_ms = t0.elapsed_time(t1) / plain
    del g, sets
    torch.cuda.empty_cache()
    return min(graph_ms, plain_ms)


def n_sets_for(w):
    per_set = w.row_bytes * w.M * w.N
    return max(3, math.ceil(3 * L2_BYTES / per_set))


def time_launches(w, rn, inp, device, steps, warmup, sampler=None, barrier=None, per_graph=100):
    """Time `steps` forward calls, issued as CUDA-graph replays of
    `per_graph` back-to-back calls over rotating input/output sets (no host
    work between kernels). Returns (total ms over the timed region, ms per
    call, clock summary)."""
    import torch
    sets, params = make_sets(w, inp, n_sets_for(w), device)
    f = step_fn(w, rn, params)
    for i in range(3):  # set-up: the library's per-kernel occupancy queries, before capture
        f(sets[i % len(sets)])
    torch.cuda.synchronize(device)
    per_graph = max(1, min(per_graph, steps))
    side = torch.cuda.Stream(device)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            for i in range(per_graph):
                f(sets[i % len(sets)])
    rest = steps % per_graph
    tail = None
    if rest:
        tail = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(tail, stream=side):
                for i in range(rest):
                    f(sets[i % len(sets)])
    graph.replay()  # uploads the graph
    torch.cuda.synchronize(device)
    stream = torch.cuda.current_stream(device)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    clocks = None
    ctx = sampler if sampler is not None else _Null()
    with ctx:
        # The W untimed warm-up steps come right before the timed region (the
        # clock sampler's start-up would otherwise leave the GPU idle for
        # 0.3 s between them), then the barrier and the synchronisation.
        for i in range(warmup):
            f(sets[i % len(sets)])
        if barrier:
            barrier()
        torch.cuda.synchronize(device)
        t0.record(stream)
        for _ in range(steps // per_graph):
            graph.replay()
        if tail is not None:
            tail.replay()
        t1.record(stream)
        torch.cuda.synchronize(device)
    if barrier:
        barrier()
    if sampler is not None:
        clocks = sampler.summary()
    total = t0.elapsed_time(t1)
    del graph, tail, sets
    torch.cuda.empty_cache()
    return total, total / steps, clocks


class _Null:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


def time_e2e_bwd(w, rn, inp, device, steps):
    """Backward end to end: H2D of dy, x, the parameter (and, for LayerNorm,
    the statistics, which ln_fwd computed once beforehand), the call, D2H of
    dx and the column gradients."""
    import torch
    ln = w.op == "ln"
    hin = {k: inp[k].pin_memory() for k in ("dy", "x", "gamma" if ln else "w")}
    din = {k: torch.empty_like(v, device=device) for k, v in hin.items()}
    if ln:
        xd = inp["x"].to(device)
        _, m, r = rn.ln_fwd(xd, inp["gamma"].to(device), inp["beta"].to(device), w.eps)
        hin["mean"], hin["rstd"] = m.cpu().pin_memory(), r.cpu().pin_memory()
        din["mean"], din["rstd"] = torch.empty_like(m), torch.empty_like(r)
        del xd
    dx = torch.empty_like(din["x"])
    hdx = torch.empty_like(hin["x"]).pin_memory()
    dg = torch.empty(w.N, dtype=torch.float32, device=device)
    db = torch.empty(w.N, dtype=torch.float32, device=device)
    hdg = torch.empty(w.N, dtype=torch.float32).pin_memory()
    hdb = torch.empty(w.N, dtype=torch.float32).pin_memory()
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    plan = rn.make_bwd_plan(w.M, w.N, w.torch_dtype, ln, True, sms)
    ws = torch.empty(max(rn.bwd_workspace_bytes(plan, w.N, ln), 16) // 4, dtype=torch.float32, device=device)
    h2d = sum(v.numel() * v.element_size() for v in hin.values())
    d2h = hdx.numel() * hdx.element_size() + (8 if ln else 4) * w.N

    def one():
        for k in hin:
            din[k].copy_(hin[k], non_blocking=True)
        if ln:
            rn.ln_bwd(din["dy"], din["x"], din["gamma"], din["mean"], din["rstd"], dx=dx, dgamma=dg, dbeta=db,
                      workspace=ws)
            hdb.copy_(db, non_blocking=True)
        else:
            rn.rms_bwd(din["dy"], din["x"], din["w"], w.eps, dx=dx, dw=dg, workspace=ws)
        hdg.copy_(dg, non_blocking=True)
        hdx.copy_(dx, non_blocking=True)

    for _ in range(3):
        one()
    torch.cuda.synchronize(device)
    stream = torch.cuda.current_stream(device)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(steps):
        one()
    t1.record(stream)
    torch.cuda.synchronize(device)
    return t0.elapsed_time(t1) / steps, h2d, d2h


def time_e2e(w, rn, inp, device, steps):
    """Host buffers in, host buffers out, through the library's public API:
    every step copies the parameters to the device and runs the call over
    the rows with ``host_rows_pipeline`` (row chunks copied in, normalised
    and copied back on three streams, so the two copy directions and the
    kernels overlap): x (and r) in, y (and h, and the statistics) out. The
    steps are a stream of batches (``wait=False``): a step's last copies
    back overlap the next step's first copies in; the timed region ends
    after every copy back of every step (``host_rows_wait``)."""
    if w.bwd:
        return time_e2e_bwd(w, rn, inp, device, steps)
    import torch
    hin = {k: v.pin_memory() for k, v in inp.items()}
    rowin = ["x"] + (["r"] if w.add else [])
    params = [k for k in hin if k not in rowin]
    dpar = {k: torch.empty_like(hin[k], device=device) for k in params}
    ydt = torch.uint8 if w.fp8 else w.torch_dtype
    hy = torch.empty(w.M, w.N, dtype=ydt).pin_memory()
    hh = torch.empty_like(hin["x"]).pin_memory() if w.add else None
    sc = torch.tensor([w.qscale], dtype=torch.float32, device=device) if w.fp8 else None
    ln = w.op == "ln"
    hm = torch.empty(w.M, dtype=torch.float32).pin_memory() if ln else None
    hr = torch.empty_like(hm).pin_memory() if ln else None
    outs = [hy] + ([hh] if w.add else []) + ([hm, hr] if ln else [])
    h2d = sum(v.numel() * v.element_size() for v in hin.values())
    d2h = hy.numel() * hy.element_size() + (hh.numel() * hh.element_size() if w.add else 0) + (8 * w.M if ln else 0)

    def call(ins, o):
        x, r = ins[0], (ins[1] if w.add else None)
        y, h = o[0], (o[1] if w.add else None)
        m, rs = (o[-2], o[-1]) if ln else (None, None)
        if w.fp8 and ln:
            rn.ln_fwd_fp8(x, dpar["gamma"], dpar["beta"], sc, w.eps, residual=r, h_out=h, out=y, mean=m, rstd=rs)
        elif w.fp8:
            rn.rms_fwd_fp8(x, dpar["w"], sc, w.eps, residual=r, h_out=h, out=y)
        elif ln and w.add:
            rn.ln_fwd_add(x, r, dpar["gamma"], dpar["beta"], w.eps, h_out=h, out=y, mean=m, rstd=rs)
        elif ln:
            rn.ln_fwd(x, dpar["gamma"], dpar["beta"], w.eps, out=y, mean=m, rstd=rs)
        elif w.add:
            rn.rms_fwd_add(x, r, dpar["w"], w.eps, h_out=h, out=y)
        else:
            rn.rms_fwd(x, dpar["w"], w.eps, out=y)

    def one():
        for k in params:
            dpar[k].copy_(hin[k], non_blocking=True)
        rn.host_rows_pipeline([hin[k] for k in rowin], outs, call, device=device, wait=False)

    for _ in range(3):
        one()
    rn.host_rows_wait(device)
    torch.cuda.synchronize(device)
    stream = torch.cuda.current_stream(device)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(steps):
        one()
    rn.host_rows_wait(device)
    t1.record(stream)
    torch.cuda.synchronize(device)
    ms = t0.elapsed_time(t1) / steps
    return ms, h2d, d2h


# ------------------------------------------------------------------ CPU oracle

def oracle_rows(w, inp, rows: int, r0: int = 0):
    """One call of the fp64 oracle over rows [r0, r0 + rows) (with an FP8
    output: the norm, then the quantisation of its values)."""
    import numpy as np
    import oracle

    def npx(t):
        import torch
        t = t.contiguous()
        return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()

    x = npx(inp["x"][r0:r0 + rows])
    e = oracle.eps_as_f32(w.eps)
    if w.bwd:
        dy = npx(inp["dy"][r0:r0 + rows])
        if w.op == "ln":
            return lambda: oracle.ln_bwd(dy, x, npx(inp["gamma"]), e)
        return lambda: oracle.rms_bwd(dy, x, npx(inp["w"]), e)
    if w.add:
        r = npx(inp["r"][r0:r0 + rows])
        if w.op == "ln":
            norm = lambda: oracle.ln_fwd_add(x, r, npx(inp["gamma"]), npx(inp["beta"]), e)[1]
        else:
            norm = lambda: oracle.rms_fwd_add(x, r, npx(inp["w"]), e)[1]
    elif w.op == "ln":
        norm = lambda: oracle.ln_fwd(x, npx(inp["gamma"]), npx(inp["beta"]), e)[0]
    else:
        norm = lambda: oracle.rms_fwd(x, npx(inp["w"]), e)[0]
    if w.fp8:
        return lambda: oracle.quant_e4m3(norm(), w.qscale)
    return norm


def cpu_baseline(w, inp, seconds: float):
    """The oracle as it stands, single-threaded, over whole passes of the
    workload until about `seconds` have elapsed."""
    run = oracle_rows(w, inp, w.M)
    passes = 0
    t0 = time.perf_counter()
    while True:
        run()
        passes += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    gbs = w.algorithmic_bytes() * passes / el / 1e9
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{passes} full pass(es) of {w.M}x{w.N} {w.dtype} in {el:.1f} s, fp64, 1 thread",
            "host_cores": os.cpu_count()}


def cpu_baseline_all_cores(w, inp, seconds: float):
    """The same oracle on every host core: the rows split into one block per
    core, each block run over and over by its own thread (the oracle is C
    called through ctypes, which releases the GIL) for about `seconds`."""
    from concurrent.futures import ThreadPoolExecutor
    n = max(1, min(os.cpu_count() or 1, w.M))
    bounds = [(w.M * i // n, w.M * (i + 1) // n) for i in range(n)]
    runs = [oracle_rows(w, inp, r1 - r0, r0) for r0, r1 in bounds]

    def spin(run):
        passes, t0 = 0, time.perf_counter()
        while True:
            run()
            passes += 1
            el = time.perf_counter() - t0
            if el >= seconds:
                return passes, el

    with ThreadPoolExecutor(n) as ex:
        res = list(ex.map(spin, runs))
    moved = sum(p * w.algorithmic_bytes(r1 - r0) for (p, _), (r0, r1) in zip(res, bounds))
    el = max(e for _, e in res)
    return {"value": round(moved / el / 1e9, 4), "unit": "GB/s", "cores": n, "kind": "oracle",
            "sample": f"{w.M} rows in {n} blocks, one thread each, {min(p for p, _ in res)}+ passes per block "
                      f"in {el:.1f} s, fp64"}


# ------------------------------------------------------------------ ranks

def max_over_ranks(ms: float, device) -> float:
    """The slowest rank's time (all ranks get it); the value itself alone."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(bytes_per_call: int, steps: int, world: int, max_ms: float) -> float:
    """Whole-job throughput: every rank normalised `steps` calls' worth of
    rows (weak scaling), timed by the slowest rank."""
    return bytes_per_call * steps * world / (max_ms / 1e3) / 1e9


# ------------------------------------------------------------------ main

def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def run_reference(args, w):
    """The reference arm: the fp64 CPU oracle (the only reference this
    method has), on this host's cores, same workload, metric and unit."""
    import torch
    from row_wise_normalization_ln_gb300 import workloads as wl
    rank, world, _ = dist_env()
    if rank != 0:
        return
    inp = wl.generate(w)
    probe_rows = max(1, min(w.M, 64))
    t0 = time.perf_counter()
    oracle_rows(w, inp, probe_rows)()
    per_row = (time.perf_counter() - t0) / probe_rows
    budget = 90.0
    rows = max(1, min(w.M, int(budget / (args.steps + args.warmup) / per_row)))
    run = oracle_rows(w, inp, rows)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    el = time.perf_counter() - t0
    gbs = w.algorithmic_bytes(rows) * args.steps / el / 1e9
    line = {
        "impl": "reference", "metric": metric_name(w), "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "op": op_name(w),
                   "io_dtype": w.dtype, "eps": w.eps, "sample_rows_per_step": rows},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{rows} of {w.M} rows per step, fp64, 1 thread"},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    from row_wise_normalization_ln_gb300 import workloads as wl
    w = wl.WORKLOADS[args.workload or wl.BENCH_WORKLOAD]
    if args.rows:
        w = w.scaled(M=args.rows)
    if args.impl == "reference":
        run_reference(args, w)
        return

    import torch
    import row_wise_normalization_ln_gb300 as rn
    rn.library()  # fails loudly if the CUDA library is not built
    rank, world, local = dist_env()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    barrier = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
        barrier = dist.barrier

    # Weak scaling: every rank normalises its own full workload (rows are
    # independent, so a row-sharded job needs no exchange at all).
    inp = wl.generate(w)
    props = torch.cuda.get_device_properties(device)
    uuid = str(getattr(props, "uuid", "")) or None
    sampler = ClockSampler(uuid) if rank == 0 else None
    total_ms, kern_ms, clocks = time_launches(w, rn, inp, device, args.steps, args.warmup, sampler, barrier)
    total_ms = max_over_ranks(total_ms, device)
    bytes_per_call = w.algorithmic_bytes()
    ms_per_step = total_ms / args.steps
    value = job_gbs(bytes_per_call, args.steps, world, total_ms)
    achieved = bytes_per_call / (kern_ms / 1e3) / 1e9
    peak, peak_src = measured_peak()
    traffic = ncu_traffic(w.name) if not args.rows else None  # the captures are of full-size launches

    e2e_ms, h2d, d2h = time_e2e(w, rn, inp, device, args.e2e_steps)

    table = None
    if not args.no_table and rank == 0:
        table = {}
        # The six configurations the headline metric is quoted on go last, so
        # that the end of the printed line (and of any log that keeps only
        # its tail) holds them.
        order = [n for n in wl.WORKLOADS if n not in wl.BASELINE_CONFIGS] + list(wl.BASELINE_CONFIGS)
        for name in order:
            wk = wl.WORKLOADS[name]
            wi = inp if name == w.name else wl.generate(wk)
            _, ms, _ = time_launches(wk, rn, wi, device, 600, 10, per_graph=60)
            us = ms * 1e3
            gbs = wk.algorithmic_bytes() / (us / 1e6) / 1e9
            copy_us = time_same_bytes_copy(wk, wi, device) * 1e3
            table[name] = {"us_per_call": round(us, 3), "GBps": round(gbs, 1),
                           "frac_of_measured_peak": round(gbs / peak, 4),
                           "same_size_copy_us": round(copy_us, 3),
                           # achieved GB/s over the same-size copy's GB/s
                           "frac_of_same_size_copy": round(
                               gbs / ((wk.row_bytes * wk.M * wk.N) / (copy_us / 1e6) / 1e9), 4),
                           "rows_per_s": round(wk.M / (us / 1e6)), "plan": plan_for(rn, wk, props.multi_processor_count)}
            del wi

    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    cpu = cpu_baseline(w, inp, args.cpu_seconds)
    cpu_all = cpu_baseline_all_cores(w, inp, args.cpu_seconds)
    line = {
        "metric": metric_name(w), "value": round(value, 2), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 6),
        "us_per_call": round(kern_ms * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "op": op_name(w), "M": w.M, "N": w.N,
                   "io_dtype": w.dtype, "eps": w.eps,
                   "algorithmic_bytes_per_call": bytes_per_call,
                   "l2": f"{n_sets_for(w)} rotating input/output sets of "
                         f"{w.row_bytes * w.M * w.N >> 20} MiB "
                         f"(> L2 between reuses)",
                   "parallelism": f"replicas x{world} (rows independent)"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": peak_src, "traffic": traffic,
                     "kernel": kernel_name(w, plan_for(rn, w, props.multi_processor_count)),
                     "kernel_hash": kernel_source_hash()},
        "e2e": {"value": round(bytes_per_call / (e2e_ms / 1e3) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4)},
        "gpu_launches": args.steps * (2 if w.bwd else 1),  # the backward adds its column-sum kernel
        "clocks": clocks,
        "cpu_baseline": cpu,
        "cpu_baseline_all_cores": cpu_all,
        "gpu": props.name,
        "workloads": table,
    }
    if w.dtype == "bf16":
        line["dtype"] = "bf16 io, f32 compute"
    if table is not None:
        # The six configurations again, compactly, as the line's last key:
        # µs per call, GB/s, fraction of the measured copy bandwidth, of the
        # nominal 8 TB/s, and the µs of a same-size copy.
        line["baseline_configs"] = {
            n: {"us": table[n]["us_per_call"], "GBps": table[n]["GBps"],
                "of_measured": table[n]["frac_of_measured_peak"],
                "of_8TBps": round(table[n]["GBps"] / 8000.0, 4), "copy_us": table[n]["same_size_copy_us"]}
            for n in wl.BASELINE_CONFIGS}
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
