#!/usr/bin/env python
"""Benchmark of the q8ta int8 quantized contraction hot path on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
  1. quantize_per_tensor        fp32 [64Mi] -> int8                (HBM bound)
  2. quantize -> q8ta_linear   fp32 [2048, 4096] -> int8 x_q + the bf16 operand,
                                then the GEMM 2048 x 4096 x 11008 with a packed
                                weight (two kernels under programmatic dependent
                                launch; tensor cores)
  3. q8ta_linear_gemv           1 x 4096 x 4096                    (HBM bound)
  4. q8ta_conv2d_transposed     [8,256,64,64] -> [8,128,128,128], K=3 s=2 p=1 op=1

value = int8 TOPS of the step: (2*M*N*K of the linear + 2*K*N of the gemv +
2 * valid-tap MACs of the transposed convolution) / step time.  Per-op
figures (GB/s, TOPS, outputs/s) are reported under "ops".

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun every rank runs its own replica (the ops are data parallel:
independent problems, no collective on the data path); value sums all ranks.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "q8ta_linear int8 TOPS & gemv/quantize HBM GB/s vs roofline; conv_t outputs/s"

# ---- workload sizes (the five benchmark workloads of the q8ta pages) -------
Q = synth.CONFIGS["quantize_64Mi"]
L = synth.CONFIGS["linear_chain_2048x4096x11008"]
G = synth.CONFIGS["gemv_1x4096x4096"]
C = synth.CONFIGS["conv_t_8x256x64x64_k3s2"]

QN = Q.dims["numel"]
LM, LK, LN = L.dims["M"], L.dims["K"], L.dims["N"]
GK, GN = G.dims["K"], G.dims["N"]
CD = C.dims
CHo, CWo = synth.output_hw(CD["H_in"], CD["W_in"], CD["Kh"], CD["Kw"], CD["s"], CD["s"], CD["p"],
                           CD["p"], CD["op"], CD["op"])


def conv_valid_macs(d, Ho, Wo):
    """Multiply-adds over valid taps only (the work the op defines): the
    valid (kh, kw) pairs of an output factor into valid rows x valid columns."""
    def valid(o, K, n_in):
        return sum(1 for k in range(K)
                   if (o + d["p"] - k) >= 0 and (o + d["p"] - k) % d["s"] == 0
                   and (o + d["p"] - k) // d["s"] < n_in)
    rows = sum(valid(o, d["Kh"], d["H_in"]) for o in range(Ho))
    cols = sum(valid(o, d["Kw"], d["W_in"]) for o in range(Wo))
    return d["N"] * d["OC"] * d["IC"] * rows * cols


OPS_LINEAR = 2 * LM * LN * LK
OPS_GEMV = 2 * GK * GN
CONV_MACS = conv_valid_macs(CD, CHo, CWo)
OPS_CONV = 2 * CONV_MACS
OPS_STEP = OPS_LINEAR + OPS_GEMV + OPS_CONV
CONV_OUTPUTS = CD["N"] * CD["OC"] * CHo * CWo
BYTES_CHAIN_PREP = LM * LK * (4 + 1 + 2)
# algorithmic bytes (each input read once, each output written once)
BYTES_QUANT = QN * (4 + 1)
BYTES_GEMV = GN * GK + GK + GN + 2 * GN * 4


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs", 6786.9), d.get("bf16_tflops", 1887.4), "measured"
    return 6800.0, 1900.0, "fallback"


# ---------------------------------------------------------------------------
# clocks sampler (nvidia-smi during the timed region)
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# inputs
# ---------------------------------------------------------------------------
def host_inputs():
    qp, lp, gp, cp = Q.params, L.params, G.params, C.params
    xq = synth.normal(Q.seed, "x", (QN,), qp["x_mean"], qp["x_var"])
    lx, lw, lws, lb = synth.linear_inputs(L.seed, LM, LK, LN, x_kind="fp32", p=lp)
    gx, gw, gws, gb = synth.linear_inputs(G.seed, 1, GK, GN, x_kind="int8", p=gp)
    cx, cw, cws, cb = synth.conv_t_inputs(C.seed, CD, cp)
    return dict(xq=xq, lx=lx, lw=lw, lws=lws, lb=lb, gx=gx, gw=gw, gws=gws, gb=gb, cx=cx, cw=cw,
                cws=cws, cb=cb)


# ---------------------------------------------------------------------------
# our CUDA path
# ---------------------------------------------------------------------------
class Path:
    """Device-resident buffers and one step of the hot path."""

    def __init__(self, h, dev, only="all"):
        import torch
        import int8_quantized_q8ta_gb300 as q8
        self.q8, self.torch, self.dev, self.only = q8, torch, dev, only
        T = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
        self.xq = T(h["xq"])
        self.q_out = torch.empty(QN, dtype=torch.int8, device=dev)
        self.lx = T(h["lx"])
        self.packed = q8.pack_weight(T(h["lw"]))
        self.lws, self.lb = T(h["lws"]), T(h["lb"])
        self.l_xq = torch.empty((LM, LK), dtype=torch.int8, device=dev)
        self.operand = q8.operand_buffer(LM, LK, dev)
        self.l_out = torch.empty((LM, LN), dtype=torch.int8, device=dev)
        self.gx, self.gw = T(h["gx"]), T(h["gw"])
        # the gemv weight is packed once too (a copy the library never sees
        # written again, so each call reads it before the previous kernel ends)
        self.g_packed = q8.pack_gemv_weight(self.gw)
        self.gws, self.gb = T(h["gws"]), T(h["gb"])
        self.g_out = torch.empty((1, GN), dtype=torch.int8, device=dev)
        self.cx, self.cw = T(h["cx"]), T(h["cw"])
        self.cws, self.cb = T(h["cws"]), T(h["cb"])
        self.c_out = torch.empty((CD["N"], CD["OC"], CHo, CWo), dtype=torch.int8, device=dev)
        # the conv_t weight is packed once, like the linear weight (load time)
        self.c_packed = q8.pack_conv2d_transposed_weight(self.cw, CD["IC"], (CD["Kh"], CD["Kw"]))
        shape = q8.conv_t_shape(tuple(self.cx.shape), tuple(self.cw.shape), CD["Kh"], CD["Kw"],
                                CHo, CWo, CD["s"], CD["p"], CD["op"])
        import ctypes
        self.c_ws = torch.empty(
            q8.lib().q8_conv2d_transposed_packed_workspace_bytes(ctypes.byref(shape)),
            dtype=torch.uint8, device=dev)
        torch.cuda.synchronize()

    LAUNCHES = {"quantize": 1, "linear": 2, "gemv": 1, "conv_t": 2}

    def launches_per_step(self):
        if self.only == "all":
            return sum(self.LAUNCHES.values())
        return self.LAUNCHES[self.only]

    # the four ops of a step, their activation inputs and outputs (attribute names)
    OPS = ("quantize", "linear", "gemv", "conv_t")
    INPUTS = {"quantize": "xq", "linear": "lx", "gemv": "gx", "conv_t": "cx"}
    OUTPUTS = {"quantize": "q_out", "linear": "l_out", "gemv": "g_out", "conv_t": "c_out"}

    def run_op(self, name, mid=None):
        """Enqueue one op on the current stream (the linear op is the
        quantize -> operand kernel and the GEMM; mid() runs between them)."""
        q8, qp, lp, gp, cp = self.q8, Q.params, L.params, G.params, C.params
        if name == "quantize":
            q8.quantize_per_tensor(self.xq, qp["in_scale"], qp["in_zp"], out=self.q_out)
        elif name == "linear":
            q8.quantize_to_operand(self.lx, lp["in_scale"], lp["in_zp"], x_q=self.l_xq,
                                   operand=self.operand)
            if mid:
                mid()
            q8.linear_operand_packed(self.operand, lp["in_scale"], self.packed, self.lws, self.lb,
                                     lp["out_scale"], lp["out_zp"], out=self.l_out)
        elif name == "gemv":
            q8.linear_gemv_packed(self.gx, gp["in_scale"], gp["in_zp"], self.g_packed, self.gws,
                                  self.gb, gp["out_scale"], gp["out_zp"], out=self.g_out)
        else:
            q8.conv2d_transposed_packed(self.cx, cp["in_scale"], cp["in_zp"], self.c_packed,
                                        self.cws, self.cb, cp["out_scale"], cp["out_zp"],
                                        stride=CD["s"], padding=CD["p"],
                                        output_padding=CD["op"], out=self.c_out,
                                        workspace=self.c_ws)

    # per-op timing slots: events 0..5 bracket quantize, the linear's operand
    # preparation, the linear GEMM, the gemv and the transposed convolution
    TIMED = ("quantize", "chain_prep", "linear", "gemv", "conv_t")

    def step(self, ev=None):
        """Enqueue one step; ev (a list of 6 CUDA events) brackets each op."""
        rec = (lambda i: ev[i].record()) if ev else (lambda i: None)
        slot = {"quantize": 0, "linear": 1, "gemv": 3, "conv_t": 4}
        for op in self.OPS:
            rec(slot[op])
            if self.only in ("all", op):
                self.run_op(op, mid=(lambda: rec(2)) if op == "linear" else None)
            elif op == "linear":
                rec(2)
        rec(5)


GEMV_CHAIN_COPIES = 24   # 24 x 16.8 MB of weights: 403 MB, more than 3x the 129 MB L2
GEMV_CHAIN_PASSES = 4    # the graph runs the 24 calls 4 times: 96 gemvs in a row
GEMV_CHAIN_REPS = 5      # graph replays per timed group
GEMV_CHAIN_GROUPS = 5    # timed groups; the median group is reported


def gemv_chain_measure(path, copies=GEMV_CHAIN_COPIES, reps=GEMV_CHAIN_REPS, packed=True,
                       passes=GEMV_CHAIN_PASSES, groups=GEMV_CHAIN_GROUPS):
    """q8ta_linear_gemv as a decode step runs it: gemvs back to back, each
    on its own weight (like successive layers), no event or host work
    between them.  `passes` rounds over `copies` weights (passes x copies
    calls, a decode step's worth) are captured once in a CUDA graph (so the
    host's per-call cost is not what is timed); a timed group is `reps`
    replays, and the median of `groups` groups is reported.  The weights
    total more than 2x L2, so every call streams its weight from HBM.
    Returns (microseconds per call, whether a graph was used); checks that
    every call's output equals the lone call's (same x, same weight
    values)."""
    torch, q8 = path.torch, path.q8
    gp = G.params
    if packed:
        weights = [q8.pack_gemv_weight(path.gw) for _ in range(copies)]
    else:
        weights = [path.gw.clone() for _ in range(copies)]
    outs = [torch.empty((1, GN), dtype=torch.int8, device=path.dev) for _ in range(copies)]

    def chain():
        for i in range(copies):
            if packed:
                q8.linear_gemv_packed(path.gx, gp["in_scale"], gp["in_zp"], weights[i], path.gws,
                                      path.gb, gp["out_scale"], gp["out_zp"], out=outs[i])
            else:
                q8.linear_gemv(path.gx, gp["in_scale"], gp["in_zp"], weights[i], None, path.gws,
                               path.gb, gp["out_scale"], gp["out_zp"], out=outs[i])

    for _ in range(2):
        chain()
    torch.cuda.synchronize()
    graph = None
    try:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            for _ in range(passes):
                chain()
        graph = g
    except RuntimeError:
        torch.cuda.synchronize()
        graph = None
    if graph is not None:
        run = graph.replay
    else:
        def run():
            for _ in range(passes):
                chain()
    for _ in range(3):
        run()
    torch.cuda.synchronize()
    per_group = []
    for _ in range(groups):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            run()
        e1.record()
        torch.cuda.synchronize()
        per_group.append(e0.elapsed_time(e1) * 1e3 / (reps * passes * copies))
    us = float(np.median(per_group))
    for o in outs:
        if not torch.equal(o, path.g_out):
            raise RuntimeError("gemv chain: a chained call's output differs from the lone call's")
    used_graph = graph is not None
    del weights, outs, graph
    return us, used_graph


def unpacked_forms_measure(path, h, reps=10, warm=2):
    """The schema entry points with raw int8 weights, no load-time packing:
    q8_linear on the prefill linear (x_q from the step) and
    q8_conv2d_transposed on the 8x256x64x64 convolution.  Each call turns
    its weight into the tensor-core operand again (and computes no weight
    bound, so its exact chunks are the int8 worst case).  Median of `reps`
    calls after `warm`, each bracketed by CUDA events; each output must
    equal the packed path's."""
    torch, q8 = path.torch, path.q8
    lp, cp = L.params, C.params
    lw = torch.from_numpy(np.ascontiguousarray(h["lw"])).to(path.dev)
    lout = torch.empty_like(path.l_out)
    lwork = torch.empty(q8.lib().q8_linear_workspace_bytes(LM, LK, LN), dtype=torch.uint8,
                        device=path.dev)
    cout = torch.empty_like(path.c_out)

    def lin():
        q8.linear(path.l_xq, lp["in_scale"], lp["in_zp"], lw, None, path.lws, path.lb,
                  lp["out_scale"], lp["out_zp"], out=lout, workspace=lwork)

    def conv():
        q8.conv2d_transposed(path.cx, cp["in_scale"], cp["in_zp"], path.cw, None, path.cws,
                             path.cb, cp["out_scale"], cp["out_zp"], (CD["Kh"], CD["Kw"]),
                             stride=CD["s"], padding=CD["p"], output_padding=CD["op"],
                             out=cout)

    res = {}
    for name, fn in (("linear", lin), ("conv_t", conv)):
        for _ in range(warm):
            fn()
        torch.cuda.synchronize()
        times = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1) * 1e3)
        res[name] = float(np.median(times))
    path.run_op("linear")
    path.run_op("conv_t")
    torch.cuda.synchronize()
    if not torch.equal(lout, path.l_out):
        raise RuntimeError("q8_linear with a raw weight differs from the packed path")
    if not torch.equal(cout, path.c_out):
        raise RuntimeError("q8_conv2d_transposed with a raw weight differs from the packed path")
    del lw, lout, lwork, cout
    return res


def small_op_latency(fn, reps=60, warm=10):
    """Median microseconds of fn() over `reps` calls, each bracketed by CUDA
    events on the launching stream (launch gaps included), after `warm`."""
    import torch
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps)]
    for a, b in evs:
        a.record()
        fn()
        b.record()
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) * 1e3 for a, b in evs)


def fused_chain_ab(path, reps=10):
    """The prefill chain both ways, interleaved, each call bracketed by CUDA
    events: two kernels (quantize -> operand, then the GEMM) and the single
    fused kernel (q8_quantize_linear_fused).  Returns median microseconds."""
    torch, q8 = path.torch, path.q8
    lp = L.params
    def two():
        path.run_op("linear")
    def one():
        q8.quantize_linear_fused(path.lx, lp["in_scale"], lp["in_zp"], path.packed, path.lws,
                                 path.lb, lp["out_scale"], lp["out_zp"], x_q=path.l_xq,
                                 out=path.l_out, operand=path.operand)
    res = {"two_kernels": [], "one_kernel": []}
    for it in range(reps + 2):
        for name, fn in (("two_kernels", two), ("one_kernel", one)):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            if it >= 2:
                res[name].append(e0.elapsed_time(e1) * 1e3)
    return {k: statistics.median(v) for k, v in res.items()}


def graph_per_call_us(fn, calls=32, reps=20):
    """Device microseconds per call of fn() with the host out of the way:
    `calls` calls captured in one CUDA graph, replayed `reps` times."""
    import torch
    fn()
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    try:
        with torch.cuda.graph(g, stream=side):
            for _ in range(calls):
                fn()
    except RuntimeError:
        torch.cuda.synchronize()
        return None
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / (calls * reps)


def small_configs_measure(dev):
    """The two latency-bound workloads: quantize -> q8ta_linear 8x64x32 and
    the 1x64x32x32 -> 1x32x64x64 transposed convolution (packed weights,
    buffers allocated once).  Returns their ops entries."""
    import torch
    import int8_quantized_q8ta_gb300 as q8
    T = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    w0 = synth.CONFIGS["linear_chain_8x64x32"]
    d0, p0 = w0.dims, w0.params
    x, w, ws, b = synth.linear_inputs(w0.seed, d0["M"], d0["K"], d0["N"], x_kind="fp32", p=p0)
    x, ws, b = T(x), T(ws), T(b)
    packed = q8.pack_weight(T(w))
    xq = torch.empty((d0["M"], d0["K"]), dtype=torch.int8, device=dev)
    operand = q8.operand_buffer(d0["M"], d0["K"], dev)
    out0 = torch.empty((d0["M"], d0["N"]), dtype=torch.int8, device=dev)

    def cfg0():
        q8.quantize_linear_fused(x, p0["in_scale"], p0["in_zp"], packed, ws, b, p0["out_scale"],
                                 p0["out_zp"], x_q=xq, out=out0, operand=operand)

    w3 = synth.CONFIGS["conv_t_1x64x32x32_k4s2"]
    d3, p3 = w3.dims, w3.params
    cx, cw, cws, cb = synth.conv_t_inputs(w3.seed, d3, p3)
    cx, cws, cb = T(cx), T(cws), T(cb)
    Ho, Wo = synth.output_hw(d3["H_in"], d3["W_in"], d3["Kh"], d3["Kw"], d3["s"], d3["s"],
                             d3["p"], d3["p"], d3["op"], d3["op"])
    cpk = q8.pack_conv2d_transposed_weight(T(cw), d3["IC"], (d3["Kh"], d3["Kw"]))
    shape = q8.conv_t_shape(tuple(cx.shape), tuple(cw.shape), d3["Kh"], d3["Kw"], Ho, Wo,
                            d3["s"], d3["p"], d3["op"])
    import ctypes
    cws_buf = torch.empty(q8.lib().q8_conv2d_transposed_packed_workspace_bytes(
        ctypes.byref(shape)), dtype=torch.uint8, device=dev)
    out3 = torch.empty((d3["N"], d3["OC"], Ho, Wo), dtype=torch.int8, device=dev)

    def cfg3():
        q8.conv2d_transposed_packed(cx, p3["in_scale"], p3["in_zp"], cpk, cws, cb,
                                    p3["out_scale"], p3["out_zp"], stride=d3["s"],
                                    padding=d3["p"], output_padding=d3["op"], out=out3,
                                    workspace=cws_buf)

    us0, g0 = small_op_latency(cfg0), graph_per_call_us(cfg0)
    us3, g3 = small_op_latency(cfg3), graph_per_call_us(cfg3)
    macs3 = conv_valid_macs(d3, Ho, Wo)
    how = ("us: median of 60 calls after 10, each bracketed by CUDA events (host launch cost "
           "and gaps included); us_graph: 32 calls captured in one CUDA graph, replayed 20x, "
           "device time per call")
    return {
        "linear_chain_8x64x32": {
            "us": us0, "us_graph": g0, "launches": 1,
            "TOPS": 2 * d0["M"] * d0["N"] * d0["K"] / us0 / 1e6,
            "method": "fused quantize -> q8ta_linear kernel; " + how},
        "q8ta_conv2d_transposed_1x64x32x32": {
            "us": us3, "us_graph": g3, "launches": 2,
            "outputs/s": d3["N"] * d3["OC"] * Ho * Wo / us3 * 1e6,
            "outputs/s_graph": d3["N"] * d3["OC"] * Ho * Wo / g3 * 1e6 if g3 else None,
            "TOPS_valid_taps": 2 * macs3 / us3 / 1e6,
            "method": "input relayout + GEMM, packed weight; " + how},
    }


def e2e_measure(paths, h, steps):
    """The step through the public API with host buffers: every activation is
    copied in from pinned host memory and every output copied back to pinned
    host memory, all inside the timed region.  As a user would, the copies
    run on their own streams and overlap the kernels: op k's inputs go in
    while op k-1 computes, and its output comes back while op k+1 computes.
    Two sets of device buffers (``paths``) alternate between steps, so a
    step's copies never wait for the previous step's kernels on the same
    buffers; events order every reuse."""
    torch = paths[0].torch
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()  # noqa: E731
    OPS, INP, OUT = Path.OPS, Path.INPUTS, Path.OUTPUTS
    hx = {op: pin(h[INP[op]]) for op in OPS}
    houts = {op: torch.empty(getattr(paths[0], OUT[op]).shape,
                             dtype=getattr(paths[0], OUT[op]).dtype).pin_memory() for op in OPS}
    h2d = sum(t.numel() * t.element_size() for t in hx.values())
    d2h = sum(t.numel() * t.element_size() for t in houts.values())
    s_in, s_run, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    consumed = {}   # (set, op) -> event: the op's kernels have read that set's inputs
    drained = {}    # (set, op) -> event: that set's output has been copied out

    def one(t):
        b = t % len(paths)
        P = paths[b]
        for op in OPS:
            with torch.cuda.stream(s_in):
                if (b, op) in consumed:
                    s_in.wait_event(consumed[(b, op)])
                getattr(P, INP[op]).copy_(hx[op], non_blocking=True)
                ready = torch.cuda.Event()
                ready.record(s_in)
            with torch.cuda.stream(s_run):
                s_run.wait_event(ready)
                if (b, op) in drained:
                    s_run.wait_event(drained[(b, op)])
                P.run_op(op)
                done = torch.cuda.Event()
                done.record(s_run)
                consumed[(b, op)] = done
            with torch.cuda.stream(s_out):
                s_out.wait_event(done)
                houts[op].copy_(getattr(P, OUT[op]), non_blocking=True)
                out = torch.cuda.Event()
                out.record(s_out)
                drained[(b, op)] = out

    for t in range(2):
        one(t)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(s_in)
    s_run.wait_stream(s_in)
    s_out.wait_stream(s_in)
    for t in range(steps):
        one(t)
    s_in.wait_stream(s_run)
    s_in.wait_stream(s_out)
    end.record(s_in)
    torch.cuda.synchronize()
    ms = start.elapsed_time(end) / steps
    return ms, h2d, d2h


# ---------------------------------------------------------------------------
# CPU oracle baseline: the whole step scaled down by the same factor in every op
# ---------------------------------------------------------------------------
ORACLE_SCALE = 64   # the oracle's step is 1/64 of the full step's work in every op


def oracle_scaled_step(h, threads=None, scale=ORACLE_SCALE):
    """Run the oracle, as it stands, on 1/scale of every op of the step and
    time it: quantize numel/scale elements; the chain's quantize and linear
    on M/scale rows; the gemv on N/scale weight rows; the transposed
    convolution on (images x output channels)/scale whole output planes.
    The work is exactly OPS_STEP/scale int8 MACs x 2, so the rate needs no
    extrapolation.  Returns (seconds, threads used, description, per-op
    seconds)."""
    import oracle
    oracle.build()
    threads = threads or (os.cpu_count() or 1)
    qp, lp, gp, cp = Q.params, L.params, G.params, C.params
    q_n = QN // scale
    l_rows = LM // scale
    g_rows = GN // scale
    planes = CD["N"] * CD["OC"] // scale
    Ho, Wo = CHo, CWo

    def chunks(n, parts):
        step = (n + parts - 1) // parts
        return [(a, min(n, a + step)) for a in range(0, n, step)]

    def run_quant(ab):
        oracle.quantize_per_tensor(h["xq"][ab[0]:ab[1]], qp["in_scale"], qp["in_zp"])

    def run_chain(r):
        xq = oracle.quantize_per_tensor(h["lx"][r:r + 1], lp["in_scale"], lp["in_zp"])
        oracle.linear(xq, lp["in_scale"], lp["in_zp"], h["lw"], h["lws"], h["lb"],
                      lp["out_scale"], lp["out_zp"])

    def run_gemv(ab):
        a, b = ab
        oracle.linear(h["gx"], gp["in_scale"], gp["in_zp"], h["gw"][a:b], h["gws"][a:b],
                      h["gb"][a:b], gp["out_scale"], gp["out_zp"])

    def run_conv(i):
        n, oc = divmod(i, CD["OC"])
        oracle.conv2d_transposed(h["cx"][n:n + 1], cp["in_scale"], cp["in_zp"],
                                 h["cw"][oc:oc + 1], CD["Kh"], CD["Kw"], h["cws"][oc:oc + 1],
                                 h["cb"][oc:oc + 1], cp["out_scale"], cp["out_zp"], Ho, Wo,
                                 (CD["s"], CD["s"]), (CD["p"], CD["p"]))

    parts = {}
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:   # ctypes releases the GIL
        def timed(name, fn, items):
            t0 = time.perf_counter()
            list(ex.map(fn, items))
            parts[name] = time.perf_counter() - t0
        timed("quantize", run_quant, chunks(q_n, threads))
        timed("chain_quantize_linear", run_chain, range(l_rows))
        timed("gemv", run_gemv, chunks(g_rows, min(threads, max(1, g_rows // 8))))
        # output planes spread over the images, as the full op's are
        timed("conv_t", run_conv, [(k * CD["N"] * CD["OC"]) // planes for k in range(planes)])
    total = sum(parts.values())
    sample = (f"1/{scale} of every op of the step, timed whole: quantize {q_n} of {QN} "
              f"elements; quantize->linear {l_rows} of {LM} rows; gemv {g_rows} of {GN} weight "
              f"rows; conv_t {planes} of {CD['N'] * CD['OC']} (image, channel) output planes; "
              f"{threads} thread(s), one oracle call per row block or plane")
    return total, threads, sample, parts


def traffic_from_profile(key):
    """DRAM read+write bytes per launch of a GEMM from the committed ncu
    summary (profiles/traffic.json), valid only while the kernel's source
    files are unchanged since the capture; otherwise None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        e = json.load(f).get(key)
    if not e:
        return None
    digest = hashlib.sha256()
    for rel in e.get("source_files", []):
        with open(os.path.join(ROOT, rel), "rb") as f:
            digest.update(f.read())
    if digest.hexdigest()[:16] != e.get("source_sha256_16"):
        return None
    return e.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------
def max_over_ranks(value, device):
    """The slowest rank's figure (every rank calls this; the job's step time
    is its slowest rank's)."""
    import torch
    import torch.distributed as tdist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world, ms_step):
    """Whole-job int8 TOPS: every rank runs one full step (weak scaling)."""
    return world * OPS_STEP / (ms_step * 1e-3) / 1e12


def run_ours(args, rank, world, local_rank):
    import torch
    dev = torch.device(f"cuda:{local_rank}")
    torch.cuda.set_device(dev)
    h = host_inputs()
    path = Path(h, dev, args.only)
    dist = world > 1
    if dist:
        import torch.distributed as tdist

    for _ in range(args.warmup):
        path.step()
    torch.cuda.synchronize()
    if dist:
        tdist.barrier()

    K = args.steps
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    t_start.record()
    for k in range(K):
        path.step()
    t_end.record()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    # Per-op times come from a second pass with an event between ops (an
    # event on the stream also stops one kernel from starting under the
    # previous one's tail, so these times include each op's own ramp).
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(K)]
    for k in range(K):
        path.step(evs[k])
    torch.cuda.synchronize()
    if dist:
        tdist.barrier()
    ms_total = t_start.elapsed_time(t_end)
    ms_step = ms_total / K
    if dist:
        ms_step = max_over_ranks(ms_step, dev)

    extra_ops = {}
    chained = args.only in ("all", "gemv") and not args.no_extra_ops
    if chained:
        chain_us, chain_graph = gemv_chain_measure(path)
        plain_us, _ = gemv_chain_measure(path, packed=False)
    if args.only == "all" and not args.no_extra_ops:
        extra_ops = small_configs_measure(dev)
        ab = fused_chain_ab(path)
        unp = unpacked_forms_measure(path, h)
        extra_ops["q8ta_linear_2048x4096x11008_raw_weight"] = {
            "us": unp["linear"], "TOPS": OPS_LINEAR / unp["linear"] / 1e6,
            "method": "q8_linear (the pages' schema) with the raw int8 weight: each call converts "
                      "x_q and the 45 MB weight to the bf16 operands, then the GEMM; median of 10 "
                      "event-bracketed calls; output equal to the packed path's"}
        extra_ops["q8ta_conv2d_transposed_8x256x64x64_raw_weight"] = {
            "us": unp["conv_t"], "outputs/s": CONV_OUTPUTS / unp["conv_t"] * 1e6,
            "method": "q8_conv2d_transposed (the pages' schema) with the raw int8 weight: each call "
                      "converts the weight (no k-block bound: worst-case exact chunks), relayouts x, "
                      "then the GEMM; "
                      "median of 10 event-bracketed calls; output equal to the packed path's"}
        extra_ops["quantize_q8ta_linear_2048x4096x11008_two_vs_one_kernel"] = {
            "us_two_kernels": ab["two_kernels"], "us_one_kernel": ab["one_kernel"],
            "method": "the prefill chain alone, each call bracketed by CUDA events, median of 10 "
                      "interleaved calls: quantize->operand + GEMM (the step's form) against "
                      "the single kernel whose warps quantize x into the operand"}

    names = list(Path.TIMED)
    per = {n: statistics.mean(evs[k][i].elapsed_time(evs[k][i + 1]) for k in range(K))
           for i, n in enumerate(names)}
    hbm, bf16, peak_src = measured_peaks()
    us = {n: per[n] * 1e3 for n in names}

    ops = {
        "quantize_64Mi": {"us": us["quantize"], "GB/s": BYTES_QUANT / us["quantize"] / 1e3,
                          "frac_hbm": BYTES_QUANT / us["quantize"] / 1e3 / hbm},
        "chain_quantize_to_operand_2048x4096": {
            "us": us["chain_prep"], "GB/s": BYTES_CHAIN_PREP / us["chain_prep"] / 1e3,
            "frac_hbm": BYTES_CHAIN_PREP / us["chain_prep"] / 1e3 / hbm},
        "q8ta_linear_2048x4096x11008": {
            "us": us["linear"], "TOPS": OPS_LINEAR / us["linear"] / 1e6,
            "frac_bf16_peak": OPS_LINEAR / us["linear"] / 1e6 / bf16},
        "q8ta_linear_gemv_1x4096x4096": {
            "us": us["gemv"], "GB/s": BYTES_GEMV / us["gemv"] / 1e3,
            "frac_hbm": BYTES_GEMV / us["gemv"] / 1e3 / hbm,
            "note": "q8_linear_gemv_packed, one launch bracketed by events inside the step pass (its launch and "
                    "DRAM ramp are not overlapped)"},
        "q8ta_conv2d_transposed_8x256x64x64": {
            "us": us["conv_t"], "outputs/s": CONV_OUTPUTS / us["conv_t"] * 1e6,
            "TOPS_valid_taps": OPS_CONV / us["conv_t"] / 1e6},
    }
    if chained:
        ops["q8ta_linear_gemv_1x4096x4096_chained"] = {
            "us_per_call": chain_us, "GB/s": BYTES_GEMV / chain_us / 1e3,
            "frac_hbm": BYTES_GEMV / chain_us / 1e3 / hbm,
            "us_per_call_unpacked_weight": plain_us,
            "method": f"{GEMV_CHAIN_PASSES * GEMV_CHAIN_COPIES} calls back to back, "
                      f"{GEMV_CHAIN_PASSES} passes over {GEMV_CHAIN_COPIES} distinct packed weight "
                      f"copies ({GEMV_CHAIN_COPIES * GN * GK / 1e6:.0f} MB, > 2x L2, so every "
                      f"call streams its weight from HBM), "
                      f"{'one CUDA graph' if chain_graph else 'eager launches'}; median of "
                      f"{GEMV_CHAIN_GROUPS} groups of {GEMV_CHAIN_REPS} replays, events only "
                      f"around each group"}
    ops.update(extra_ops)
    achieved = OPS_LINEAR / us["linear"] / 1e6
    roofline = {"kernel": "tc_gemm_kernel<240,12,0,2,2> (q8ta_linear 2048x4096x11008)",
                "bound": "tensor",
                "achieved": achieved, "peak": bf16,
                "peak_source": f"{peak_src} bf16 dense burst (MEASURED_PEAKS.json)",
                "unit": "TFLOP/s", "frac": achieved / bf16,
                "traffic": traffic_from_profile("tc_gemm_linear_2048x4096x11008"),
                "algorithmic_flops_per_launch": OPS_LINEAR}

    result = {
        "metric": METRIC, "value": job_throughput(world, ms_step),
        "unit": "int8 TOPS (2 x int8 MACs of linear + gemv + conv_t valid taps, per step)",
        "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int8", "data": "synthetic",
        "config": {"workload": "q8ta hot path: quantize_per_tensor 64Mi; quantize->q8ta_linear "
                               "2048x4096x11008; q8ta_linear_gemv 1x4096x4096; "
                               "q8ta_conv2d_transposed 8x256x64x64 k3 s2 p1 op1",
                   "inputs": "seeded synthetic, distributions of the five workloads",
                   "l2": "each step streams > 0.5 GB (L2 is 129 MB), so no input is L2-resident "
                         "from the previous step",
                   "weights": "linear and conv_t weights packed to bf16 once, outside the "
                              "timed region (load time, as the pages' ahead-of-time weight "
                              "reshape); the gemv weight copied once into a packed (never rewritten) "
                              "int8 buffer, also outside the timed region",
                   "parallelism": f"replicas x{world}"},
        "ops": ops, "roofline": roofline, "clocks": clocks,
        "gpu_launches": path.launches_per_step() * K,
    }
    if args.only != "all":
        result["config"]["only"] = args.only
    if rank == 0 and not args.no_e2e and args.only == "all":
        # as many steps as the timed loop (at most 50): the pipeline's fill and
        # drain are a smaller share of more steps
        e2e_ms, h2d, d2h = e2e_measure([path, Path(h, dev, "all")], h, max(3, min(K, 50)))
        result["e2e"] = {"value": world * OPS_STEP / (e2e_ms * 1e-3) / 1e12,
                         "unit": result["unit"], "ms_per_step": e2e_ms,
                         "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                         "note": "activations copied in from pinned host memory and every output "
                                 "copied back each step, on copy streams overlapping the "
                                 "kernels (two alternating device buffer sets); weights "
                                 "resident"}
    if rank == 0 and not args.no_cpu_baseline and args.only == "all":
        t_cpu, cores, sample, parts = oracle_scaled_step(h)
        t_one, _, _, parts_one = oracle_scaled_step(h, threads=1)
        result["cpu_baseline"] = {"value": OPS_STEP / ORACLE_SCALE / t_cpu / 1e12,
                                  "unit": result["unit"], "cores": cores, "kind": "oracle",
                                  "sample": sample, "seconds_per_sample": t_cpu,
                                  "seconds_by_op": parts,
                                  "single_thread": {
                                      "value": OPS_STEP / ORACLE_SCALE / t_one / 1e12,
                                      "cores": 1, "seconds_per_sample": t_one,
                                      "seconds_by_op": parts_one}}
    return result


def run_reference(args):
    """The oracle as it stands, on the host cores; each step is the full step
    scaled down by ORACLE_SCALE in every op (see oracle_scaled_step)."""
    h = host_inputs()
    for _ in range(args.warmup):
        oracle_scaled_step(h)
    ts, last = [], None
    for _ in range(args.steps):
        t, cores, sample, parts = oracle_scaled_step(h)
        ts.append(t)
        last = (cores, sample)
    t = statistics.median(ts)
    v = OPS_STEP / ORACLE_SCALE / t / 1e12
    unit = "int8 TOPS (2 x int8 MACs of linear + gemv + conv_t valid taps, per step)"
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": unit, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8",
            "data": "synthetic",
            "config": {"workload": f"q8ta hot path (the CUDA arm's step) scaled by 1/{ORACLE_SCALE} "
                                   "in every op; CPU oracle on all host cores",
                       "step": "one step = 1/64 of the full step's work, timed whole"},
            "cpu_baseline": {"value": v, "unit": unit, "cores": last[0], "kind": "oracle",
                             "sample": last[1]},
            "e2e": {"value": v, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--only", choices=["all", "quantize", "linear", "gemv", "conv_t"],
                    default="all", help="run one op per step (for profiling)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra-ops", action="store_true",
                    help="skip the chained gemv and the two small workloads (for launch lists)")
    args = ap.parse_args()
    if args.warmup < 3 and args.only == "all":
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(local_rank)
        tdist.init_process_group("nccl")
    res = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as tdist
        tdist.barrier()
        tdist.destroy_process_group()


if __name__ == "__main__":
    main()
