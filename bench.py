#!/usr/bin/env python3
"""Benchmark of the DiT elementwise hot path on GB300.

Metric: achieved HBM GB/s (algorithmic bytes / device time) and its fraction
of the measured GB300 copy bandwidth, with microseconds per call per kernel.

Default workload ("hotpath"): one step is one pass of every operation of the
path over the largest broadcast shape, [B, L, D] = [1, 32640, 4096] bf16
(about 267 MB per tensor; shape from sglang PR #29361, B200 kernel benchmark
table, ltx2_bcast_s32640_c4096):

  rga_bcast          out = hidden + update * gate[1,1,D]
  rga_bcast_inplace  hidden += update * gate[1,1,D]
  rga_full           out = hidden + update * gate[1,L,D]
  mod_bcast          out = rms_norm(x, 1e-6) * (1 + scale[1,1,D]) + shift[1,1,D]
  fused_bcast        residual, modulated = both in one pass

Every op reads its own input tensors, each larger than the 129 MB L2, so no
op or step re-reads another's data from L2.  Other workloads: "chain" (the
8-block DiT chain at B=2, 25 launches per step) and "shapes" (one line per
workload shape and op, for the per-shape table).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun every rank runs the same workload on its own GPU (the rows of
these ops are independent: no data-path collective); value = bytes of all
ranks / max over ranks of the timed region.  --impl reference times the CPU
oracle (the reference arm of this repository) on a bounded sample.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "achieved HBM GB/s and % of GB300 peak per shape; µs/call (device-timed)"
FALLBACK_HBM_GBS = 6800.0
EPS = 1e-6


# ---------------------------------------------------------------------------
# environment
# ---------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, period_ms: int = 50):
        self.index = index
        self.period_ms = period_ms
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", f"-lms={self.period_ms}"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread:
                self.thread.join(timeout=5)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def _code_only(text):
    """C/C++/CUDA source without its comments, trailing blanks and blank
    lines (string and character literals kept as they are)."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    lines = (line.rstrip() for line in "".join(out).split("\n"))
    return "\n".join(line for line in lines if line)


def kernel_source_hash():
    """Hash of the CUDA sources' code (ties a stored ncu traffic figure to
    them; an edit of comments only keeps it)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "diffusion_transformer_elementwise_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode())
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def stored_traffic(kernel_key):
    """DRAM bytes per launch from profiles/traffic.json, if taken on the
    current sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            data = json.load(f)
    except (OSError, ValueError):
        return None
    entry = data.get(kernel_key)
    if not entry or entry.get("source_sha") != kernel_source_hash():
        return None
    return entry.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------

# ops that launch the same kernel as another op (for the roofline's dominant kernel)
KERNEL_OF = {"rga_bcast_inplace": "rga_bcast"}


class Op:
    def __init__(self, name, fn, nbytes, inputs, outputs, sample, launches=1, touches=()):
        self.launches = launches  # kernels one call of fn launches
        self.touches = list(touches)  # device tensors fn reads or writes besides inputs/outputs
        self.name = name
        self.fn = fn            # enqueue the op on the current stream
        self.bytes = nbytes     # algorithmic bytes per call
        self.inputs = inputs    # device tensors copied in for the e2e number
        self.outputs = outputs  # device tensors copied out for the e2e number
        self.sample = sample    # callable(rows) -> oracle callable for the CPU baseline


def hotpath_ops(device, B=1, L=32640, D=4096, dtype="bf16", only=None):
    """The five ops of the hot-path step, each with its own input tensors.
    only: build just the op of that name."""
    import torch

    import diffusion_transformer_elementwise_gb300 as dit
    from diffusion_transformer_elementwise_gb300.synth import draw, seed_for

    es = 2 if dtype != "fp32" else 4
    N = B * L * D
    vb = B * D * es

    def act(name):
        return draw("act", (B, L, D), seed_for("bench", name), dtype, device)

    def vec(kind, name):
        return draw(kind, (B, 1, D), seed_for("bench", name), dtype, device)

    def sampler(kind, tensors, layout=None):
        def make(rows):
            import oracle
            host = [t[:, :rows].contiguous().cpu() if t.shape[1] == L else t.cpu()
                    for t in tensors]
            outs = [torch.empty((B, rows, D), dtype=host[0].dtype) for _ in range(2)]

            def run(threads):
                if kind == "rga":
                    oracle.residual_gate_add(outs[0], host[0], host[1], host[2], B, rows, D,
                                             dtype, layout, threads=threads)
                elif kind == "mod":
                    oracle.rmsnorm_modulate(outs[0], host[0], host[1], host[2], B, rows, D,
                                            EPS, dtype, "bcast", threads=threads)
                else:
                    oracle.gate_add_rmsnorm_modulate(outs[0], outs[1], *host, B, rows, D, EPS,
                                                     dtype, "bcast", "bcast", threads=threads)
            return run
        return make

    def rga_bcast():
        h, u, g, o = act("h1"), act("u1"), vec("gate", "gate_b"), None
        o = torch.empty_like(h)
        return Op("rga_bcast", lambda: dit.residual_gate_add(h, u, g, out=o),
                  3 * N * es + vb, [h, u, g], [o], sampler("rga", [h, u, g], "bcast"))

    def rga_bcast_inplace():
        h, u, g = act("h2"), act("u2"), vec("gate", "gate_b")
        return Op("rga_bcast_inplace", lambda: dit.residual_gate_add(h, u, g, out=h),
                  3 * N * es + vb, [h, u, g], [h], sampler("rga", [h, u, g], "bcast"))

    def rga_full():
        h, u = act("h3"), act("u3")
        g = draw("gate", (B, L, D), seed_for("bench", "gate_f"), dtype, device)
        o = torch.empty_like(h)
        return Op("rga_full", lambda: dit.residual_gate_add(h, u, g, out=o),
                  4 * N * es, [h, u, g], [o], sampler("rga", [h, u, g], "full"))

    def mod_bcast():
        x, sc, sh = act("x4"), vec("mod", "scale"), vec("mod", "shift")
        o = torch.empty_like(x)
        return Op("mod_bcast", lambda: dit.rmsnorm_modulate(x, sc, sh, EPS, out=o),
                  2 * N * es + 2 * vb, [x, sc, sh], [o], sampler("mod", [x, sc, sh]))

    def fused_bcast():
        h, u = act("h5"), act("u5")
        g, sc, sh = vec("gate", "gate_b"), vec("mod", "scale"), vec("mod", "shift")
        r, m = torch.empty_like(h), torch.empty_like(h)
        return Op("fused_bcast",
                  lambda: dit.gate_add_rmsnorm_modulate(h, u, g, sc, sh, EPS, residual_out=r,
                                                        modulated_out=m),
                  4 * N * es + 3 * vb, [h, u, g, sc, sh], [r, m],
                  sampler("fused", [h, u, g, sc, sh]))

    def gelu_ffn():
        # the feed-forward activation: [B, L, 4D]
        x = draw("act", (B, L, 4 * D), seed_for("bench", "ffn"), dtype, device)
        o = torch.empty_like(x)
        n4 = 4 * N

        def make(rows):
            import oracle
            host = x[:, :rows].contiguous().cpu()
            res = torch.empty_like(host)
            return lambda threads: oracle.gelu_tanh(res, host, dtype)
        return Op("gelu_ffn", lambda: dit.gelu_tanh(x, out=o), 2 * n4 * es, [x], [o], make)

    def mod_fp8():
        # the modulation with its output in E4M3 (the input of an FP8 GEMM)
        x = draw("act", (B, L, D), seed_for("bench", "x8"), dtype, device)
        sc = draw("mod", (B, 1, D), seed_for("bench", "sc8"), dtype, device)
        sh = draw("mod", (B, 1, D), seed_for("bench", "sh8"), dtype, device)
        qs = torch.full((1,), 0.05, dtype=torch.float32, device=device)
        o = torch.empty((B, L, D), dtype=torch.uint8, device=device)
        return Op("mod_fp8", lambda: dit.rmsnorm_modulate_fp8(x, sc, sh, qs, EPS, out=o),
                  N * es + N + 2 * vb, [x], [o], None)

    def fused_fp8():
        h = draw("act", (B, L, D), seed_for("bench", "h8"), dtype, device)
        u = draw("act", (B, L, D), seed_for("bench", "u8"), dtype, device)
        g = draw("gate", (B, 1, D), seed_for("bench", "g8"), dtype, device)
        sc = draw("mod", (B, 1, D), seed_for("bench", "sc8f"), dtype, device)
        sh = draw("mod", (B, 1, D), seed_for("bench", "sh8f"), dtype, device)
        qs = torch.full((1,), 0.05, dtype=torch.float32, device=device)
        r = torch.empty_like(h)
        o = torch.empty((B, L, D), dtype=torch.uint8, device=device)
        return Op("fused_fp8", lambda: dit.gate_add_rmsnorm_modulate_fp8(
            h, u, g, sc, sh, qs, EPS, residual_out=r, out=o),
            3 * N * es + N + 3 * vb, [h, u], [r, o], None)

    builders = [rga_bcast, rga_bcast_inplace, rga_full, mod_bcast, fused_bcast]
    extra = {"gelu_ffn": gelu_ffn, "mod_fp8": mod_fp8, "fused_fp8": fused_fp8}
    if only in extra:
        return [extra[only]()]
    if only is not None:
        builders = [f for f in builders if f.__name__ == only]
        if not builders:
            raise SystemExit(f"unknown --op {only}")
    return [f() for f in builders]


def chain_ops(device, B=2, L=32640, D=4096, blocks=8, dtype="bf16", graph=False):
    """The chain as one op per launch (so each kernel is timed), or, with
    graph=True, as one op that replays the whole chain captured in a CUDA
    graph (timed as a whole)."""
    import torch

    import diffusion_transformer_elementwise_gb300 as dit
    from diffusion_transformer_elementwise_gb300 import chain

    es = 2 if dtype != "fp32" else 4
    x, updates, tables = chain.make_inputs(B, L, D, blocks, dtype, device, seed_tag="bench")
    m = torch.empty_like(x)
    N, vb = B * L * D, B * D * es
    if graph:
        chain.run(x, updates, tables, EPS, m=m)  # first calls outside the capture
        g, _ = chain.capture(x, updates, tables, EPS, m=m)
        return [Op("chain_graph", g.replay, chain.algorithmic_bytes(B, L, D, blocks, es),
                   [x] + updates, [x, m], None, launches=chain.launches(blocks),
                   touches=[x, m] + updates)]
    sites = chain.site_list(blocks)
    ops = []
    s0 = tables[0][chain.SITES[0]]
    every = [x, m] + updates  # every site reads or writes these
    ops.append(Op("chain_mod", lambda: dit.rmsnorm_modulate(x, s0[1], s0[0], EPS, out=m),
                  2 * N * es + 2 * vb, [x] + updates, [], None, touches=every))
    for j, (blk, k) in enumerate(sites):
        gate = tables[blk][chain.SITES[k]][2]
        u = updates[k]
        if j + 1 < len(sites):
            nb, nk = sites[j + 1]
            shf, scl, _ = tables[nb][chain.SITES[nk]]
            fn = (lambda u=u, gate=gate, scl=scl, shf=shf:
                  dit.gate_add_rmsnorm_modulate(x, u, gate, scl, shf, EPS, residual_out=x,
                                                modulated_out=m))
            ops.append(Op("chain_fused", fn, 4 * N * es + 3 * vb, [], [], None, touches=every))
        else:
            # the step's results: the residual stream and the last modulated input
            ops.append(Op("chain_rga", lambda u=u, gate=gate:
                          dit.residual_gate_add(x, u, gate, out=x), 3 * N * es + vb, [],
                          [x, m], None, touches=every))
    return ops


def chain_av_ops(device, video, audio, blocks=8, dtype="bf16", graph=False, grouped=True):
    """The chain over a video and an audio stream as ONE op per step: the
    grouped launches (1 + 3 * blocks kernels) or one launch per stream and
    site (twice as many), eager or replayed as a CUDA graph."""
    import torch

    from diffusion_transformer_elementwise_gb300 import chain

    es = 2 if dtype != "fp32" else 4
    streams = [chain.make_inputs(*shape, blocks, dtype, device, seed_tag=f"bench-av{i}")
               for i, shape in enumerate((video, audio))]
    ms = [torch.empty_like(x) for x, _, _ in streams]
    nbytes = sum(chain.algorithmic_bytes(*shape, blocks, es) for shape in (video, audio))
    n_launch = chain.launches(blocks) * (1 if grouped else 2)
    chain.run_streams(streams, EPS, ms=ms, grouped=grouped)  # first calls outside any capture
    if graph:
        g, _ = chain.capture_streams(streams, EPS, ms=ms, grouped=grouped)
        fn = g.replay
    else:
        def fn():
            chain.run_streams(streams, EPS, ms=ms, grouped=grouped)
    name = "chain_av_" + ("grouped" if grouped else "separate") + ("_graph" if graph else "")
    ins = [t for x, us, _ in streams for t in [x] + us]
    outs = [t for x, _, _ in streams for t in [x]] + ms
    return [Op(name, fn, nbytes, ins, outs, None, launches=n_launch)]


# ---------------------------------------------------------------------------
# timing
# ---------------------------------------------------------------------------

def time_steps(ops, steps, warmup, dist=None):
    """Warm up, then time exactly `steps` steps with CUDA events on the
    current stream (one event pair per op, and one around everything)."""
    import torch
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        for op in ops:
            op.fn()
    torch.cuda.synchronize()
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in ops] for _ in range(steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    start.record(stream)
    for s in range(steps):
        for i, op in enumerate(ops):
            ev[s][i][0].record(stream)
            op.fn()
            ev[s][i][1].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    total_ms = start.elapsed_time(end)
    per_op = {}
    for i, op in enumerate(ops):
        t = [ev[s][i][0].elapsed_time(ev[s][i][1]) for s in range(steps)]
        d = per_op.setdefault(op.name, {"ms": [], "bytes": op.bytes, "calls": 0})
        d["ms"].extend(t)
        d["calls"] += steps
    return total_ms, per_op


def time_e2e(ops, steps):
    """The same step through the public API from pinned host buffers: every
    step copies each op's inputs host -> device, runs the op and copies its
    results device -> host, all inside the timed region.  The copies are
    pipelined with the kernels on two more streams -- op i+1's inputs go in
    while op i runs and op i-1's results come out (host->device and
    device->host use separate copy engines) -- with per-tensor events for
    every hazard: a copy into a tensor waits for its last use and its last
    read-out in the previous step; an op waits for its inputs' copies and for
    any read-out of a tensor it touches."""
    import torch
    pin = {}

    def host(t):
        if id(t) not in pin:
            pin[id(t)] = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
        return pin[id(t)]
    for op in ops:
        for t in op.inputs:
            host(t).copy_(t)
    h2d = sum(t.numel() * t.element_size() for op in ops for t in op.inputs)
    d2h = sum(t.numel() * t.element_size() for op in ops for t in op.outputs)
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    last_use, last_out = {}, {}  # id(tensor) -> event of the previous step

    def step():
        for op in ops:
            touched = {id(t): t for t in list(op.touches) + list(op.inputs) + list(op.outputs)}
            if op.inputs:
                for t in op.inputs:
                    for ev in (last_use.get(id(t)), last_out.get(id(t))):
                        if ev is not None:
                            s_in.wait_event(ev)
                with torch.cuda.stream(s_in):
                    for t in op.inputs:
                        t.copy_(host(t), non_blocking=True)
                ev_in = torch.cuda.Event()
                ev_in.record(s_in)
                comp.wait_event(ev_in)
            for k in touched:
                if last_out.get(k) is not None:
                    comp.wait_event(last_out[k])
            op.fn()
            ev_op = torch.cuda.Event()
            ev_op.record(comp)
            for k in touched:
                last_use[k] = ev_op
            if op.outputs:
                s_out.wait_event(ev_op)
                with torch.cuda.stream(s_out):
                    for t in op.outputs:
                        host(t).copy_(t, non_blocking=True)
                ev_out = torch.cuda.Event()
                ev_out.record(s_out)
                for t in op.outputs:
                    last_out[id(t)] = ev_out

    step()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(comp)
    s_in.wait_stream(comp)
    s_out.wait_stream(comp)
    for _ in range(steps):
        step()
    comp.wait_stream(s_in)
    comp.wait_stream(s_out)
    end.record(comp)
    torch.cuda.synchronize()
    return start.elapsed_time(end), h2d, d2h


def cpu_baseline(ops, budget_s=12.0, rows=512):
    """The oracle (as it stands) on the host cores: the same ops on the first
    `rows` rows, repeated for about budget_s seconds, all cores and one core."""
    import torch  # noqa: F401
    cores = os.cpu_count() or 1
    runs = [(op, op.sample(rows)) for op in ops if op.sample is not None]
    frac = rows / 32640

    def rate(threads, seconds):
        done, t0 = 0.0, time.perf_counter()
        while True:
            for op, run in runs:
                run(threads)
                done += op.bytes * frac
            el = time.perf_counter() - t0
            if el >= seconds:
                return done / el / 1e9, el

    multi, el_m = rate(cores, budget_s * 0.75)
    single, el_s = rate(1, budget_s * 0.25)
    return {"value": multi, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "single_thread_value": single,
            "sample": f"the step's {len(runs)} ops on the first {rows} of 32640 rows "
                      f"([1,{rows},4096] bf16), repeated for {el_m:.1f} s on {cores} threads "
                      f"and {el_s:.1f} s on 1 thread; GB/s on the same algorithmic bytes"}


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------

def hotpath_config():
    """The config of the headline workload (both arms print it)."""
    return {"workload": "ltx2_bcast_s32640_c4096 hot path: rga_bcast, rga_bcast_inplace, "
                        "rga_full, mod_bcast, fused_bcast",
            "B": 1, "L": 32640, "D": 4096, "eps": EPS,
            "l2": "no flush: every op reads its own inputs, each 267 MB or more, "
                  "above the 129 MB L2"}


def run_reference(args):
    """The reference arm: the CPU oracle on the host cores, each step a
    bounded sample of the hot-path workload."""
    import torch
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    from diffusion_transformer_elementwise_gb300.synth import draw, seed_for
    B, L, D, es = 1, 32640, 4096, 2
    cores = os.cpu_count() or 1
    total_steps = args.steps + args.warmup
    rows = max(16, min(1024, int(32 * 300 / max(total_steps, 1))))
    h = draw("act", (B, rows, D), seed_for("ref", "h"), "bf16")
    u = draw("act", (B, rows, D), seed_for("ref", "u"), "bf16")
    gb = draw("gate", (B, 1, D), seed_for("ref", "gb"), "bf16")
    gf = draw("gate", (B, rows, D), seed_for("ref", "gf"), "bf16")
    sc = draw("mod", (B, 1, D), seed_for("ref", "sc"), "bf16")
    sh = draw("mod", (B, 1, D), seed_for("ref", "sh"), "bf16")
    o, o2 = torch.empty_like(h), torch.empty_like(h)
    hh = h.clone()  # updated in place every step
    n = B * rows * D
    vb = B * D * es
    step_bytes = 2 * (3 * n * es + vb) + 4 * n * es + (2 * n * es + 2 * vb) + (4 * n * es + 3 * vb)

    def step():
        oracle.residual_gate_add(o, h, u, gb, B, rows, D, "bf16", "bcast", threads=cores)
        oracle.residual_gate_add(hh, hh, u, gb, B, rows, D, "bf16", "bcast", threads=cores)
        oracle.residual_gate_add(o, h, u, gf, B, rows, D, "bf16", "full", threads=cores)
        oracle.rmsnorm_modulate(o, h, sc, sh, B, rows, D, EPS, "bf16", "bcast", threads=cores)
        oracle.gate_add_rmsnorm_modulate(o, o2, h, u, gb, sc, sh, B, rows, D, EPS, "bf16",
                                         "bcast", "bcast", threads=cores)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    value = step_bytes * args.steps / el / 1e9
    sample = (f"each step: the 5 hot-path ops on {rows} of the 32640 rows of "
              f"[1,32640,4096] bf16 on {cores} threads")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el * 1e3 / max(args.steps, 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": hotpath_config(),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import torch
    world, rank, local = dist_env()
    dist = None
    if world > 1:
        import torch.distributed as tdist
        torch.cuda.set_device(local)
        tdist.init_process_group("nccl", device_id=torch.device("cuda", local))
        dist = tdist
    else:
        torch.cuda.set_device(0)
    device = torch.device("cuda", torch.cuda.current_device())

    from diffusion_transformer_elementwise_gb300.build import build
    if rank == 0:
        build()
    if dist is not None:
        dist.barrier()
    build()  # no-op when up to date

    if args.workload == "fp8":
        ops = hotpath_ops(device, only="mod_fp8") + hotpath_ops(device, only="fused_fp8")
        workload = {"workload": "ltx2_bcast_s32640_c4096 modulation and fused op with an E4M3 "
                                "(FP8) modulated output, per-tensor scale",
                    "B": 1, "L": 32640, "D": 4096}
    elif args.workload == "gelu":
        ops = hotpath_ops(device, only="gelu_ffn")
        workload = {"workload": "ltx2 feed-forward tanh-GELU on [1,32640,16384] bf16",
                    "B": 1, "L": 32640, "D": 16384}
    elif args.workload == "chain_av":
        video = tuple(int(v) for v in args.chain_shape.split(","))
        audio = tuple(int(v) for v in args.audio_shape.split(","))
        ops = chain_av_ops(device, video, audio, graph=args.graph, grouped=not args.separate)
        B, L, D = video
        workload = {"workload": f"ltx2 video {list(video)} + audio {list(audio)} bf16 chain: "
                                f"8 DiT blocks x 3 sites, "
                                + ("one launch per stream and site" if args.separate else
                                   "one grouped launch per site for both streams")
                                + (", replayed as one CUDA graph" if args.graph else ""),
                    "video": list(video), "audio": list(audio), "blocks": 8}
    elif args.workload == "chain":
        B, L, D = (int(v) for v in args.chain_shape.split(","))
        ops = chain_ops(device, B, L, D, graph=args.graph)
        workload = {"workload": f"ltx2_chain_b{B}_s{L}_c{D}: 8 DiT blocks x 3 sites "
                                "(1 modulation + 23 fused + 1 residual gate per step)"
                                + (", replayed as one CUDA graph" if args.graph else ""),
                    "B": B, "L": L, "D": D, "blocks": 8}
    else:
        ops = hotpath_ops(device, only=args.op)
        workload = hotpath_config()
        if args.op:
            workload["workload"] = f"ltx2_bcast_s32640_c4096 {args.op} only (profiling)"
    big = args.workload not in ("chain", "chain_av") or B * L * D * 2 > (129 << 20)
    if args.workload != "hotpath" or args.op:
        workload["l2"] = ("no flush: every op reads its own inputs, each 267 MB or more, "
                          "above the 129 MB L2" if big else
                          "no flush: the chain's buffers fit in the L2 (launch-bound case)")
        workload["eps"] = EPS

    with ClockSampler(local) as clk:
        total_ms, per_op = time_steps(ops, args.steps, args.warmup, dist)
    clocks = clk.summary()

    from diffusion_transformer_elementwise_gb300.replicas import aggregate_gbs, max_over_ranks
    max_ms = max_over_ranks(total_ms, device)
    step_bytes = sum(op.bytes for op in ops)
    value = aggregate_gbs(step_bytes, args.steps, world, max_ms)

    peak, peak_kind = hbm_peak()
    table = {}
    for name, d in per_op.items():
        avg_ms = sum(d["ms"]) / len(d["ms"])
        gbs = d["bytes"] / (avg_ms * 1e-3) / 1e9
        table[name] = {"us_per_call": avg_ms * 1e3, "median_us": statistics.median(d["ms"]) * 1e3,
                       "min_us": min(d["ms"]) * 1e3, "bytes": d["bytes"], "GB_s": gbs,
                       "frac_of_peak": gbs / peak, "calls": d["calls"],
                       "share": sum(d["ms"]) / sum(sum(x["ms"]) for x in per_op.values())}
    # the dominant KERNEL: ops that launch the same kernel (the [1,1,D]-gate
    # residual gate out of place and in place) are counted together
    kernels = {}
    for op in ops:
        d = per_op[op.name]
        k = kernels.setdefault(KERNEL_OF.get(op.name, op.name), {"ms": 0.0, "bytes": 0, "calls": 0})
        k["ms"] += sum(d["ms"])
        k["bytes"] += d["bytes"] * d["calls"]
        k["calls"] += d["calls"]
    dom = max(kernels, key=lambda k: kernels[k]["ms"])
    kd = kernels[dom]
    achieved = kd["bytes"] / (kd["ms"] * 1e-3) / 1e9
    traffic = stored_traffic(dom)
    roof = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak,
            "unit": "GB/s", "frac": achieved / peak,
            "share": kd["ms"] / sum(k["ms"] for k in kernels.values()),
            "peak_source": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
            if peak_kind == "measured" else "fallback 6.8 TB/s",
            "traffic": traffic,
            "algorithmic_bytes_per_launch": kd["bytes"] / kd["calls"]}

    e2e = None
    if not args.no_e2e:
        e_steps = max(3, min(args.steps, 20))
        e_ms, h2d, d2h = time_e2e(ops, e_steps)
        e_max = max_over_ranks(e_ms, device)
        e2e = {"value": aggregate_gbs(step_bytes, e_steps, world, e_max), "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e_steps,
               "ms_per_step": e_max / e_steps}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu and args.workload == "hotpath":
        cpu = cpu_baseline(ops)

    if dist is not None:
        dist.barrier()
    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": max_ms / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic", "config": workload, "roofline": roof,
                "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": sum(op.launches for op in ops) * args.steps, "clocks": clocks,
                "statistic": args.statistic, "per_op": table}
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def run_copy(args):
    """Reference copies of 512 MB of bf16 (256 Mi elements) back to back, with
    the clocking of the library's kernels: torch's copy_ (a device-to-device
    memcpy, the copy MEASURED_PEAKS.json's peak was taken with; ncu profiles
    kernels only, so it cannot see it) and the same bytes through an SM
    kernel ncu can profile -- torch's elementwise multiply by one (exact),
    reading 512 MB and writing 512 MB.  Bytes per call = read + write = 1 GiB.
    No kernel of this library runs."""
    import torch
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    n = 256 << 20
    a = torch.ones(n, dtype=torch.bfloat16, device=dev)
    b = torch.empty_like(a)
    nbytes = 2 * n * 2
    peak, _ = hbm_peak()
    calls = {"copy_": lambda: b.copy_(a), "mul_by_one_kernel": lambda: torch.mul(a, 1.0, out=b)}
    out = {}
    with ClockSampler(0) as clk:
        for name, fn in calls.items():
            for _ in range(args.warmup):
                fn()
            torch.cuda.synchronize()
            times = []
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            for _ in range(args.steps):
                s.record()
                fn()
                e.record()
                torch.cuda.synchronize()
                times.append(s.elapsed_time(e))
            med = statistics.median(times)
            out[name] = {"median_us": med * 1e3, "min_us": min(times) * 1e3,
                         "GB_s": nbytes / (med * 1e-3) / 1e9,
                         "GB_s_best": nbytes / (min(times) * 1e-3) / 1e9,
                         "of_measured_peak": nbytes / (med * 1e-3) / 1e9 / peak}
    print(json.dumps({"workload": "copy of [268435456] bf16 (512 MB read + 512 MB written per "
                                  "call)", "bytes": nbytes, "steps": args.steps,
                      "results": out, "clocks": clk.summary(), "gpu_launches": 0}), flush=True)
    return 0


def run_shapes(args):
    """One line per (shape, op): device-timed us per call with an L2 flush
    before every call, outside the timed region.  The flush *reads* a buffer
    of 4x the L2 size: a write-flush would leave the L2 full of dirty lines
    whose write-back then falls inside the next timed call.  Beside the
    single-call median (whose resolution is the event timer's ~2 us step):
    cold_us, 30 x (flush + call) minus 30 x flush, from which GB_s and
    frac_of_peak are computed; back-to-back and CUDA-graph means of 20 calls.
    Shapes with a full [B, L, D] gate also time the per-token modulation
    (modulate_full) and the fused op with full gate, scale and shift."""
    shapes = [("ltx2_full_s126_c2048", 1, 126, 2048, "full", "bf16"),
              ("flux2_bcast_s4608_c3072", 1, 4608, 3072, "bcast", "bf16"),
              ("ideogram4_bcast_s4096_c4608", 1, 4096, 4608, "bcast", "bf16"),
              ("flux2_bcast_s4096_c3072", 1, 4096, 3072, "bcast", "bf16"),
              ("flux2_bcast_s512_c3072", 1, 512, 3072, "bcast", "bf16"),
              ("ltx2_full_s8160_c4096", 1, 8160, 4096, "full", "bf16"),
              ("ltx2_bcast_s32640_c4096", 1, 32640, 4096, "bcast", "bf16")]
    shapes += [(f"tail_s4097_c{D}_{dt}", 1, 4097, D, "bcast", dt)
               for D in (3080, 3076, 3077) for dt in ("bf16", "fp16", "fp32")]
    shapes += [(f"flux2_bcast_s4608_c3072_{dt}", 1, 4608, 3072, "bcast", dt)
               for dt in ("fp16", "fp32")]
    if args.shape:
        wanted = set(args.shape.split(","))
        unknown = wanted - {s[0] for s in shapes}
        if unknown:
            raise SystemExit(f"unknown --shape {sorted(unknown)}; known: {[s[0] for s in shapes]}")
        shapes = [s for s in shapes if s[0] in wanted]
    import torch

    import diffusion_transformer_elementwise_gb300 as dit
    from diffusion_transformer_elementwise_gb300.build import build
    from diffusion_transformer_elementwise_gb300.synth import draw, seed_for
    build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.ones(4 * l2 // 4, dtype=torch.float32, device=dev)
    sink = torch.empty((), dtype=torch.float32, device=dev)
    peak, _ = hbm_peak()
    for name, B, L, D, lay, dt in shapes:
        es = 4 if dt == "fp32" else 2
        N, vbytes = B * L * D, B * D * es
        shp = (B, L, D) if lay == "full" else (B, 1, D)
        h = draw("act", (B, L, D), seed_for(name, "h"), dt, dev)
        u = draw("act", (B, L, D), seed_for(name, "u"), dt, dev)
        g = draw("gate", shp, seed_for(name, "g"), dt, dev)
        sc = draw("mod", (B, 1, D), seed_for(name, "sc"), dt, dev)
        sh = draw("mod", (B, 1, D), seed_for(name, "sh"), dt, dev)
        o, o2 = torch.empty_like(h), torch.empty_like(h)
        cases = [("residual_gate_" + lay, lambda: dit.residual_gate_add(h, u, g, out=o),
                  (4 * N * es) if lay == "full" else (3 * N * es + vbytes)),
                 ("modulate_bcast", lambda: dit.rmsnorm_modulate(h, sc, sh, EPS, out=o),
                  2 * N * es + 2 * vbytes),
                 ("fused_" + lay + "_bcast",
                  lambda: dit.gate_add_rmsnorm_modulate(h, u, g, sc, sh, EPS, residual_out=o,
                                                        modulated_out=o2),
                  4 * N * es + (3 * vbytes if lay == "bcast" else N * es + 2 * vbytes))]
        if lay == "full":  # per-token modulation: [B, L, D] scale and shift
            scf = draw("mod", (B, L, D), seed_for(name, "scf"), dt, dev)
            shf = draw("mod", (B, L, D), seed_for(name, "shf"), dt, dev)
            cases += [("modulate_full", lambda: dit.rmsnorm_modulate(h, scf, shf, EPS, out=o),
                       4 * N * es),
                      ("fused_full_full",
                       lambda: dit.gate_add_rmsnorm_modulate(h, u, g, scf, shf, EPS,
                                                             residual_out=o, modulated_out=o2),
                       7 * N * es)]
        if lay == "bcast" and dt == "bf16" and name.startswith(("ltx2", "flux2_bcast_s4608")):
            xf = draw("act", (B, L, 4 * D), seed_for(name, "ffn"), dt, dev)
            of = torch.empty_like(xf)
            cases.append(("gelu_tanh_ffn_4D", lambda: dit.gelu_tanh(xf, out=of), 2 * 4 * N * es))
        for op, fn, nbytes in cases:
            for _ in range(10):
                fn()
            times, hot = [], []
            for _ in range(max(args.steps, 30)):
                torch.amax(flush, dim=0, out=sink)  # read-only eviction of the L2
                s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                s.record()
                fn()
                e.record()
                torch.cuda.synchronize()
                times.append(s.elapsed_time(e))
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            for _ in range(20):
                fn()
            e.record()
            torch.cuda.synchronize()
            b2b = s.elapsed_time(e) / 20
            # the same 20 calls captured in a CUDA graph: no host work per launch
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=side):
                for _ in range(20):
                    fn()
            torch.cuda.current_stream().wait_stream(side)
            graph.replay()
            s.record()
            graph.replay()
            e.record()
            torch.cuda.synchronize()
            graph_us = s.elapsed_time(e) / 20 * 1e3
            del graph
            # the cold call without the event timer's ~2 us step: 30 x (flush
            # + call) minus 30 x flush, back to back (the call's write-back,
            # which lands in the next flush, counts against the call)
            def run_n(call, n=30):
                s.record()
                for _ in range(n):
                    call()
                e.record()
                torch.cuda.synchronize()
                return s.elapsed_time(e) / n
            def flush_only():
                torch.amax(flush, dim=0, out=sink)
            def flush_then_call():
                torch.amax(flush, dim=0, out=sink)
                fn()
            pairs = [(run_n(flush_only), run_n(flush_then_call)) for _ in range(3)]
            cold_us = statistics.median(b - a for a, b in pairs) * 1e3
            med = statistics.median(times)
            # bandwidth from cold_us (the event timer's step would inflate
            # the single-call median of a few-us call); the median's beside it
            gbs = nbytes / (cold_us * 1e-6) / 1e9 if cold_us > 0 else float("nan")
            gbs_med = nbytes / (med * 1e-3) / 1e9
            print(json.dumps({"shape": name, "op": op, "dtype": dt, "B": B, "L": L, "D": D,
                              "statistic": dit.get_statistic(),
                              "bytes": nbytes, "cold_us": cold_us, "GB_s": gbs,
                              "frac_of_peak": gbs / peak, "median_us": med * 1e3,
                              "min_us": min(times) * 1e3, "GB_s_median": gbs_med,
                              "frac_of_peak_median": gbs_med / peak,
                              "back_to_back_us": b2b * 1e3,
                              "graph_us": graph_us}), flush=True)
        del h, u, g, o, o2
        if lay == "full":
            del scf, shf
    return 0


def main():
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=["hotpath", "chain", "chain_av", "shapes", "gelu", "fp8",
                                          "copy"],
                   default="hotpath")
    p.add_argument("--chain-shape", default="2,32640,4096",
                   help="B,L,D of --workload chain (e.g. 1,126,2048: the audio stream)")
    p.add_argument("--audio-shape", default="1,126,2048",
                   help="B,L,D of the audio stream of --workload chain_av")
    p.add_argument("--graph", action="store_true",
                   help="--workload chain / chain_av: replay the chain as one captured CUDA graph")
    p.add_argument("--separate", action="store_true",
                   help="--workload chain_av: one launch per stream and site instead of "
                        "one grouped launch per site")
    p.add_argument("--shape", default=None,
                   help="--workload shapes: only these shapes (comma-separated names)")
    p.add_argument("--statistic", choices=["fast", "exact"], default="fast",
                   help="row statistic of the modulating operations (dit_set_statistic)")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--op", default=None,
                   help="time one op of the hot path only (rga_bcast, rga_bcast_inplace, "
                        "rga_full, mod_bcast, fused_bcast, gelu_ffn, mod_fp8, fused_fp8): "
                        "for profiling")
    args = p.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.statistic != "fast":
        from diffusion_transformer_elementwise_gb300.build import build
        build()
        import diffusion_transformer_elementwise_gb300 as dit
        dit.set_statistic(args.statistic)
    if args.workload == "shapes":
        return run_shapes(args)
    if args.workload == "copy":
        return run_copy(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
