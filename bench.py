#!/usr/bin/env python3
"""Benchmark of the gated delta rule forward pass on one GB300 per rank.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload hymo_bf16]

A step is one ``gdn_fwd`` call over the whole workload (every step of the hot
path runs inside it).  The workload is the HyMo-shaped bf16 layer (B=8,
T=4096, H=16, dk=dv=64).  Inputs live in HBM before the timed region; two
input sets of 201 MB each (larger than the 129 MB L2) alternate between
steps so no step reads inputs the previous step left in L2.  Under torchrun
(N > 1) every rank runs its own replica (weak scaling, no data-path
collective); the timed region is bracketed by a barrier and a device
synchronisation on both sides and the maximum time over ranks is reported.

``--impl reference`` times the fp64 CPU oracle (the only reference for this
method) on the host cores instead, on one batch row of the workload per step.
"""
from __future__ import annotations

import argparse
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from linear_attention_recurrence_gated_gb300 import workloads as W  # noqa: E402

METRIC = "GDN fwd tokens/s and TFLOP/s (% of GB300 bf16 roofline), 1 GPU"
UNIT = "tokens/s"
CHUNK = 64
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# --------------------------------------------------------------------------
# algorithmic work (per head-token; chunk C = 64; MMA flops = 2 per FMA)
# --------------------------------------------------------------------------
def flops_per_head_token(dk: int, dv: int, C: int = CHUNK) -> float:
    """KK^T, QK^T, W, U~, W.H, K~^T U, Q.H, P.U and the triangular inverse, per token."""
    return C * (6 * dk + 4 * dv) + 6 * dk * dv + C * C / 3.0


def bytes_per_head_token(dk: int, dv: int, elem: int) -> float:
    """q, k, v, beta read and o written at `elem` bytes, g read as fp32."""
    return elem * (2 * dk + 2 * dv + 1) + 4


def algorithmic_bytes(w: W.Workload, tokens: int, N: int, with_init: bool) -> float:
    elem = 4 if w.dtype == "fp32" else 2
    state = 4 * w.dk * w.dv * N * w.H * (2 if with_init else 1)
    return tokens * w.H * bytes_per_head_token(w.dk, w.dv, elem) + state


def algorithmic_flops(w: W.Workload, tokens: int) -> float:
    return tokens * w.H * flops_per_head_token(w.dk, w.dv)


# --------------------------------------------------------------------------
# distributed plumbing (barrier + max over ranks; no data-path collective)
# --------------------------------------------------------------------------
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not torch.distributed.is_initialized():
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        torch.distributed.init_process_group(backend=backend)
    return rank, world, local


def barrier(world: int):
    if world > 1:
        if torch.distributed.get_backend() == "nccl":
            torch.distributed.barrier(device_ids=[torch.cuda.current_device()])
        else:
            torch.distributed.barrier()


def capture_steps(launch, steps: int, dev, stream, eager: bool):
    """The K timed steps as one CUDA graph (None when timing eagerly).

    launch(i, s) issues step i on stream s.  The graph is captured on a side
    stream and replayed once, untimed, so that its upload is not timed either.
    Replaying the graph runs every launch of every step; it only removes the
    host's per-call overhead (argument marshalling, launch) from the timed
    region, where back-to-back launches of a 20-150 us kernel would otherwise
    leave the GPU idle between them."""
    if eager:
        return None
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(stream)
    # relaxed: the library sets kernel attributes from the launching thread
    with torch.cuda.graph(g, stream=cap, capture_error_mode="relaxed"):
        for i in range(steps):
            launch(i, cap)
    stream.wait_stream(cap)
    g.replay()
    torch.cuda.synchronize(dev)
    return g


def run_steps(graph, launch, steps: int, stream):
    """Issue the K timed steps on `stream`: the captured graph, or eagerly."""
    if graph is not None:
        graph.replay()
    else:
        for i in range(steps):
            launch(i, stream)


TIMING_NOTE = {False: "the K steps captured as one CUDA graph, replayed once between CUDA events "
                      "(every launch runs; host launch overhead is not timed)",
               True: "the K steps launched one by one from the host between CUDA events"}


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------
# clocks sampled during the timed region
# --------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("timestamp,index,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, period_ms: int = 50):
        self.rows = []
        self.proc = None
        self.period_ms = period_ms
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.period_ms)], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self._t is not None:
                self._t.join(timeout=5)

    def summary(self, t0: float, t1: float, bus_id: str | None):
        sel = []
        for ts, line in self.rows:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 11:
                continue
            if bus_id and bus_id.lower() not in parts[2].lower():
                continue
            sel.append((ts, parts))
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"],
                    "samples": 0}
        inside = [p for ts, p in sel if t0 - 0.06 <= ts <= t1 + 0.06]
        use = inside or [min(sel, key=lambda r: min(abs(r[0] - t0), abs(r[0] - t1)))[1]]

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[3]) for p in use if num(p[3]) is not None]
        mx = [num(p[4]) for p in use if num(p[4]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in use for i in range(4)
                          if p[7 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(inside), "power_w_max": max(
                    (num(p[5]) for p in use if num(p[5]) is not None), default=None)}


# --------------------------------------------------------------------------
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


# The translation unit each kernel is compiled from; with the shared headers it
# fixes the machine code whose counters a profile summary records.
KERNEL_SOURCES = {
    "decode": "gdn_decode.cu",
    "simt_fp32": "gdn_fwd_simt.cu",
    "simt_bf16": "gdn_fwd_simt.cu",
    "tc64_bf16": "gdn_fwd_tc64.cu",
    "tc128_bf16": "gdn_fwd_tc128.cu",
    "tcc32_bf16": "gdn_fwd_tcc.cu",
    "tcc128_bf16": "gdn_fwd_tcc.cu",
    "diag_bf16": "gdn_diag.cu",
    "diag_fp32": "gdn_diag.cu",
    "diag_delta_bf16": "gdn_diag_delta.cu",
    "diag_delta_fp32": "gdn_diag_delta.cu",
    "conv_bf16": "gdn_conv.cu",
    "conv_fp32": "gdn_conv.cu",
    "bwd_chunk": "gdn_bwd_chunk.cu",
}


def code_only(text: str) -> str:
    """C/C++/CUDA source without its comments, trailing blanks and empty lines:
    the part of a file that decides what a kernel does."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        elif c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(c)
            i += 1
    lines = [ln.rstrip() for ln in "".join(out).splitlines()]
    return "\n".join(ln for ln in lines if ln)


def kernel_sources_hash(kernel: str) -> str:
    """sha256 prefix over the code (comments left out) of the kernel's .cu
    file, every csrc header and the public header (host-side files such as the
    ABI layer are left out).  A profile's counters stay valid while it matches."""
    import glob
    import hashlib
    csrc = os.path.join(ROOT, "linear_attention_recurrence_gated_gb300", "csrc")
    files = [os.path.join(csrc, KERNEL_SOURCES[kernel])]
    files += sorted(glob.glob(os.path.join(csrc, "*.cuh")))
    files.append(os.path.join(ROOT, "include", "gdn.h"))
    h = hashlib.sha256()
    for p in files:
        with open(p, encoding="utf-8") as f:
            h.update(code_only(f.read()).encode())
    return h.hexdigest()[:16]


def committed_traffic(kernel: str, workload: str):
    """dram bytes per launch from the committed ncu summary of this kernel and
    workload, or None when absent or taken on other kernel sources."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    s = re.search(r"source_sha:\s*([0-9a-f]+)", text)
    if not m or not s or kernel not in KERNEL_SOURCES or s.group(1) != kernel_sources_hash(kernel):
        return None
    return float(m.group(1))


def run_cpu_baseline(w: W.Workload, inputs, rows=None):
    """Time the oracle as it stands on the host cores; return (tokens/s, cores, secs)."""
    import oracle
    oracle.build()
    sel = slice(None) if rows is None else rows
    q, k, v = inputs["q"][sel], inputs["k"][sel], inputs["v"][sel]
    g, beta = inputs["g"][sel], inputs["beta"][sel]
    s0 = inputs["initial_state"]
    if s0 is not None and rows is not None:
        s0 = s0[sel]
    cores = oracle.default_threads()
    t = time.perf_counter()
    oracle.forward(q, k, v, g, beta, s0, inputs["cu_seqlens"], threads=cores)
    dt = time.perf_counter() - t
    return q.shape[0] * q.shape[1] / dt, cores, dt


# --------------------------------------------------------------------------
def bench_reference(args, w: W.Workload, rank: int, world: int):
    if rank != 0:
        return 0
    inputs = W.generate(w)
    B = inputs["q"].shape[0]
    for i in range(args.warmup):
        run_cpu_baseline(w, inputs, rows=slice(i % B, i % B + 1))
    times, toks = [], 0
    cores = 1
    for i in range(args.steps):
        rate, cores, dt = run_cpu_baseline(w, inputs, rows=slice(i % B, i % B + 1))
        times.append(dt)
        toks += w.T
    total = sum(times)
    value = toks / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "dk": w.dk, "dv": w.dv,
                   "storage": w.dtype, "chunk": CHUNK,
                   "step": "one batch row (T tokens x H heads) per step"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"one batch row of {w.name} per step ({w.T} tokens x "
                                   f"{w.H} heads), {args.steps} steps"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def bench_ours(args, w: W.Workload, rank: int, world: int, local: int):
    from linear_attention_recurrence_gated_gb300 import gdn as G
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU (no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    G.lib()

    host = W.generate(W.with_seed(w, w.seed + rank))
    N, tokens = host["N"], host["tokens"]
    names = ("q", "k", "v", "g", "beta")
    fused = getattr(args, "fused", False)
    if fused:  # the block parts fused into gdn_fwd: raw q/k, beta logits, skip and gate
        ex = W.generate_block_extras(host, w.H, seed=w.seed + 1000 + rank, dtype=w.dtype)
        host = dict(host, q=ex["q_raw"], k=ex["k_raw"], beta=ex["beta_logits"],
                    D_skip=ex["D_skip"], out_gate=ex["out_gate"])
        names = names + ("D_skip", "out_gate")
    split = getattr(args, "seq_split", False)
    segments = 1
    if split:
        segments = G.gdn_fwd_split_segments(N, host["q"].shape[1], w.H, w.dk, w.dv,
                                            host["q"].dtype, G.GDN_SEQ_SPLIT, args.chunk,
                                            varlen=host["cu_seqlens"] is not None)
    fkw = lambda d: dict(  # noqa: E731
        **(dict(D_skip=d["D_skip"], out_gate=d["out_gate"], beta_logits=True, qk_l2norm=True)
           if fused else {}), **(dict(seq_split=True) if split else {}))
    sets = []
    for _ in range(2):  # two resident input sets, alternated between steps
        d = {n: host[n].to(dev) for n in names}
        d["initial_state"] = None if host["initial_state"] is None else host["initial_state"].to(dev)
        d["cu_seqlens"] = None if host["cu_seqlens"] is None else host["cu_seqlens"].to(dev)
        d["o"] = torch.empty_like(d["v"])
        d["final_state"] = torch.empty((N, w.H, w.dk, w.dv), dtype=torch.float32, device=dev)
        sets.append(d)
    ws = G.new_workspace(N, w.H, w.dk, w.dv, G.GDN_SEQ_SPLIT if split else 0, device=dev,
                         seq_len=host["q"].shape[1] if split and host["cu_seqlens"] is None else None)
    kname = G.gdn_fwd_kernel_name(w.dk, w.dv, host["q"].dtype, G.GDN_QK_L2NORM if fused else 0,
                                  chunk_size=args.chunk)
    stream = torch.cuda.current_stream(dev)

    def step(i, s=stream):
        d = sets[i & 1]
        G.gdn_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"],
                  d["cu_seqlens"], o=d["o"], final_state=d["final_state"], workspace=ws,
                  chunk_size=args.chunk, stream=s, **fkw(d))

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    st = G.gdn_check(ws, stream)
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {G.status_string(st)}")

    graph = capture_steps(step, args.steps, dev, stream, args.eager)
    clocks = ClockSampler()
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize(dev)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    t_start.record(stream)
    run_steps(graph, step, args.steps, stream)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    wall1 = time.time()
    barrier(world)
    time.sleep(0.15)
    clocks.stop()
    st = G.gdn_check(ws, stream)
    if st != 0:
        raise RuntimeError(f"device status after timed steps: {G.status_string(st)}")

    local_ms = t_start.elapsed_time(t_end)
    total_ms = max_over_ranks(local_ms, world)
    per_launch_ms = local_ms / args.steps   # one gdn_fwd call per step
    value = tokens * world * args.steps / (total_ms / 1e3)

    # ---- end to end: pinned host inputs -> device -> gdn_fwd -> host result ----
    # Double-buffered over the two device sets, as a serving loop would run it:
    # the host-to-device copy of step i+1's inputs runs on its own stream while
    # step i computes, and step i's result is read back on a third stream.
    # Every step copies its whole input set in and its whole result out inside
    # the timed region; a set is refilled only after the step that last read
    # it has finished, and recomputed only after its result has been read back.
    pinned = {n: host[n].pin_memory() for n in names}
    s0_pinned = None if host["initial_state"] is None else host["initial_state"].pin_memory()
    o_host = torch.empty(host["v"].shape, dtype=host["v"].dtype).pin_memory()
    s_host = torch.empty((N, w.H, w.dk, w.dv), dtype=torch.float32).pin_memory()
    e2e_steps = max(1, min(args.steps, 50))
    h2d = sum(pinned[n].numel() * pinned[n].element_size() for n in names) + \
        (0 if s0_pinned is None else s0_pinned.numel() * 4)
    d2h = o_host.numel() * o_host.element_size() + s_host.numel() * 4
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    h2d_done = [torch.cuda.Event(), torch.cuda.Event()]
    comp_done = [torch.cuda.Event(), torch.cuda.Event()]
    d2h_done = [torch.cuda.Event(), torch.cuda.Event()]

    def e2e_step(i):
        b = i & 1
        d = sets[b]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(comp_done[b])    # step i-2 has read this input set
            for n in names:
                d[n].copy_(pinned[n], non_blocking=True)
            if s0_pinned is not None:
                d["initial_state"].copy_(s0_pinned, non_blocking=True)
            h2d_done[b].record(s_in)
        stream.wait_event(h2d_done[b])
        if i >= 2:
            stream.wait_event(d2h_done[b])       # step i-2's result has been read back
        G.gdn_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"],
                  d["cu_seqlens"], o=d["o"], final_state=d["final_state"], workspace=ws,
                  chunk_size=args.chunk, stream=stream, **fkw(d))
        comp_done[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[b])
            o_host.copy_(d["o"], non_blocking=True)
            s_host.copy_(d["final_state"], non_blocking=True)
            d2h_done[b].record(s_out)

    def e2e_run(nsteps, e_begin=None, e_end=None):
        if e_begin is not None:
            e_begin.record(stream)
        s_in.wait_stream(stream)
        s_out.wait_stream(stream)
        for i in range(nsteps):
            e2e_step(i)
        for b in range(min(nsteps, 2)):
            stream.wait_event(d2h_done[b])
        if e_end is not None:
            e_end.record(stream)

    e2e_run(3)
    torch.cuda.synchronize(dev)
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e2e_run(e2e_steps, e0, e1)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    barrier(world)
    st = G.gdn_check(ws, stream)
    if st != 0:
        raise RuntimeError(f"device status after e2e steps: {G.status_string(st)}")
    e2e_value = tokens * world * e2e_steps / (e2e_ms / 1e3)

    if rank != 0:
        return 0

    hbm_gbs, bf16_tflops, peak_src = measured_peaks()
    alg_bytes = algorithmic_bytes(w, tokens, N, host["initial_state"] is not None)
    if fused:   # the fp32 output gate is read too (D_skip: H floats)
        alg_bytes += tokens * w.H * 4 + w.H * 4
    alg_flops = algorithmic_flops(w, tokens)   # counted at the 64-token chunk
    achieved_gbs = alg_bytes / (per_launch_ms / 1e3) / 1e9
    achieved_tflops = alg_flops / (per_launch_ms / 1e3) / 1e12
    traffic = committed_traffic(kname, w.name)
    cpu_rate, cores, cpu_secs = run_cpu_baseline(w, host)
    clk = clocks.summary(wall0, wall1, _bus_id(local))
    arith = "f32" if kname.startswith("simt") else "bf16"
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": arith, "data": "synthetic",
        "timing": TIMING_NOTE[args.eager],
        "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "dk": w.dk, "dv": w.dv,
                   "storage": w.dtype, "chunk": args.chunk, "kernel": kname,
                   **({"fused": "q/k L2 norm + beta logits (sigmoid) + (o + D v) * out_gate "
                                "epilogue in the kernel"} if fused else {}),
                   **({"seq_split": f"GDN_SEQ_SPLIT: {segments} segment(s) per sequence"
                                    + (" (one launch: segment 0 + the later segments from zero "
                                       "and from the identity; composition steps; output "
                                       "correction; kernel_ms is the whole call)" if segments > 1
                                       else " (not split: the units fill the SMs)")}
                      if split else {}),
                   "l2": "two resident input sets of "
                         f"{sum(sets[0][n].numel() * sets[0][n].element_size() for n in names) / 1e6:.0f}"
                         " MB each (> 129 MB L2) alternate between steps",
                   "parallelism": f"replicas x{world}"},
        "tflops": achieved_tflops, "head_tokens_per_s": value * w.H,
        "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": hbm_gbs, "unit": "GB/s",
                     "frac": achieved_gbs / hbm_gbs, "traffic": traffic,
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_src == "measured" else "fallback 6.8 TB/s",
                     "algorithmic_bytes_per_launch": alg_bytes,
                     "kernel_ms": per_launch_ms,
                     "tensor_frac": achieved_tflops / bf16_tflops},
        "cpu_baseline": {"value": cpu_rate, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"the whole {w.name} workload ({tokens} tokens x {w.H} "
                                   f"heads), one pass, {cpu_secs:.1f} s"},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "overlap": "two device sets: step i+1's inputs copy in while step i "
                           "computes and step i-1's result copies out"},
        # a split call: the segments, the composition steps and the correction
        "gpu_launches": args.steps * (3 if segments > 1 else launches_per_step(kname)),
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)
    return 0


def decode_bytes(w: W.Workload) -> float:
    """HBM bytes of one decode step: the fp32 state read and written, q, k, v,
    g, beta read and o written, for every (sequence, head)."""
    e = 4 if w.dtype == "fp32" else 2
    per_head = 2 * w.dk * w.dv * 4 + e * (2 * w.dk + 2 * w.dv + 1) + 4
    return float(w.B * w.H * per_head)


def bench_decode(args, w: W.Workload, rank: int, world: int, local: int):
    """One recurrent step per sequence (gdn_decode), the state updated in place."""
    from linear_attention_recurrence_gated_gb300 import gdn as G
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU (no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    G.lib()
    host = W.generate_decode(W.with_seed(w, w.seed + rank))
    names = ("q", "k", "v", "g", "beta")
    d = {n: host[n].to(dev) for n in names}
    state = host["state"].to(dev)
    o = torch.empty_like(d["v"])
    stream = torch.cuda.current_stream(dev)

    def step(i=0, s=stream):
        G.gdn_decode(d["q"], d["k"], d["v"], d["g"], d["beta"], state, o=o, state_out=state,
                     stream=s)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    graph = capture_steps(step, args.steps, dev, stream, args.eager)
    clocks = ClockSampler()
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize(dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    t0.record(stream)
    run_steps(graph, step, args.steps, stream)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    wall1 = time.time()
    barrier(world)
    time.sleep(0.15)
    clocks.stop()
    total_ms = max_over_ranks(t0.elapsed_time(t1), world)
    per_launch_ms = t0.elapsed_time(t1) / args.steps   # one launch per step
    tokens = w.B  # one token per sequence per step
    value = tokens * world * args.steps / (total_ms / 1e3)

    # end to end: the step's token inputs from pinned host memory, o back; the
    # state stays resident on the device between steps, as in a serving loop
    pinned = {n: host[n].pin_memory() for n in names}
    o_host = torch.empty(host["v"].shape, dtype=host["v"].dtype).pin_memory()
    h2d = sum(pinned[n].numel() * pinned[n].element_size() for n in names)
    d2h = o_host.numel() * o_host.element_size()
    e2e_steps = max(1, min(args.steps, 50))

    def e2e_step():
        for n in names:
            d[n].copy_(pinned[n], non_blocking=True)
        step()
        o_host.copy_(o, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize(dev)
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    barrier(world)
    if rank != 0:
        return 0

    hbm_gbs, _, peak_src = measured_peaks()
    alg_bytes = decode_bytes(w)
    achieved = alg_bytes / (per_launch_ms / 1e3) / 1e9
    # CPU baseline: the oracle on a sample of the sequences, as one-token steps
    import oracle
    oracle.build()
    rows = slice(0, 128)
    t_c = time.perf_counter()
    oracle.forward(host["q"][rows, None], host["k"][rows, None], host["v"][rows, None],
                   host["g"][rows, None], host["beta"][rows, None], host["state"][rows], None,
                   threads=oracle.default_threads())
    cpu_secs = time.perf_counter() - t_c
    clk = clocks.summary(wall0, wall1, _bus_id(local))
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "timing": TIMING_NOTE[args.eager],
        "config": {"workload": w.name, "B": w.B, "T": 1, "H": w.H, "dk": w.dk, "dv": w.dv,
                   "storage": w.dtype, "kernel": "decode",
                   "l2": f"the {w.B * w.H * w.dk * w.dv * 4 / 1e6:.0f} MB state (> 129 MB L2) "
                         "is read and written every step",
                   "parallelism": f"replicas x{world}"},
        "head_tokens_per_s": value * w.H,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                     "frac": achieved / hbm_gbs, "traffic": committed_traffic("decode", w.name),
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_src == "measured" else "fallback 6.8 TB/s",
                     "algorithmic_bytes_per_launch": alg_bytes, "kernel_ms": per_launch_ms},
        "cpu_baseline": {"value": 128 / cpu_secs, "unit": UNIT, "cores": oracle.default_threads(),
                         "kind": "oracle",
                         "sample": f"128 of the {w.B} sequences x {w.H} heads, one step, "
                                   f"{cpu_secs:.2f} s"},
        "e2e": {"value": tokens * world * e2e_steps / (e2e_ms / 1e3), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps},
        "gpu_launches": args.steps,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)
    return 0


def diag_bytes(w: W.DiagWorkload) -> float:
    """HBM bytes of one gdn_diag_fwd (or gdn_diag_delta_fwd) call: v, b, c (and
    beta) read and o written in the storage dtype, g read as fp32, per (token,
    head); the fp32 final state
    written (and the initial state read, when given) per (batch row, head)."""
    e = 4 if w.dtype == "fp32" else 2
    per_head_token = e * (2 * w.D + 2 * w.S + (1 if w.delta else 0)) + 4   # + beta
    state = 4 * w.S * w.D * w.B * w.H * (2 if w.init_state else 1)
    return float(w.B * w.T * w.H * per_head_token + state)


def _diag_oracle_pass(host, b_rows=None):
    import oracle.diag
    sel = slice(None) if b_rows is None else b_rows
    h0 = host["initial_state"]
    t = time.perf_counter()
    if "beta" in host:
        oracle.diag.forward_delta(host["v"][sel], host["b"][sel], host["c"][sel], host["g"][sel],
                                  host["A_log"], host["beta"][sel], None if h0 is None else h0[sel])
    else:
        oracle.diag.forward(host["v"][sel], host["b"][sel], host["c"][sel], host["g"][sel],
                            host["A_log"], None if h0 is None else h0[sel])
    return time.perf_counter() - t


def bench_diag_reference(args, w: W.DiagWorkload, rank: int, world: int):
    """The fp64 oracle of the diagonal-decay recurrence on the host, one batch
    row of the workload per step."""
    if rank != 0:
        return 0
    host = W.generate_diag(w)
    for i in range(args.warmup):
        _diag_oracle_pass(host, slice(i % w.B, i % w.B + 1))
    total = sum(_diag_oracle_pass(host, slice(i % w.B, i % w.B + 1)) for i in range(args.steps))
    value = w.T * args.steps / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "S": w.S, "D": w.D,
                   "storage": w.dtype, "step": "one batch row (T tokens x H heads) per step"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"one batch row of {w.name} per step ({w.T} tokens x "
                                   f"{w.H} heads), {args.steps} steps"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def bench_diag(args, w: W.DiagWorkload, rank: int, world: int, local: int):
    """The pages' diagonal-decay recurrence (gdn_diag_fwd), or the same decay
    combined with the delta rule (gdn_diag_delta_fwd), one call per step."""
    from linear_attention_recurrence_gated_gb300 import gdn as G
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU (no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    G.lib()
    from dataclasses import replace
    host = W.generate_diag(replace(w, seed=w.seed + rank))
    names = ("v", "b", "c", "g") + (("beta",) if w.delta else ())
    sets = []
    for _ in range(2):  # two resident input sets, alternated between steps
        d = {n: host[n].to(dev) for n in names}
        d["A_log"] = host["A_log"].to(dev)
        d["initial_state"] = None if host["initial_state"] is None else host["initial_state"].to(dev)
        d["o"] = torch.empty_like(d["v"])
        d["final_state"] = torch.empty((w.B, w.H, w.S, w.D), dtype=torch.float32, device=dev)
        sets.append(d)
    if w.delta:
        ws = G.new_diag_delta_workspace(w.B, w.T, w.H, w.S, w.D, device=dev)
        kname = "diag_delta_" + w.dtype
    else:
        ws = G.new_diag_workspace(w.B, w.T, w.H, w.S, w.D, device=dev)
        kname = "diag_" + w.dtype
    stream = torch.cuda.current_stream(dev)

    def call(d, s=stream):
        if w.delta:
            G.gdn_diag_delta_fwd(d["v"], d["b"], d["c"], d["g"], d["A_log"], d["beta"],
                                 d["initial_state"], o=d["o"], final_state=d["final_state"],
                                 workspace=ws, stream=s)
        else:
            G.gdn_diag_fwd(d["v"], d["b"], d["c"], d["g"], d["A_log"], d["initial_state"],
                           o=d["o"], final_state=d["final_state"], workspace=ws, stream=s)

    for i in range(args.warmup):
        call(sets[i & 1])
    torch.cuda.synchronize(dev)
    st = G.gdn_check(ws, stream)
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {G.status_string(st)}")
    graph = capture_steps(lambda i, s: call(sets[i & 1], s), args.steps, dev, stream, args.eager)
    clocks = ClockSampler()
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize(dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    t0.record(stream)
    run_steps(graph, lambda i, s: call(sets[i & 1], s), args.steps, stream)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    wall1 = time.time()
    barrier(world)
    time.sleep(0.15)
    clocks.stop()
    st = G.gdn_check(ws, stream)
    if st != 0:
        raise RuntimeError(f"device status after timed steps: {G.status_string(st)}")
    total_ms = max_over_ranks(t0.elapsed_time(t1), world)
    per_launch_ms = t0.elapsed_time(t1) / args.steps   # one launch per step
    tokens = w.B * w.T
    value = tokens * world * args.steps / (total_ms / 1e3)

    # end to end: pinned host inputs -> device -> gdn_diag_fwd -> o and final state back
    pinned = {n: host[n].pin_memory() for n in names}
    o_host = torch.empty(host["v"].shape, dtype=host["v"].dtype).pin_memory()
    s_host = torch.empty((w.B, w.H, w.S, w.D), dtype=torch.float32).pin_memory()
    h2d = sum(pinned[n].numel() * pinned[n].element_size() for n in names)
    d2h = o_host.numel() * o_host.element_size() + s_host.numel() * 4
    e2e_steps = max(1, min(args.steps, 50))
    d = sets[0]

    def e2e_step():
        for n in names:
            d[n].copy_(pinned[n], non_blocking=True)
        call(d)
        o_host.copy_(d["o"], non_blocking=True)
        s_host.copy_(d["final_state"], non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize(dev)
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    barrier(world)
    st = G.gdn_check(ws, stream)
    if st != 0:
        raise RuntimeError(f"device status after e2e steps: {G.status_string(st)}")
    if rank != 0:
        return 0

    hbm_gbs, _, peak_src = measured_peaks()
    alg_bytes = diag_bytes(w)
    achieved = alg_bytes / (per_launch_ms / 1e3) / 1e9
    cpu_secs = _diag_oracle_pass(host)
    clk = clocks.summary(wall0, wall1, _bus_id(local))
    in_mb = sum(sets[0][n].numel() * sets[0][n].element_size() for n in names) / 1e6
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
        "timing": TIMING_NOTE[args.eager],
        "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "S": w.S, "D": w.D,
                   "storage": w.dtype, "a_log": w.a_log, "kernel": kname,
                   "l2": f"two resident input sets of {in_mb:.0f} MB each alternate between "
                         f"steps ({2 * in_mb:.0f} MB > 129 MB L2)",
                   "parallelism": f"replicas x{world}"},
        "head_tokens_per_s": value * w.H,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                     "frac": achieved / hbm_gbs, "traffic": committed_traffic(kname, w.name),
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_src == "measured" else "fallback 6.8 TB/s",
                     "algorithmic_bytes_per_launch": alg_bytes, "kernel_ms": per_launch_ms},
        "cpu_baseline": {"value": tokens / cpu_secs, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"the whole {w.name} workload ({tokens} tokens x {w.H} "
                                   f"heads), one pass of the numpy oracle, {cpu_secs:.1f} s"},
        "e2e": {"value": tokens * world * e2e_steps / (e2e_ms / 1e3), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps},
        "gpu_launches": args.steps,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)
    return 0


def bench_conv(args, w: W.ConvWorkload, rank: int, world: int, local: int):
    """The GDN block prologue (gdn_conv_silu), one call per step."""
    from linear_attention_recurrence_gated_gb300 import gdn as G
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU (no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    G.lib()
    from dataclasses import replace
    host = W.generate_conv(replace(w, seed=w.seed + rank))
    nsets = 4   # 4 x (input + output) > 129 MB L2 for the pages' shape
    sets = [{"x": host["x"].to(dev), "y": torch.empty_like(host["x"], device=dev)}
            for _ in range(nsets)]
    wd = host["w"].to(dev)
    stream = torch.cuda.current_stream(dev)
    kname = "conv_" + w.dtype

    def call(d, s=stream):
        G.gdn_conv_silu(d["x"], wd, y=d["y"], stream=s)

    for i in range(args.warmup):
        call(sets[i % nsets])
    torch.cuda.synchronize(dev)
    graph = capture_steps(lambda i, s: call(sets[i % nsets], s), args.steps, dev, stream, args.eager)
    clocks = ClockSampler()
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize(dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    t0.record(stream)
    run_steps(graph, lambda i, s: call(sets[i % nsets], s), args.steps, stream)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    wall1 = time.time()
    barrier(world)
    time.sleep(0.15)
    clocks.stop()
    total_ms = max_over_ranks(t0.elapsed_time(t1), world)
    per_launch_ms = t0.elapsed_time(t1) / args.steps   # one launch per step
    tokens = w.B * w.T
    value = tokens * world * args.steps / (total_ms / 1e3)
    # end to end: pinned x in, y back
    x_pin = host["x"].pin_memory()
    y_host = torch.empty(host["x"].shape, dtype=host["x"].dtype).pin_memory()
    d = sets[0]
    e2e_steps = max(1, min(args.steps, 50))

    def e2e_step():
        d["x"].copy_(x_pin, non_blocking=True)
        call(d)
        y_host.copy_(d["y"], non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize(dev)
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    barrier(world)
    if rank != 0:
        return 0
    hbm_gbs, _, peak_src = measured_peaks()
    e = 4 if w.dtype == "fp32" else 2
    alg_bytes = 2.0 * w.B * w.T * w.C * e + w.C * w.K * 4
    achieved = alg_bytes / (per_launch_ms / 1e3) / 1e9
    import oracle.block
    rows = slice(0, 1)
    t_c = time.perf_counter()
    oracle.block.conv_silu(host["x"][rows], host["w"])
    cpu_secs = time.perf_counter() - t_c
    clk = clocks.summary(wall0, wall1, _bus_id(local))
    nbytes = host["x"].numel() * host["x"].element_size()
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "timing": TIMING_NOTE[args.eager],
        "config": {"workload": w.name, "B": w.B, "T": w.T, "C": w.C, "K": w.K,
                   "storage": w.dtype, "kernel": kname,
                   "l2": f"{nsets} resident input/output sets of {2 * nbytes / 1e6:.0f} MB "
                         f"alternate between steps ({2 * nsets * nbytes / 1e6:.0f} MB > 129 MB L2)",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                     "frac": achieved / hbm_gbs, "traffic": committed_traffic(kname, w.name),
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_src == "measured" else "fallback 6.8 TB/s",
                     "algorithmic_bytes_per_launch": alg_bytes, "kernel_ms": per_launch_ms},
        "cpu_baseline": {"value": w.T / cpu_secs, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"one batch row of {w.name} ({w.T} tokens x {w.C} channels), "
                                   f"numpy oracle, {cpu_secs:.2f} s"},
        "e2e": {"value": tokens * world * e2e_steps / (e2e_ms / 1e3), "unit": UNIT,
                "h2d_bytes_per_step": nbytes, "d2h_bytes_per_step": nbytes, "steps": e2e_steps},
        "gpu_launches": args.steps,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)
    return 0


def bwd_bytes(w: W.Workload, tokens: int, N: int) -> float:
    """HBM bytes of one gdn_bwd call at its algorithmic minimum: q, k, v, beta,
    d_o read in the storage dtype and g as fp32; dq, dk, dv, dg, dbeta written
    in fp32; the fp32 d initial state written per (sequence, head)."""
    e = 4 if w.dtype == "fp32" else 2
    per = e * (2 * w.dk + 2 * w.dv + 1) + 4 + 4 * (2 * w.dk + w.dv + 2)
    return float(tokens * w.H * per + 4 * w.dk * w.dv * N * w.H)


# kernels per gdn_bwd call: (count, what they are), by path
BWD_LAUNCHES = {
    False: (2, "4 zero fills, the checkpoint scan, the backward"),
    True: (4, "chunked: prep, forward state chain, reverse chain, gradients"),
}


def bench_bwd(args, w: W.Workload, rank: int, world: int, local: int):
    """The backward pass (gdn_bwd) on a forward workload, one call per step."""
    from linear_attention_recurrence_gated_gb300 import gdn as G
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU (no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    G.lib()
    host = W.generate(W.with_seed(w, w.seed + rank))
    N, tokens = host["N"], host["tokens"]
    names = ("q", "k", "v", "g", "beta")
    rng = __import__("numpy").random.default_rng(17 + rank)
    d_o_host = torch.from_numpy(rng.standard_normal(tuple(host["v"].shape))).to(host["v"].dtype)
    d = {n: host[n].to(dev) for n in names}
    d["d_o"] = d_o_host.to(dev)
    s0 = None if host["initial_state"] is None else host["initial_state"].to(dev)
    cu = None if host["cu_seqlens"] is None else host["cu_seqlens"].to(dev)
    B, T = host["q"].shape[:2]
    ws = torch.zeros(G.gdn_bwd_workspace_size(N, T, w.H, w.dk, w.dv), dtype=torch.uint8,
                     device=dev)
    f32 = dict(dtype=torch.float32, device=dev)
    grads = {"dq": torch.empty((B, T, w.H, w.dk), **f32),
             "dk": torch.empty((B, T, w.H, w.dk), **f32),
             "dv": torch.empty((B, T, w.H, w.dv), **f32), "dg": torch.empty((B, T, w.H), **f32),
             "dbeta": torch.empty((B, T, w.H), **f32),
             "dh0": torch.empty((N, w.H, w.dk, w.dv), **f32)}
    stream = torch.cuda.current_stream(dev)

    def call(i=0, s=stream):
        G.gdn_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["d_o"], s0, cu, None,
                  grads=grads, workspace=ws, stream=s)

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize(dev)
    st = G.gdn_check(ws, stream)
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {G.status_string(st)}")
    graph = capture_steps(call, args.steps, dev, stream, args.eager)
    clocks = ClockSampler()
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize(dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    t0.record(stream)
    run_steps(graph, call, args.steps, stream)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    wall1 = time.time()
    barrier(world)
    time.sleep(0.15)
    clocks.stop()
    total_ms = max_over_ranks(t0.elapsed_time(t1), world)
    per_ms = total_ms / args.steps
    value = tokens * world * args.steps / (total_ms / 1e3)
    # end to end: inputs and d_o from pinned host memory, the five gradients back.
    # Double-buffered over two device sets, as a training loop would run it:
    # step i+1's inputs copy in on one stream while step i computes, and step
    # i's gradients copy out on a third; a set is refilled only after the step
    # that read it has finished, and recomputed only after its gradients have
    # been read back.
    pinned = {n: host[n].pin_memory() for n in names}
    do_pin = d_o_host.pin_memory()
    back = {n: torch.empty(t.shape, dtype=torch.float32).pin_memory()
            for n, t in grads.items() if n != "dh0"}
    h2d = sum(t.numel() * t.element_size() for t in pinned.values()) + do_pin.numel() * do_pin.element_size()
    d2h = sum(t.numel() * 4 for t in back.values())
    e2e_steps = max(1, min(args.steps, 10))
    sets = [(d, grads)]
    d2 = {n: torch.empty_like(t) for n, t in d.items()}
    sets.append((d2, {n: torch.empty_like(t) for n, t in grads.items()}))
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    h2d_done = [torch.cuda.Event(), torch.cuda.Event()]
    comp_done = [torch.cuda.Event(), torch.cuda.Event()]
    d2h_done = [torch.cuda.Event(), torch.cuda.Event()]

    def e2e_step(i):
        bsel = i & 1
        dd, gg = sets[bsel]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(comp_done[bsel])   # step i-2 has read this input set
            for n in names:
                dd[n].copy_(pinned[n], non_blocking=True)
            dd["d_o"].copy_(do_pin, non_blocking=True)
            h2d_done[bsel].record(s_in)
        stream.wait_event(h2d_done[bsel])
        if i >= 2:
            stream.wait_event(d2h_done[bsel])      # step i-2's gradients have been read back
        G.gdn_bwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dd["d_o"], s0, cu, None,
                  grads=gg, workspace=ws, stream=stream)
        comp_done[bsel].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[bsel])
            for n, t in back.items():
                t.copy_(gg[n], non_blocking=True)
            d2h_done[bsel].record(s_out)

    def e2e_run(nsteps, e_begin=None, e_end=None):
        if e_begin is not None:
            e_begin.record(stream)
        s_in.wait_stream(stream)
        s_out.wait_stream(stream)
        for i in range(nsteps):
            e2e_step(i)
        for bsel in range(min(nsteps, 2)):
            stream.wait_event(d2h_done[bsel])
        if e_end is not None:
            e_end.record(stream)

    e2e_run(2)
    torch.cuda.synchronize(dev)
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_run(e2e_steps, e0, e1)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    barrier(world)
    if rank != 0:
        return 0
    hbm_gbs, _, peak_src = measured_peaks()
    alg = bwd_bytes(w, tokens, N)
    chunked = w.dtype == "bf16" and w.dk <= 128 and w.dv <= 128
    achieved = alg / (per_ms / 1e3) / 1e9
    # CPU baseline: the autograd oracle on one head of one batch row, at most
    # 4096 tokens of it (about 4 s), scaled to the workload's heads
    import oracle.grad
    ts = min(T, 4096)
    t_c = time.perf_counter()
    oracle.grad.backward(host["q"][:1, :ts, :1], host["k"][:1, :ts, :1], host["v"][:1, :ts, :1],
                         host["g"][:1, :ts, :1], host["beta"][:1, :ts, :1], None,
                         d_o_host[:1, :ts, :1], None)
    cpu_secs = time.perf_counter() - t_c
    clk = clocks.summary(wall0, wall1, _bus_id(local))
    line = {
        "metric": "GDN backward tokens/s (gdn_bwd), 1 GPU", "value": value, "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        # the chunked path multiplies bf16 operands with fp32 accumulation; the
        # token-serial path computes in fp32
        "dtype": "bf16" if chunked else "f32", "data": "synthetic",
        "timing": TIMING_NOTE[args.eager],
        "config": {"workload": w.name, "pass": "backward", "B": w.B, "T": w.T, "H": w.H,
                   "dk": w.dk, "dv": w.dv, "storage": w.dtype, "kernel": "bwd",
                   "l2": "inputs, d_o and the fp32 gradients (> 129 MB) stream every step",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                     "frac": achieved / hbm_gbs,
                     # DRAM bytes of the four kernels of one call, from the committed summary
                     "traffic": committed_traffic("bwd_chunk", w.name) if chunked else None,
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_src == "measured" else "fallback 6.8 TB/s",
                     "algorithmic_bytes_per_launch": alg, "kernel_ms": per_ms,
                     "launches_per_step": BWD_LAUNCHES[chunked][1]},
        "cpu_baseline": {"value": ts / cpu_secs / w.H, "unit": UNIT, "cores": 1,
                         "kind": "oracle",
                         "sample": f"one head of one batch row ({ts} tokens), torch.autograd "
                                   f"fp64 oracle, {cpu_secs:.1f} s; value scaled to {w.H} heads"},
        "e2e": {"value": tokens * world * e2e_steps / (e2e_ms / 1e3), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "overlap": "two device sets: step i+1's inputs copy in while step i "
                           "computes, step i's gradients copy out on a third stream"},
        "gpu_launches": args.steps * BWD_LAUNCHES[chunked][0],
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)
    return 0


def launches_per_step(kernel_name: str) -> int:
    return 1


def _bus_id(local: int):
    try:
        p = torch.cuda.get_device_properties(local)
        dom = getattr(p, "pci_domain_id", None)
        bus = getattr(p, "pci_bus_id", None)
        devid = getattr(p, "pci_device_id", None)
        if bus is None:
            return None
        return f"{bus:02X}:{devid or 0:02X}" if dom is None else f"{dom:08X}:{bus:02X}:{devid or 0:02X}"
    except Exception:
        return None


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--pass", dest="pass_", choices=("fwd", "bwd"), default="fwd",
                    help="fwd: gdn_fwd; bwd: gdn_bwd (the prefill workloads)")
    ap.add_argument("--chunk", type=int, default=CHUNK, choices=(32, 64, 128),
                    help="chunk size of gdn_fwd (32 and 128: the tensor-core chunk-size variants "
                         "for bf16 with head_dim_k 64)")
    ap.add_argument("--workload", default="hymo_bf16",
                    choices=sorted(W.WORKLOADS) + sorted(W.DECODE_WORKLOADS) +
                    sorted(W.DIAG_WORKLOADS) + sorted(W.CONV_WORKLOADS))
    ap.add_argument("--eager", action="store_true",
                    help="time the steps launched one by one instead of as one CUDA graph")
    ap.add_argument("--seq-split", action="store_true",
                    help="fwd: GDN_SEQ_SPLIT (dense head_dim_k 128 sequences cut into segments "
                         "computed in parallel when units alone leave SMs idle)")
    ap.add_argument("--fused", action="store_true",
                    help="fwd: raw q/k normalised in-kernel, beta as logits and the block "
                         "epilogue (o + D v) * out_gate, all fused into gdn_fwd")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local = dist_setup()
    try:
        if args.workload in W.CONV_WORKLOADS:
            if args.impl == "reference":
                raise SystemExit("the reference arm times the recurrence workloads only")
            return bench_conv(args, W.CONV_WORKLOADS[args.workload], rank, world, local)
        if args.workload in W.DIAG_WORKLOADS:
            dw = W.DIAG_WORKLOADS[args.workload]
            if args.impl == "reference":
                return bench_diag_reference(args, dw, rank, world)
            return bench_diag(args, dw, rank, world, local)
        if args.workload in W.DECODE_WORKLOADS:
            if args.impl == "reference":
                raise SystemExit("the reference arm times the prefill workloads only")
            return bench_decode(args, W.DECODE_WORKLOADS[args.workload], rank, world, local)
        w = W.WORKLOADS[args.workload]
        if args.pass_ == "bwd":
            if args.impl == "reference":
                raise SystemExit("the reference arm times the forward pass only")
            return bench_bwd(args, w, rank, world, local)
        if args.impl == "reference":
            return bench_reference(args, w, rank, world)
        return bench_ours(args, w, rank, world, local)
    finally:
        if world > 1 and torch.distributed.is_initialized():
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
