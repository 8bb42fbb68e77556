#!/usr/bin/env python
"""SSD forward benchmark on GB300: prints ONE JSON line.

Default workload: the Mamba-2 2.7B-layer-shaped SSD forward (batch 4,
seqlen 4096, 80 heads, headdim 64, dstate 128, 1 group, chunk 256, bf16
x/B/C, f32 dt/A/D, zero initial state, final state returned).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--no-cpu-baseline]

Decode workloads (``--workload decode-...``) time ssd_decode_step instead:
one step is one token for every sequence of the batch on its carried f32
state, and the line's metric is decode tokens (sequences) per second.

Under torchrun (N > 1) every rank runs the same workload on its own GPU (the
units -- batch rows and heads -- are independent; no collective on the data
path), so scaling is weak and `value` counts the tokens of all ranks.

A step is one whole SSD forward (every stage) over one batch of synthetic
input resident in HBM.  Each timed step is bracketed by CUDA events on the
launching stream; L2 is flushed (512 MB write) before every timed step,
outside the events.  The step calls the same C-ABI stage entry points that
ssd_fwd dispatches to, with an event between stages, so the dominant
kernel's own duration is measured live for the roofline object.  `e2e`
times the public host-buffer call ssd_fwd_host (pinned inputs in, y and the
final state out, the copies overlapped with the kernels) inside the timed
region; a workload that also returns every chunk state times ssd_fwd
between explicit copies instead.
"""
from __future__ import annotations

import argparse
import dataclasses
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

import numpy as np  # noqa: E402
import torch  # noqa: E402

from state_space_sequence_cumsum_gb300.inputs import (EXTREME_256K, LAYER_2P7B, LONG_S256_G8,  # noqa: E402
                                                      PAGES_EXAMPLE, TINY_FP32, Shape,
                                                      make_inputs, sweep_shape)

METRIC = "SSD forward tokens/sec on 1 GB300 and % of roofline (H=80,P=64,S=128)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# name -> (shape, dtype, init, want chunk states)
WORKLOADS = {
    "mamba2-2.7b-layer-B4-L4096-H80-P64-S128-T256": (LAYER_2P7B, torch.bfloat16, "zero", False),
    "tiny-fp32-B1-L256-H2-P16-S16-T64": (TINY_FP32, torch.float32, "zero", False),
    "long-B2-L32768-H64-P64-S256-G8-T256": (LONG_S256_G8, torch.bfloat16, "randn", False),
    "extreme-B1-L262144-H32-P64-S512-T128-states": (EXTREME_256K, torch.bfloat16, "zero", True),
    "pages-example-B4-L16384-H8-P64-S128-T128": (PAGES_EXAMPLE, torch.bfloat16, "zero", False),
    # an eighth of the extreme-length shape (same kernels, 1.2 GB of chunk
    # states): the size the profiles of its kernels are captured on
    "extreme-slice-B1-L32768-H32-P64-S512-T128-states": (
        Shape(1, 32768, 32, 64, 512, 1, 128), torch.bfloat16, "zero", True),
}
# the length x dstate sweep with the chunk size chosen by the library's tuner
# (chunk_size 0: it times {64, 128, 256} once per shape before the warm-up)
for _L in (1024, 4096, 16384, 65536, 262144, 4095):
    for _S in (64, 128, 256, 512):
        _sh = sweep_shape(_L, _S, 0)
        WORKLOADS[f"sweep-B{_sh.batch}-L{_L}-H64-P64-S{_S}-Tauto"] = (_sh, torch.bfloat16, "zero",
                                                                      False)
TUNE_CANDIDATES = (64, 128, 256)
DEFAULT = "mamba2-2.7b-layer-B4-L4096-H80-P64-S128-T256"
# single-token decode steps on a carried state: name -> (batch, H, P, S, G, dtype)
DECODE = {
    "decode-B128-H80-P64-S128": (128, 80, 64, 128, 1, torch.bfloat16),
    "decode-B4-H80-P64-S128": (4, 80, 64, 128, 1, torch.bfloat16),
}
DECODE_METRIC = "SSD decode step: sequences (tokens) per second on 1 GB300, carried f32 state"
# gated RMS norm after the scan: name -> (tokens, dim, group_size, dtype)
NORM = {"gated-norm-B4-L4096-H80-P64": (4 * 4096, 80 * 64, 80 * 64, torch.bfloat16)}
NORM_METRIC = "Gated RMS norm (y * silu(z), one group per token) tokens/sec on 1 GB300"
# backward passes: name -> forward workload whose gradients are taken
BACKWARD = {"bwd-mamba2-2.7b-layer-B4-L4096-H80-P64-S128": "mamba2-2.7b-layer-B4-L4096-H80-P64-S128-T256"}
BWD_METRIC = "SSD backward tokens/sec on 1 GB300 (all input gradients from dy and dfinal)"


# ------------------------------------------------------------------ accounting

def elem_bytes(dtype):
    return 2 if dtype == torch.bfloat16 else 4


def compulsory_bytes(s: Shape, dtype, init: str, want_states: bool) -> int:
    """Bytes the forward must move at least once: read x, B, C, dt, A, D (and
    init), write y and the final state (and chunk states when requested)."""
    e = elem_bytes(dtype)
    n = 2 * s.batch * s.seqlen * s.nheads * s.headdim * e          # x read, y written
    n += 2 * s.batch * s.seqlen * s.ngroups * s.dstate * e          # B, C
    n += s.batch * s.seqlen * s.nheads * 4 + 2 * s.nheads * 4       # dt, A, D
    st = s.batch * s.nheads * s.headdim * s.dstate * 4
    n += st                                                          # final state
    if init == "randn":
        n += st
    if want_states:
        n += st * s.nchunks
    return n


def algorithmic_flops(s: Shape) -> int:
    """Per (batch, chunk of Tc tokens): per head 4 Tc S P (C h^T and the state
    jump) + P Tc (Tc + 1) (causal scores x X); per group S Tc (Tc + 1) (causal CB^T)."""
    total = 0
    for c in range(s.nchunks):
        tc = min(s.chunk_size, s.seqlen - c * s.chunk_size)
        per_head = 4 * tc * s.dstate * s.headdim + s.headdim * tc * (tc + 1)
        per_group = s.dstate * tc * (tc + 1)
        total += s.batch * (s.nheads * per_head + s.ngroups * per_group)
    return total


def kernel_bytes(kernel: str, s: Shape, dtype, init: str, want_states: bool) -> int:
    """Algorithmic bytes one launch of `kernel` must move (each operand once)."""
    e = elem_bytes(dtype)
    blh = s.batch * s.seqlen * s.nheads
    xb = blh * s.headdim * e
    bb = s.batch * s.seqlen * s.ngroups * s.dstate * e
    st = s.batch * s.nheads * s.headdim * s.dstate * 4
    states = st * s.nchunks
    init_b = st if init == "randn" else 0
    if kernel == "chunk_cumsum":
        return blh * 4 + blh * 8 + s.nheads * 4
    if kernel == "state_pass":
        return xb + bb + 2 * blh * 4 + init_b + states + st
    if kernel == "chunk_out":
        return xb + 2 * bb + 2 * blh * 4 + states + s.nheads * 4 + xb
    if kernel == "fused_pair":  # the whole forward in one kernel, G formed in the kernel
        return (xb + 2 * bb + blh * 4 + 2 * s.nheads * 4 + init_b + xb + st +
                (states if want_states else 0))
    if kernel == "state_out":  # fused stages 2+3
        return (xb + 2 * bb + 2 * blh * 4 + s.nheads * 4 + init_b + xb + st +
                (states if want_states else 0))
    raise KeyError(kernel)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def source_digest(files) -> str:
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, or
    None if absent or if the kernel's source changed since the capture."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        ent = d[kernel][workload]
        if ent["source_digest"] != source_digest(ent["sources"]):
            return None
        return int(ent["dram_bytes_per_launch"])
    except (OSError, ValueError, KeyError):
        return None


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 20 ms.  The sampler
    is started before the timed region (and waited for until it has written
    its first line); the summary keeps the samples whose timestamps fall in
    the marked region, or the two nearest ones if the region is shorter than
    the sampling interval."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            deadline = time.time() + 5.0
            while time.time() < deadline and os.path.getsize(self.path) == 0:
                time.sleep(0.01)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.05)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        samples = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                    samples.append((ts, float(parts[2]), float(parts[3]),
                                    [n for n, v in zip(names, parts[6:10]) if v.lower() == "active"]))
                except (ValueError, IndexError):
                    continue
        os.unlink(self.path)
        if not samples:
            return None
        t0, t1 = self.t0 or samples[0][0], self.t1 or samples[-1][0]
        inside = [s for s in samples if t0 <= s[0] <= t1]
        if not inside:  # region shorter than the interval: the nearest samples
            inside = sorted(samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))[:2]
        return {"sm_mhz": statistics.median(s[1] for s in inside),
                "sm_max_mhz": max(s[2] for s in inside),
                "reasons": sorted({r for s in inside for r in s[3]}), "samples": len(inside)}


# ------------------------------------------------------------------ oracle leg

def oracle_row(inp, s: Shape, b: int, threads: int):
    """Run the float64 oracle on batch row b (every head, the full sequence);
    return (seconds, tokens processed)."""
    import oracle
    sl = slice(b, b + 1)
    args = [oracle._f64(v) for v in (inp["x"][sl], inp["dt"][sl], inp["A"], inp["B"][sl],
                                     inp["C"][sl], inp["D"])]
    init = oracle._f64(None if inp["init"] is None else inp["init"][sl])
    # y and the final state do not depend on the chunk size (no chunk states
    # are asked for here), so a library-chosen one is timed at 128
    T = s.chunk_size or 128
    t0 = time.perf_counter()
    oracle.fwd(*args, T, init=init, nthreads=threads)
    return time.perf_counter() - t0, s.seqlen


def cpu_baseline(inp, s: Shape, budget_s: float = 12.0):
    """The oracle as it stands on the host cores, on a bounded sample: whole
    batch rows (all heads, the full sequence) in turn until about budget_s
    seconds of wall time have been spent."""
    import oracle
    oracle.build()
    threads = oracle.cpu_cores()
    t_acc, tokens, rows = 0.0, 0, 0
    while t_acc < budget_s:
        t, n = oracle_row(inp, s, rows % s.batch, threads)
        t_acc += t
        tokens += n
        rows += 1
    return {"value": round(tokens / t_acc, 1), "unit": "tokens/s", "cores": threads,
            "kind": "oracle",
            "sample": (f"float64 recurrence, {rows} batch rows (all {s.nheads} heads x "
                       f"{s.seqlen} tokens each, rows of the {s.batch}-row workload taken in "
                       f"turn) = {tokens} tokens in {t_acc:.2f} s wall")}


# ------------------------------------------------------------------ our arm

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, ws: int, device) -> float:
    """The largest of every rank's x: the job's step time is its slowest
    replica's.  One rank: x itself (no process group needed)."""
    if ws <= 1:
        return x
    t = torch.tensor([x], device=device, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(ws: int, units_per_rank: float, ms: float) -> float:
    """Whole-job units per second: every replica processes units_per_rank
    units in the (max-over-ranks) time ms."""
    return ws * units_per_rank / (ms / 1e3)


def run_ours(args):
    import state_space_sequence_cumsum_gb300 as ssd
    from state_space_sequence_cumsum_gb300 import _lib

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    shape, dtype, init, want_states = WORKLOADS[args.workload]
    T = shape.chunk_size
    auto = T == 0
    inp = make_inputs(shape, dtype=dtype, init=init, seed=rank)
    lib = _lib.load()

    g = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
    y = torch.empty_like(g["x"])
    fin = torch.empty((shape.batch, shape.nheads, shape.headdim, shape.dstate), device=dev)
    wsp = ssd.Workspace()
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    tuned = None
    if auto:
        # the library's per-shape choice: the first chunk_size=0 call times the
        # candidates and fixes the fastest (before the warm-up, untimed)
        ssd.ssd_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], chunk_size=0,
                    initial_state=g["init"], y=y, final_state=fin, workspace=wsp)
        torch.cuda.synchronize(dev)
        dims = (shape.batch, shape.seqlen, shape.nheads, shape.headdim, shape.dstate,
                shape.ngroups, dtype)
        T = ssd.ssd_fwd_chosen_chunk_size(*dims)
        tuned = ssd.ssd_fwd_chunk_size_was_timed(*dims)
        shape = dataclasses.replace(shape, chunk_size=T)
    states = (torch.empty((shape.batch, shape.nheads, shape.nchunks, shape.headdim,
                           shape.dstate), device=dev) if want_states else None)

    plan = ssd.ssd_fwd_plan(g["x"], g["B"], T, want_states=want_states)
    # the one-call path passes chunk_size 0 so the tuned plan choice applies
    plan["call_chunk_size"] = 0 if auto else T

    def step(events=None):
        return ssd.ssd_fwd_staged(plan, g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"],
                                  g["init"], y, fin, states, wsp, events=events)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    st = ssd.ssd_stream_status()
    if st != 0:
        raise RuntimeError(f"kernel status {st} during warm-up")

    nk = len(plan["kernels"])
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)] for _ in range(args.steps)]
    launches0 = lib.ssd_launch_count()
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        clk.mark_start()
        t_wall0 = time.perf_counter()
        for k in range(args.steps):
            flush.fill_(float(k))
            step(events=ev[k])
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter() - t_wall0
        clk.mark_end()
    if ws > 1:
        torch.distributed.barrier()
    launches = lib.ssd_launch_count() - launches0
    per_kernel = [[ev[k][i].elapsed_time(ev[k][i + 1]) for k in range(args.steps)]
                  for i in range(nk)]
    step_ms = [sum(per_kernel[i][k] for i in range(nk)) for k in range(args.steps)]
    ms = statistics.mean(step_ms)
    ms = max_over_ranks(ms, ws, dev)
    tokens = shape.tokens
    value = job_throughput(ws, tokens, ms)

    # dominant kernel and its roofline
    means = [statistics.mean(v) for v in per_kernel]
    dom = int(np.argmax(means))
    kname = plan["kernels"][dom]
    peaks, peak_src = load_peaks()
    kb = kernel_bytes(kname, shape, dtype, init, want_states)
    achieved = kb / (means[dom] / 1e3) / 1e9
    traffic = profiled_traffic(kname, args.workload)
    roofline = {"bound": "hbm", "kernel": kname, "achieved": round(achieved, 1),
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                "traffic": traffic, "algorithmic_bytes": kb, "kernel_ms": round(means[dom], 5),
                "peak_source": peak_src}
    # whole-step roofline: max(compulsory bytes / HBM, algorithmic flops / bf16 peak)
    cb = compulsory_bytes(shape, dtype, init, want_states)
    fl = algorithmic_flops(shape)
    t_roof = max(cb / (peaks["hbm_gbs"] * 1e9), fl / (peaks["bf16_tflops"] * 1e12))
    if auto:
        # a library-chosen chunk size: the roofline is the least over the
        # candidates, so a larger chunk cannot loosen it
        fls = {c: algorithmic_flops(dataclasses.replace(shape, chunk_size=c))
               for c in TUNE_CANDIDATES}
        c_min = min(fls, key=lambda c: max(cb / (peaks["hbm_gbs"] * 1e9),
                                           fls[c] / (peaks["bf16_tflops"] * 1e12)))
        fl = fls[c_min]
        t_roof = max(cb / (peaks["hbm_gbs"] * 1e9), fl / (peaks["bf16_tflops"] * 1e12))
    step_roof = {"compulsory_bytes": cb, "algorithmic_flops": fl,
                 "t_roof_us": round(t_roof * 1e6, 2), "frac": round(t_roof / (ms / 1e3), 4),
                 "bound": "hbm" if cb / peaks["hbm_gbs"] >= fl / (peaks["bf16_tflops"] * 1e3)
                 else "tensor"}
    if auto:
        step_roof["flops_at_chunk_size"] = c_min

    # e2e: public ssd_fwd call, pinned host inputs in, y + final out, per step
    host_in = {k: (None if v is None else v.pin_memory()) for k, v in inp.items()}
    y_host = torch.empty(y.shape, dtype=y.dtype).pin_memory()
    fin_host = torch.empty(fin.shape, dtype=fin.dtype).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in host_in.values() if v is not None)
    d2h = y_host.numel() * y_host.element_size() + fin_host.numel() * fin_host.element_size()

    # ssd_fwd_host (host buffers in and out, copies overlapped with the
    # kernels) when the step returns y and the final state; a step that also
    # returns every chunk state keeps them on the device, so it runs ssd_fwd
    # between explicit copies instead (ssd_fwd_host returns no chunk states).
    e2e_api = "ssd_fwd + copies" if want_states else "ssd_fwd_host"
    wsp_host = ssd.Workspace()

    def e2e_step():
        if not want_states:
            ssd.ssd_fwd_host(host_in["x"], host_in["dt"], host_in["A"], host_in["B"],
                             host_in["C"], host_in["D"], chunk_size=plan["call_chunk_size"],
                             initial_state=host_in["init"], y=y_host, final_state=fin_host,
                             workspace=wsp_host, device=dev, stream=stream)
            return
        for k, v in host_in.items():
            if v is not None:
                g[k].copy_(v, non_blocking=True)
        ssd.ssd_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], chunk_size=T,
                    initial_state=g["init"], y=y, final_state=fin, chunk_states=states,
                    return_chunk_states=want_states, workspace=wsp)  # explicit-T copy path
        y_host.copy_(y, non_blocking=True)
        fin_host.copy_(fin, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    e_ms = []
    for k in range(args.steps):
        flush.fill_(float(k))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        e2e_step()
        b.record(stream)
        b.synchronize()
        e_ms.append(a.elapsed_time(b))
    e_ms_mean = statistics.mean(e_ms)
    e_ms_mean = max_over_ranks(e_ms_mean, ws, dev)

    # the host link's own ceiling for the same bytes: the step's input copies
    # from pinned memory and its output copies back, plain copies on one
    # stream with no kernel between them (best of 5)
    def copies_only():
        for k, v in host_in.items():
            if v is not None:
                g[k].copy_(v, non_blocking=True)
        y_host.copy_(y, non_blocking=True)
        fin_host.copy_(fin, non_blocking=True)

    copies_only()
    c_ms = []
    for k in range(5):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        copies_only()
        b.record(stream)
        b.synchronize()
        c_ms.append(a.elapsed_time(b))
    copy_ms = min(c_ms)
    st = ssd.ssd_stream_status()
    if st != 0:
        raise RuntimeError(f"kernel status {st} in the timed region")

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if dtype == torch.bfloat16 else "f32", "data": "synthetic",
        "config": {"workload": args.workload, "batch": shape.batch, "seqlen": shape.seqlen,
                   "nheads": shape.nheads, "headdim": shape.headdim, "dstate": shape.dstate,
                   "ngroups": shape.ngroups, "chunk_size": T,
                   "chunk_size_choice": ("timed by the library over {64, 128, 256}" if tuned else
                                         "the library's static choice") if auto else "fixed",
                   "init": init,
                   "chunk_states": want_states, "parallelism": f"replicas{ws}",
                   "l2": "flushed before every timed step (512 MB write, outside the events)",
                   "path": plan["path"]},
        "roofline": roofline, "step_roofline": step_roof,
        "per_kernel_ms": {n: round(m, 5) for n, m in zip(plan["kernels"], means)},
        "wall_s_timed_loop": round(t_wall, 4),
        "e2e": {"value": round(job_throughput(ws, tokens, e_ms_mean), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e_ms_mean, 4), "api": e2e_api,
                "copies_alone_ms": round(copy_ms, 4),
                "copies_alone_gbs": round((h2d + d2h) / (copy_ms / 1e3) / 1e9, 1)},
        "gpu_launches": int(launches),
    }
    clocks = clk.summary()
    if clocks:
        line["clocks"] = clocks
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(inp, shape)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


# ------------------------------------------------------------------ decode step

def decode_bytes(b, H, P, S, G, dtype) -> int:
    """Algorithmic bytes of one decode step: the f32 state read and written
    once, x read and y written, B and C, dt, A and D."""
    e = elem_bytes(dtype)
    return 2 * b * H * P * S * 4 + 2 * b * H * P * e + 2 * b * G * S * e + b * H * 4 + 2 * H * 4


def run_decode(args):
    """Decode steps of a batch of sequences on their carried states: one step
    is one ssd_decode_step call (one token per sequence)."""
    import state_space_sequence_cumsum_gb300 as ssd
    from state_space_sequence_cumsum_gb300 import _lib

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    b, H, P, S, G, dtype = DECODE[args.workload]
    steps_tok = max(3, args.warmup) + 2 * args.steps + 2
    shape = Shape(b, steps_tok, H, P, S, G, 64)
    inp = make_inputs(shape, dtype=dtype, init="randn", seed=rank, init_std=0.5)
    lib = _lib.load()
    g = {k: v.to(dev) for k, v in inp.items()}
    # per-token inputs, each its own (aligned) tensor
    tok = [tuple(g[k][:, t:t + 1].contiguous() for k in ("x", "dt", "B", "C"))
           for t in range(steps_tok)]
    state = g["init"].clone()
    y = torch.empty_like(tok[0][0])
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(t):
        x, dt, Bt, Ct = tok[t]
        ssd.ssd_decode_step(x, dt, g["A"], Bt, Ct, g["D"], state, y=y)

    t_next = 0
    for _ in range(max(3, args.warmup)):
        step(t_next)
        t_next += 1
    torch.cuda.synchronize(dev)
    if ssd.ssd_stream_status() != 0:
        raise RuntimeError("kernel status during warm-up")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    launches0 = lib.ssd_launch_count()
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        clk.mark_start()
        for k in range(args.steps):
            flush.fill_(float(k))
            ev[k][0].record(stream)
            step(t_next)
            ev[k][1].record(stream)
            t_next += 1
        torch.cuda.synchronize(dev)
        clk.mark_end()
    if ws > 1:
        torch.distributed.barrier()
    launches = lib.ssd_launch_count() - launches0
    ms = statistics.mean(a.elapsed_time(c) for a, c in ev)
    ms = max_over_ranks(ms, ws, dev)
    peaks, peak_src = load_peaks()
    kb = decode_bytes(b, H, P, S, G, dtype)
    achieved = kb / (ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "kernel": "decode", "achieved": round(achieved, 1),
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                "traffic": profiled_traffic("decode", args.workload), "algorithmic_bytes": kb,
                "kernel_ms": round(ms, 5), "peak_source": peak_src}

    # e2e: the step's token inputs from pinned host memory, y back; the state
    # stays resident on the device, as it does between decode steps
    host = [tuple(v.cpu().pin_memory() for v in tok[t]) for t in range(2)]
    dev_in = tuple(torch.empty_like(v) for v in tok[0])
    y_host = torch.empty(y.shape, dtype=y.dtype).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in host[0])
    d2h = y_host.numel() * y_host.element_size()

    def e2e_step(k):
        for d, h in zip(dev_in, host[k % 2]):
            d.copy_(h, non_blocking=True)
        ssd.ssd_decode_step(dev_in[0], dev_in[1], g["A"], dev_in[2], dev_in[3], g["D"], state, y=y)
        y_host.copy_(y, non_blocking=True)

    for k in range(2):
        e2e_step(k)
    torch.cuda.synchronize(dev)
    e_ms = []
    for k in range(args.steps):
        flush.fill_(float(k))
        a, c = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        e2e_step(k)
        c.record(stream)
        c.synchronize()
        e_ms.append(a.elapsed_time(c))
    e_ms_mean = max_over_ranks(statistics.mean(e_ms), ws, dev)
    if ssd.ssd_stream_status() != 0:
        raise RuntimeError("kernel status in the timed region")
    line = {
        "metric": DECODE_METRIC, "value": round(job_throughput(ws, b, ms), 1), "unit": "tokens/s",
        "n_gpus": ws, "steps": args.steps, "warmup": max(3, args.warmup),
        "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if dtype == torch.bfloat16 else "f32",
        "data": "synthetic",
        "config": {"workload": args.workload, "batch": b, "nheads": H, "headdim": P,
                   "dstate": S, "ngroups": G, "state": "f32, updated in place",
                   "parallelism": f"replicas{ws}",
                   "l2": "flushed before every timed step (512 MB write, outside the events)"},
        "roofline": roofline,
        "e2e": {"value": round(job_throughput(ws, b, e_ms_mean), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e_ms_mean, 4)},
        "gpu_launches": int(launches),
    }
    clocks = clk.summary()
    if clocks:
        line["clocks"] = clocks
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = decode_cpu_baseline(inp)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def decode_cpu_baseline(inp, budget_s: float = 5.0):
    """The oracle as it stands on a bounded sample: one-token calls on the
    carried state of one batch row at a time, rows in turn."""
    import oracle
    oracle.build()
    threads = oracle.cpu_cores()
    nb = inp["x"].shape[0]
    t_acc, n, rows = 0.0, 0, 0
    while t_acc < budget_s:
        r = slice(rows % nb, rows % nb + 1)
        args_ = [oracle._f64(v) for v in (inp["x"][r, :1], inp["dt"][r, :1], inp["A"],
                                          inp["B"][r, :1], inp["C"][r, :1], inp["D"])]
        init = oracle._f64(inp["init"][r])
        t0 = time.perf_counter()
        oracle.fwd(*args_, 1, init=init, nthreads=threads)
        t_acc += time.perf_counter() - t0
        n += 1
        rows += 1
    return {"value": round(n / t_acc, 1), "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"float64 one-token recurrence on {n} single-row states in {t_acc:.2f} s wall"}


# ------------------------------------------------------------------ gated norm

def run_norm(args):
    """One step = one ssd_gated_rmsnorm call over every token of the workload."""
    import state_space_sequence_cumsum_gb300 as ssd
    from state_space_sequence_cumsum_gb300 import _lib

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    ntok, dim, gs, dtype = NORM[args.workload]
    gen = torch.Generator().manual_seed(rank)
    y = torch.randn((ntok, dim), generator=gen).to(dtype)
    z = torch.randn((ntok, dim), generator=gen).to(dtype)
    w = 1.0 + 0.1 * torch.randn(dim, generator=gen)
    lib = _lib.load()
    yd, zd, wd = y.to(dev), z.to(dev), w.to(dev)
    out = torch.empty_like(yd)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(max(3, args.warmup)):
        ssd.ssd_gated_rmsnorm(yd, zd, wd, group_size=gs, out=out)
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    launches0 = lib.ssd_launch_count()
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        clk.mark_start()
        for k in range(args.steps):
            flush.fill_(float(k))
            ev[k][0].record(stream)
            ssd.ssd_gated_rmsnorm(yd, zd, wd, group_size=gs, out=out)
            ev[k][1].record(stream)
        torch.cuda.synchronize(dev)
        clk.mark_end()
    launches = lib.ssd_launch_count() - launches0
    ms = statistics.mean(a.elapsed_time(c) for a, c in ev)
    ms = max_over_ranks(ms, ws, dev)
    peaks, peak_src = load_peaks()
    kb = 3 * ntok * dim * elem_bytes(dtype) + dim * 4
    achieved = kb / (ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "kernel": "gated_rmsnorm", "achieved": round(achieved, 1),
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                "traffic": profiled_traffic("gated_rmsnorm", args.workload), "algorithmic_bytes": kb,
                "kernel_ms": round(ms, 5), "peak_source": peak_src}
    hy, hz = y.pin_memory(), z.pin_memory()
    ho = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    e_ms = []
    for k in range(args.steps + 1):
        flush.fill_(float(k))
        a, c = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        yd.copy_(hy, non_blocking=True)
        zd.copy_(hz, non_blocking=True)
        ssd.ssd_gated_rmsnorm(yd, zd, wd, group_size=gs, out=out)
        ho.copy_(out, non_blocking=True)
        c.record(stream)
        c.synchronize()
        if k:
            e_ms.append(a.elapsed_time(c))
    e_ms_mean = max_over_ranks(statistics.mean(e_ms), ws, dev)
    line = {
        "metric": NORM_METRIC, "value": round(job_throughput(ws, ntok, ms), 1), "unit": "tokens/s",
        "n_gpus": ws, "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if dtype == torch.bfloat16 else "f32", "data": "synthetic",
        "config": {"workload": args.workload, "tokens": ntok, "dim": dim, "group_size": gs,
                   "parallelism": f"replicas{ws}",
                   "l2": "flushed before every timed step (512 MB write, outside the events)"},
        "roofline": roofline,
        "e2e": {"value": round(job_throughput(ws, ntok, e_ms_mean), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": 2 * ntok * dim * elem_bytes(dtype),
                "d2h_bytes_per_step": ntok * dim * elem_bytes(dtype), "ms_per_step": round(e_ms_mean, 4)},
        "gpu_launches": int(launches),
    }
    clocks = clk.summary()
    if clocks:
        line["clocks"] = clocks
    if rank == 0 and not args.no_cpu_baseline:
        import oracle
        n, t_acc = 0, 0.0
        while t_acc < 5.0 and n < ntok:
            t0 = time.perf_counter()
            oracle.gated_rmsnorm(y[n:n + 256], z[n:n + 256], w, 1e-5, gs)
            t_acc += time.perf_counter() - t0
            n += 256
        line["cpu_baseline"] = {"value": round(n / t_acc, 1), "unit": "tokens/s", "cores": 1,
                                "kind": "oracle",
                                "sample": f"numpy float64 on {n} tokens in blocks of 256, {t_acc:.2f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


# ------------------------------------------------------------------ backward pass

def bwd_compulsory_bytes(s: Shape, dtype, init: str) -> int:
    """Read x, dy, B, C, dt, A, D (and init), the final-state gradient; write
    dx, dB, dC, ddt, dA, dD and the initial-state gradient."""
    e = elem_bytes(dtype)
    blh = s.batch * s.seqlen * s.nheads
    st = s.batch * s.nheads * s.headdim * s.dstate * 4
    n = 3 * blh * s.headdim * e                                   # x, dy read; dx written
    n += 4 * s.batch * s.seqlen * s.ngroups * s.dstate * e         # B, C read; dB, dC written
    n += 2 * blh * 4 + 4 * s.nheads * 4                            # dt, ddt; A, D, dA, dD
    n += 2 * st + (st if init == "randn" else 0)                   # dfinal, dinit (, init)
    return n


def bwd_flops(s: Shape, T: int = 64) -> int:
    """Contractions per (batch, chunk of Tc tokens): per head dy x^T, the
    masked score products for dx, dB, dC (T^2 (P + 2 S)) and seven T S P
    products (the forward state pass, the reverse state pass, the state
    terms of dx, dB, dC, C h_in^T and B dS^T); per group C B^T (T^2 S)."""
    total = 0
    for c in range((s.seqlen + T - 1) // T):
        tc = min(T, s.seqlen - c * T)
        per_head = tc * tc * (2 * s.headdim + 2 * s.dstate) + 7 * tc * s.dstate * s.headdim
        total += 2 * s.batch * (s.nheads * per_head + s.ngroups * tc * tc * s.dstate)
    return total


def run_bwd(args):
    """One step = one ssd_bwd call (every stage of the backward) on the
    forward workload's inputs with random dy and dfinal."""
    import state_space_sequence_cumsum_gb300 as ssd
    from state_space_sequence_cumsum_gb300 import _lib

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    fwd_name = BACKWARD[args.workload]
    shape, dtype, init, _ = WORKLOADS[fwd_name]
    inp = make_inputs(shape, dtype=dtype, init=init, seed=rank)
    rng = np.random.default_rng(rank + 11)
    dy = torch.from_numpy(rng.standard_normal((shape.batch, shape.seqlen, shape.nheads,
                                               shape.headdim)).astype(np.float32)).to(dtype)
    dfin = torch.from_numpy(rng.standard_normal((shape.batch, shape.nheads, shape.headdim,
                                                 shape.dstate)).astype(np.float32))
    lib = _lib.load()
    g = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
    dyd, dfd = dy.to(dev), dfin.to(dev)
    wsp = ssd.Workspace()
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        return ssd.ssd_bwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], dyd,
                           initial_state=g["init"], dfinal=dfd, workspace=wsp)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    if ssd.ssd_stream_status() != 0:
        raise RuntimeError("kernel status during warm-up")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    launches0 = lib.ssd_launch_count()
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        clk.mark_start()
        for k in range(args.steps):
            flush.fill_(float(k))
            ev[k][0].record(stream)
            step()
            ev[k][1].record(stream)
        torch.cuda.synchronize(dev)
        clk.mark_end()
    launches = lib.ssd_launch_count() - launches0
    ms = statistics.mean(a.elapsed_time(c) for a, c in ev)
    ms = max_over_ranks(ms, ws, dev)
    peaks, peak_src = load_peaks()
    cb = bwd_compulsory_bytes(shape, dtype, init)
    fl = bwd_flops(shape)
    t_bytes = cb / (peaks["hbm_gbs"] * 1e9)
    t_flops = fl / (peaks["bf16_tflops"] * 1e12)
    bound = "hbm" if t_bytes >= t_flops else "tensor"
    t_roof = max(t_bytes, t_flops)
    roofline = ({"bound": "hbm", "achieved": round(cb / (ms / 1e3) / 1e9, 1), "peak": peaks["hbm_gbs"],
                 "unit": "GB/s"} if bound == "hbm" else
                {"bound": "tensor", "achieved": round(fl / (ms / 1e3) / 1e12, 2),
                 "peak": peaks["bf16_tflops"], "unit": "TFLOP/s"})
    roofline.update({"frac": round(t_roof / (ms / 1e3), 4), "traffic": None, "kernel": "ssd_bwd (whole call)",
                     "algorithmic_bytes": cb, "algorithmic_flops": fl, "peak_source": peak_src})

    # e2e: the step's inputs (x, dt, B, C, dy, dfinal and init) from pinned host
    # memory, every gradient back
    host = {"x": inp["x"], "dt": inp["dt"], "B": inp["B"], "C": inp["C"], "dy": dy, "df": dfin}
    if inp["init"] is not None:
        host["init"] = inp["init"]
    host = {k: v.pin_memory() for k, v in host.items()}
    dev_in = {k: torch.empty_like(v, device=dev) for k, v in host.items()}
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    res = step()
    outs_host = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in res.items()
                 if v is not None}
    d2h = sum(v.numel() * v.element_size() for v in outs_host.values())

    def e2e_step():
        for k, v in host.items():
            dev_in[k].copy_(v, non_blocking=True)
        r = ssd.ssd_bwd(dev_in["x"], dev_in["dt"], g["A"], dev_in["B"], dev_in["C"], g["D"],
                        dev_in["dy"], initial_state=dev_in.get("init"), dfinal=dev_in["df"],
                        workspace=wsp)
        for k, v in outs_host.items():
            v.copy_(r[k], non_blocking=True)

    e2e_step()
    torch.cuda.synchronize(dev)
    e_ms = []
    for k in range(args.steps):
        flush.fill_(float(k))
        a, c = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        e2e_step()
        c.record(stream)
        c.synchronize()
        e_ms.append(a.elapsed_time(c))
    e_ms_mean = max_over_ranks(statistics.mean(e_ms), ws, dev)
    if ssd.ssd_stream_status() != 0:
        raise RuntimeError("kernel status in the timed region")
    tokens = shape.tokens
    line = {
        "metric": BWD_METRIC, "value": round(job_throughput(ws, tokens, ms), 1), "unit": "tokens/s",
        "n_gpus": ws, "steps": args.steps, "warmup": max(3, args.warmup),
        "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if dtype == torch.bfloat16 else "f32",
        "data": "synthetic",
        "config": {"workload": args.workload, "forward": fwd_name, "batch": shape.batch,
                   "seqlen": shape.seqlen, "nheads": shape.nheads, "headdim": shape.headdim,
                   "dstate": shape.dstate, "ngroups": shape.ngroups, "chunk_size": 64,
                   "parallelism": f"replicas{ws}",
                   "l2": "flushed before every timed step (512 MB write, outside the events)"},
        "roofline": roofline,
        "e2e": {"value": round(job_throughput(ws, tokens, e_ms_mean), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e_ms_mean, 4)},
        "gpu_launches": int(launches),
    }
    clocks = clk.summary()
    if clocks:
        line["clocks"] = clocks
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = bwd_cpu_baseline(inp, dy, dfin, shape)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def bwd_cpu_baseline(inp, dy, dfin, s: Shape, budget_s: float = 10.0):
    """The oracle's adjoint as it stands, on a bounded sample: one batch row
    (every head) over a prefix of the sequence, prefixes doubled until about
    budget_s of wall time is reached."""
    import oracle
    oracle.build()
    threads = oracle.cpu_cores()
    Lp, t_acc, tok = 256, 0.0, 0
    while t_acc < budget_s and Lp <= s.seqlen:
        sl = (slice(0, 1), slice(0, Lp))
        t0 = time.perf_counter()
        oracle.bwd(inp["x"][sl], inp["dt"][sl], inp["A"], inp["B"][sl], inp["C"][sl], inp["D"],
                   dy[sl], init=None if inp["init"] is None else inp["init"][:1],
                   dfinal=dfin[:1], nthreads=threads)
        t_acc += time.perf_counter() - t0
        tok += Lp
        Lp *= 2
    return {"value": round(tok / t_acc, 1), "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": (f"float64 adjoint recurrence, batch row 0 (all {s.nheads} heads), sequence "
                       f"prefixes of 256, 512, ... tokens: {tok} tokens in {t_acc:.2f} s wall")}


# ------------------------------------------------------------------ reference arm

def run_reference(args):
    """The oracle as it stands, on the host cores, on a bounded sample per step."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    shape, dtype, init, want_states = WORKLOADS[args.workload]
    inp = make_inputs(shape, dtype=dtype, init=init, seed=0)
    threads = oracle.cpu_cores()
    for k in range(max(1, args.warmup)):
        oracle_row(inp, shape, k % shape.batch, threads)
    times, toks = [], 0
    for k in range(args.steps):
        t, n = oracle_row(inp, shape, k % shape.batch, threads)
        times.append(t)
        toks = n
    sec = statistics.mean(times)
    value = toks / sec
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": "tokens/s",
        "n_gpus": ws, "steps": args.steps, "warmup": max(1, args.warmup),
        "ms_per_step": round(sec * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "batch": shape.batch, "seqlen": shape.seqlen,
                   "nheads": shape.nheads, "headdim": shape.headdim, "dstate": shape.dstate,
                   "ngroups": shape.ngroups, "chunk_size": shape.chunk_size},
        "cpu_baseline": {"value": round(value, 1), "unit": "tokens/s", "cores": threads,
                         "kind": "oracle",
                         "sample": (f"each step: float64 recurrence over one batch row of the "
                                    f"workload (all {shape.nheads} heads x {shape.seqlen} "
                                    f"tokens = {toks} tokens), rows taken in turn")},
        "e2e": {"value": round(value, 1), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_decode_reference(args):
    """Reference arm of a decode workload: the oracle on the host cores, one
    single-row one-token call per step."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    b, H, P, S, G, dtype = DECODE[args.workload]
    inp = make_inputs(Shape(b, 1, H, P, S, G, 64), dtype=dtype, init="randn", seed=0,
                      init_std=0.5)
    cb = decode_cpu_baseline(inp, budget_s=max(1.0, 0.05 * args.steps))
    line = {
        "impl": "reference", "metric": DECODE_METRIC, "value": cb["value"], "unit": "tokens/s",
        "n_gpus": ws, "steps": args.steps, "warmup": max(1, args.warmup),
        "ms_per_step": round(1e3 / cb["value"], 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "batch": b, "nheads": H, "headdim": P,
                   "dstate": S, "ngroups": G},
        "cpu_baseline": cb,
        "e2e": {"value": cb["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_bwd_reference(args):
    """Reference arm of a backward workload: the oracle's adjoint on the host
    cores, a bounded sample per step."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    shape, dtype, init, _ = WORKLOADS[BACKWARD[args.workload]]
    inp = make_inputs(shape, dtype=dtype, init=init, seed=0)
    rng = np.random.default_rng(11)
    dy = torch.from_numpy(rng.standard_normal((shape.batch, shape.seqlen, shape.nheads,
                                               shape.headdim)).astype(np.float32)).to(dtype)
    dfin = torch.from_numpy(rng.standard_normal((shape.batch, shape.nheads, shape.headdim,
                                                 shape.dstate)).astype(np.float32))
    cb = bwd_cpu_baseline(inp, dy, dfin, shape, budget_s=max(2.0, 0.5 * args.steps))
    line = {
        "impl": "reference", "metric": BWD_METRIC, "value": cb["value"], "unit": "tokens/s",
        "n_gpus": ws, "steps": args.steps, "warmup": max(1, args.warmup),
        "ms_per_step": round(1e3 * shape.tokens / cb["value"], 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "forward": BACKWARD[args.workload]},
        "cpu_baseline": cb,
        "e2e": {"value": cb["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def spawn_ranks(n: int) -> int:
    """--gpus N outside torchrun: relaunch this command as N ranks of one node
    (one per GPU) under torch.distributed.run, rendezvous on 127.0.0.1."""
    if torch.cuda.device_count() < n:
        print(f"bench.py: --gpus {n} but only {torch.cuda.device_count()} GPU(s) visible",
              file=sys.stderr)
        return 2
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={n}", "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.abspath(__file__), *sys.argv[1:]]
    return subprocess.call(cmd)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT,
                    choices=sorted(WORKLOADS) + sorted(DECODE) + sorted(BACKWARD) + sorted(NORM))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if args.gpus < 1:
        ap.error("--gpus must be at least 1")
    if args.gpus != ws:
        if ws == 1 and "LOCAL_RANK" not in os.environ:
            sys.exit(spawn_ranks(args.gpus))
        print(f"bench.py: --gpus {args.gpus} but WORLD_SIZE is {ws}", file=sys.stderr)
        sys.exit(2)
    if args.workload in NORM:
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the gated norm's reference arm is "
                              "the oracle sample reported as cpu_baseline on our arm's line"}))
        else:
            run_norm(args)
    elif args.workload in BACKWARD:
        if args.impl == "reference":
            run_bwd_reference(args)
        else:
            run_bwd(args)
    elif args.workload in DECODE:
        if args.impl == "reference":
            run_decode_reference(args)
        else:
            run_decode(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
