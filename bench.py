#!/usr/bin/env python
"""Throughput of the memory-bound MoE glue path on GB300.

One step = one pass of the whole path over one batch of synthetic input:
moe_route (softmax, top-k, histogram/scan, permutation) -> moe_expand ->
moe_swiglu -> moe_combine, all through the C ABI. The headline workload is
the largest layer, the prefill batch: T=8192 tokens, H=4096, E=8 experts,
top-2 (renormalised), I=14336 (1.81 GB of algorithmic traffic per step).
Inputs are seeded and synthetic (memory_bound_moe_gb300.workloads); the
expert GEMMs are not part of the path, so their outputs (gate_up,
expert_out) are inputs here.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload prefill|mid|skewed|decode|tiny]

Prints one JSON line (rank 0). Timing: CUDA events on the launching stream
around K back-to-back steps (one prefill step streams 1.81 GB, inputs
1.14 GB, through the 129 MB L2, so inputs come from HBM every step; no flush
writes, whose dirty lines would be written back inside the next step), plus
events between the four calls for the per-kernel split; device-resident
`value` and an end-to-end `e2e` measured through the public Python binding
with pinned host buffers and the host<->device copies inside the timed
region. The other workloads (mid, skewed, decode, tiny) are timed the same
way and reported under `workloads`. With N > 1 (torchrun) every rank runs
its own replica on its own batch (weak scaling, no collective on the data
path); the step time is the max over ranks. `--impl reference` times the CPU
oracle (plain C) on the host cores on bounded samples of the same workload.
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

WORKLOAD = "prefill"
SIDE_WORKLOADS = ("mid", "skewed", "decode", "tiny")
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20
KERNELS = ("route", "expand", "swiglu", "combine")
METRIC = "tokens/s and achieved HBM GB/s (% of peak) for route+expand+SwiGLU+combine"


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD, help="workload name (default: prefill)")
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of oracle CPU work for the cpu_baseline leg (0 = skip)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the decode-latency and wider-entry-point measurements")
    ap.add_argument("--extra-reps", type=int, default=0,
                    help="repetitions per case in those measurements (0: 2000 decode, 240 others)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# accounting
# ---------------------------------------------------------------------------

def algorithmic_bytes(w) -> dict:
    """Minimum unique HBM traffic per launch of each kernel: every input byte
    read once, every output byte written once."""
    T, H, E, k, I, S = w.T, w.H, w.E, w.k, w.I, w.S
    return {
        "route": 4 * T * E + 16 * S + 4 * E + 4 * (E + 1),  # logits; ids, weights, perm, inv_perm; counts, offsets
        "expand": 2 * T * H + 2 * S * H + 4 * S,             # x once; S rows; inv_perm
        "swiglu": 6 * S * I,                                 # gate_up (4SI) + act (2SI)
        "combine": 2 * S * H + 8 * S + 2 * T * H,            # expert rows; weights + inv_perm; out
    }


def peak_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            v = float(json.load(fh)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


KERNEL_SOURCES = {
    "route": ["route.cu", "route_device.cuh", "rows_common.cuh"],
    "expand": ["expand.cu", "rows_common.cuh"],
    "swiglu": ["swiglu.cu", "rows_common.cuh"],
    "combine": ["combine.cu", "rows_common.cuh"],
}


def kernel_source_sha(kernel: str) -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "memory_bound_moe_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel] + ["moe_device.cuh"]:
        with open(os.path.join(csrc, name), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_from_profiles(kernel: str, workload: str):
    """DRAM bytes per launch (read + write) from the committed ncu summary
    ``profiles/dram_traffic.txt``, if it was taken on the current source of
    that kernel; else None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    sha = kernel_source_sha(kernel)
    with open(path) as fh:
        for line in fh:
            parts = line.split("#", 1)[0].split()
            if len(parts) >= 4 and parts[0] == kernel and parts[1] == workload and parts[3] == sha:
                return int(float(parts[2]))
    return None


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, uuid: str):
        self.uuid = uuid.lower()
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            if self.uuid and self.uuid not in f[0].lower():
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for name, val in zip(self.NAMES, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "reasons": sorted(reasons), "samples": len(sm)}


BAD_REASONS = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}


# ---------------------------------------------------------------------------
# the device-resident step
# ---------------------------------------------------------------------------

class Step:
    """All buffers of one batch resident in HBM plus the raw C-ABI argument
    tuples, so a step is four direct library calls on one stream."""

    def __init__(self, w, inputs, dev):
        import torch
        import memory_bound_moe_gb300 as moe
        self.torch = torch
        self.lib = moe.load_library()
        self.w = w
        T, H, E, k, I, S = w.T, w.H, w.E, w.k, w.I, w.S
        self.logits = inputs["logits"].to(dev)
        self.x = inputs["x"].to(dev)
        self.gate_up = inputs["gate_up"].to(dev)
        self.expert_out = inputs["expert_out"].to(dev)
        i32 = dict(dtype=torch.int32, device=dev)
        self.topk_ids = torch.empty((T, k), **i32)
        self.topk_weights = torch.empty((T, k), dtype=torch.float32, device=dev)
        self.counts = torch.empty((E,), **i32)
        self.offsets = torch.empty((E + 1,), **i32)
        self.perm = torch.empty((S,), **i32)
        self.inv_perm = torch.empty((S,), **i32)
        self.ws_bytes = moe.moe_route_workspace_size(T, E, k)
        self.ws = torch.empty((max(self.ws_bytes, 16),), dtype=torch.uint8, device=dev)
        self.expanded = torch.empty((S, H), dtype=torch.bfloat16, device=dev)
        self.act = torch.empty((S, I), dtype=torch.bfloat16, device=dev)
        self.out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        self.route_args = (self.logits.data_ptr(), T, E, k, int(w.renorm), self.topk_ids.data_ptr(),
                           self.topk_weights.data_ptr(), self.counts.data_ptr(), self.offsets.data_ptr(),
                           self.perm.data_ptr(), self.inv_perm.data_ptr(), self.ws.data_ptr(),
                           self.ws.numel())
        self.expand_args = (self.x.data_ptr(), T, H, k, self.inv_perm.data_ptr(), self.expanded.data_ptr())
        self.swiglu_args = (self.gate_up.data_ptr(), S, I, self.act.data_ptr())
        self.combine_args = (self.expert_out.data_ptr(), T, H, k, self.topk_weights.data_ptr(),
                             self.inv_perm.data_ptr(), self.out.data_ptr())
        # our kernel launches per step: route is one block-level kernel for
        # small batches and two kernels otherwise; the row kernels one each
        self.launches_per_step = (2 if self.ws_bytes > 0 else 1) + 3

    def run(self, stream_ptr, events=None):
        lib = self.lib
        if events is not None:
            events[0].record()
        st = lib.moe_route(*self.route_args, stream_ptr)
        if events is not None:
            events[1].record()
        st |= lib.moe_expand(*self.expand_args, stream_ptr)
        if events is not None:
            events[2].record()
        st |= lib.moe_swiglu(*self.swiglu_args, stream_ptr)
        if events is not None:
            events[3].record()
        st |= lib.moe_combine(*self.combine_args, stream_ptr)
        if events is not None:
            events[4].record()
        if st != 0:
            raise RuntimeError(f"C-ABI call failed with status {st}")


def _run_ahead(scratch):
    """~2 ms of unrelated GPU work (a write then a read of buffers larger than
    L2, leaving it clean) so the host enqueues ahead of the GPU and no step
    waits on the host."""
    for _ in range(4):
        scratch[0].zero_()
        scratch[1].sum()


def time_device_resident(step, steps, warmup, dev, scratch):
    """K back-to-back steps on one stream; the step time is the elapsed time
    between events before the first and after the last step, divided by K.
    Nothing is recorded between the calls, so consecutive kernels overlap
    their launch as they do in use (programmatic dependent launch)."""
    torch = step.torch
    sp = torch.cuda.current_stream(dev).cuda_stream
    for _ in range(warmup):
        step.run(sp)
    torch.cuda.synchronize(dev)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    _run_ahead(scratch)
    start.record()
    for _ in range(steps):
        step.run(sp)
    end.record()
    torch.cuda.synchronize(dev)
    barrier()
    return start.elapsed_time(end) / steps, time.perf_counter() - t0


def time_per_kernel(step, steps, dev, scratch):
    """The same steps with an event between the calls: the per-kernel split
    (each event boundary also stops the next launch from overlapping)."""
    torch = step.torch
    sp = torch.cuda.current_stream(dev).cuda_stream
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
    torch.cuda.synchronize(dev)
    _run_ahead(scratch)
    for i in range(steps):
        step.run(sp, evs[i])
    torch.cuda.synchronize(dev)
    per_kernel = {name: [] for name in KERNELS}
    for e in evs:
        for j, name in enumerate(KERNELS):
            per_kernel[name].append(e[j].elapsed_time(e[j + 1]))
    return per_kernel


def time_e2e(w, inputs, steps, warmup, dev, n_copy_streams=4, chunk_bytes=32 << 20):
    """The same step through the public binding, end to end from host memory:
    every step copies its four inputs from pinned host buffers (split into
    ~32 MB chunks over several copy streams, so several copy engines run at
    once) into one of two device buffer sets, runs the four calls on the
    compute stream once its copies have landed, and copies the combined
    output back to pinned host memory on a third stream. Copies for step
    i + 1 overlap the compute of step i (double buffering)."""
    import torch
    import memory_bound_moe_gb300 as moe
    names = ("logits", "x", "gate_up", "expert_out")
    host = {kk: inputs[kk].pin_memory() for kk in names}
    T, E, k, S = w.T, w.E, w.k, w.S
    i32 = dict(dtype=torch.int32, device=dev)
    sets = []
    for _ in range(2):
        d = {kk: torch.empty_like(host[kk], device=dev) for kk in names}
        d["r"] = moe.RouteResult(torch.empty((T, k), **i32),
                                 torch.empty((T, k), dtype=torch.float32, device=dev),
                                 torch.empty((E,), **i32), torch.empty((E + 1,), **i32),
                                 torch.empty((S,), **i32), torch.empty((S,), **i32))
        d["ws"] = torch.empty((max(moe.moe_route_workspace_size(T, E, k), 16),), dtype=torch.uint8, device=dev)
        d["ex"] = torch.empty((S, w.H), dtype=torch.bfloat16, device=dev)
        d["act"] = torch.empty((S, w.I), dtype=torch.bfloat16, device=dev)
        d["out"] = torch.empty((T, w.H), dtype=torch.bfloat16, device=dev)
        d["consumed"] = torch.cuda.Event()   # compute done with this set's inputs
        d["drained"] = torch.cuda.Event()    # its output copied back to the host
        sets.append(d)
    out_host = [torch.empty((T, w.H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    compute = torch.cuda.current_stream(dev)
    copiers = [torch.cuda.Stream(dev) for _ in range(n_copy_streams)]
    d2h = torch.cuda.Stream(dev)
    chunks = []   # (name, start, stop) over the flattened byte views
    for kk in names:
        nbytes = host[kk].numel() * host[kk].element_size()
        for a in range(0, nbytes, chunk_bytes):
            chunks.append((kk, a, min(nbytes, a + chunk_bytes)))
    hbytes = {kk: host[kk].view(-1).view(torch.uint8) for kk in names}
    dbytes = [{kk: d[kk].view(-1).view(torch.uint8) for kk in names} for d in sets]

    def issue_copies(i):
        d = sets[i % 2]
        evs = []
        for ci, cs in enumerate(copiers):
            cs.wait_event(d["consumed"])
            with torch.cuda.stream(cs):
                for kk, a, b in chunks[ci::n_copy_streams]:
                    dbytes[i % 2][kk][a:b].copy_(hbytes[kk][a:b], non_blocking=True)
                e = torch.cuda.Event()
                e.record(cs)
                evs.append(e)
        return evs

    def issue_compute(i, evs):
        d = sets[i % 2]
        for e in evs:
            compute.wait_event(e)
        compute.wait_event(d["drained"])     # do not overwrite out before it is copied back
        r = moe.moe_route(d["logits"], k, w.renorm, out=d["r"], workspace=d["ws"])
        moe.moe_expand(d["x"], r.inv_perm, k, out=d["ex"])
        moe.moe_swiglu(d["gate_up"], out=d["act"])
        moe.moe_combine(d["expert_out"], r.topk_weights, r.inv_perm, out=d["out"])
        d["consumed"].record(compute)
        d2h.wait_event(d["consumed"])
        with torch.cuda.stream(d2h):
            out_host[i % 2].copy_(d["out"], non_blocking=True)
        d["drained"].record(d2h)

    def run(n):
        pending = issue_copies(0)
        for i in range(n):
            nxt = issue_copies(i + 1) if i + 1 < n else None
            issue_compute(i, pending)
            pending = nxt

    run(warmup)
    torch.cuda.synchronize(dev)
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(compute)
    for cs in copiers + [d2h]:
        cs.wait_event(e0)
    run(steps)
    for cs in copiers + [d2h]:
        ev = torch.cuda.Event()
        ev.record(cs)
        compute.wait_event(ev)
    e1.record(compute)
    torch.cuda.synchronize(dev)
    barrier()
    ms = e0.elapsed_time(e1) / steps
    h2d = sum(host[kk].numel() * host[kk].element_size() for kk in names)
    d2h_bytes = out_host[0].numel() * out_host[0].element_size()
    return ms, h2d, d2h_bytes


def decode_latency(dev, reps=2000, layers=16):
    """Latency of one MoE-layer pass on the decode workload (T=16, H=7168,
    E=256, top-8, I=2048): the four calls (route, expand, SwiGLU, combine)
    and the three calls with routing and expansion in one launch
    (moe_route_expand), each issued back to back through direct C-ABI calls,
    and replayed from CUDA graphs: one graph holding `layers` consecutive
    layer passes (as a decode step's graph holds every layer of the model),
    and, for comparison, a graph of a single pass replayed back to back
    (every replay then starts with a full kernel boundary: programmatic
    launch overlap does not cross graph launches). Per-layer time = elapsed
    time / layer passes."""
    import torch
    import memory_bound_moe_gb300 as moe
    from memory_bound_moe_gb300.workloads import WORKLOADS, generate
    lib = moe.load_library()
    w = WORKLOADS["decode"]
    inp = {kk: v.to(dev) for kk, v in generate(w, seed=0).items()}
    T, E, k, S, H, I = w.T, w.E, w.k, w.S, w.H, w.I
    i32 = dict(dtype=torch.int32, device=dev)
    ids = torch.empty((T, k), **i32)
    wts = torch.empty((T, k), dtype=torch.float32, device=dev)
    cnt = torch.empty((E,), **i32)
    off = torch.empty((E + 1,), **i32)
    perm = torch.empty((S,), **i32)
    inv = torch.empty((S,), **i32)
    ex = torch.empty((S, H), dtype=torch.bfloat16, device=dev)
    act = torch.empty((S, I), dtype=torch.bfloat16, device=dev)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    p = lambda t: t.data_ptr()
    rn = int(w.renorm)

    def four(sp):
        st = lib.moe_route(p(inp["logits"]), T, E, k, rn, p(ids), p(wts), p(cnt), p(off), p(perm),
                           p(inv), 0, 0, sp)
        st |= lib.moe_expand(p(inp["x"]), T, H, k, p(inv), p(ex), sp)
        st |= lib.moe_swiglu(p(inp["gate_up"]), S, I, p(act), sp)
        st |= lib.moe_combine(p(inp["expert_out"]), T, H, k, p(wts), p(inv), p(out), sp)
        assert st == 0

    def three(sp):
        st = lib.moe_route_expand(p(inp["logits"]), T, E, k, rn, p(inp["x"]), H, p(ids), p(wts),
                                  p(cnt), p(off), p(perm), p(inv), p(ex), 0, 0, sp)
        st |= lib.moe_swiglu(p(inp["gate_up"]), S, I, p(act), sp)
        st |= lib.moe_combine(p(inp["expert_out"]), T, H, k, p(wts), p(inv), p(out), sp)
        assert st == 0

    def timed(fn, passes=1, n=reps):
        sp = torch.cuda.current_stream(dev).cuda_stream
        for _ in range(20):
            fn(sp)
        torch.cuda.synchronize(dev)
        torch.cuda._sleep(8_000_000)     # let the host enqueue ahead of the GPU
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(n):
            fn(sp)
        b.record()
        torch.cuda.synchronize(dev)
        return 1e3 * a.elapsed_time(b) / (n * passes)

    def graphed(fn, passes):
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            fn(side.cuda_stream)
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(passes):
                fn(torch.cuda.current_stream(dev).cuda_stream)
        return lambda sp: g.replay()

    n_graph = max(1, reps // layers)
    res = {"four_calls_stream_us": timed(four), "route_expand_stream_us": timed(three),
           "four_calls_graph_us": timed(graphed(four, layers), layers, n_graph),
           "route_expand_graph_us": timed(graphed(three, layers), layers, n_graph),
           "four_calls_graph_1layer_us": timed(graphed(four, 1)),
           "route_expand_graph_1layer_us": timed(graphed(three, 1)),
           "graph_layers": layers, "workload": w.describe()}
    return {kk: (round(v, 3) if isinstance(v, float) else v) for kk, v in res.items()}


def extras_measurement(dev, reps=240, n_sets=3):
    """The wider entry points on the mid workload (T=4096, H=2048, E=128,
    top-8, I=768), each launched back to back over three sets of inputs AND
    outputs (each set larger than half of L2, so every launch reads from and
    writes back to HBM): MXFP8 SwiGLU and expand against their bfloat16
    versions, NVFP4 (tensor scale 64) and MXFP4 SwiGLU and expand, and the
    bfloat16 combine; one tensor-parallel rank's local routing (experts [0, 32) of
    128, segments padded to 128 rows) with its padded expand and partial
    combine; and the QK RMSNorm of a Qwen3-30B-A3B-like attention layer
    (T=8192, 32 q heads, 4 k heads, head_dim 128, in place). GB/s =
    algorithmic bytes / time."""
    import torch
    import memory_bound_moe_gb300 as moe
    from memory_bound_moe_gb300.workloads import WORKLOADS, generate
    lib = moe.load_library()
    w = WORKLOADS["mid"]
    T, H, E, k, I, S = w.T, w.H, w.E, w.k, w.I, w.S
    peak, _ = peak_hbm()
    sp = torch.cuda.current_stream(dev).cuda_stream
    p = lambda t: t.data_ptr()
    u8 = dict(dtype=torch.uint8, device=dev)
    bf = dict(dtype=torch.bfloat16, device=dev)
    e0, e1, pad = 0, 32, 128
    rows = moe.moe_route_local_rows(T, k, e0, e1, pad)
    ws = torch.empty((max(moe.moe_route_local_workspace_size(T, E, k, e0, e1), 16),), **u8)
    sets = []
    for seed in range(n_sets):
        d = {kk: v.to(dev) for kk, v in generate(w, seed=seed).items()}
        d["r"] = moe.moe_route(d["logits"], k, True)
        d["act"] = torch.empty((S, I), **bf)
        d["act_c"], d["act_s"] = torch.empty((S, I), **u8), torch.empty((S, I // 32), **u8)
        d["ex"] = torch.empty((S, H), **bf)
        d["ex_c"], d["ex_s"] = torch.empty((S, H), **u8), torch.empty((S, H // 32), **u8)
        d["act4"], d["ex4"] = torch.empty((S, I // 2), **u8), torch.empty((S, H // 2), **u8)
        d["act4_s"], d["ex4_s"] = torch.empty((S, I // 16), **u8), torch.empty((S, H // 16), **u8)
        d["loc"] = moe.moe_route_local(d["logits"], k, True, e0, e1, pad)
        d["lex"] = torch.empty((rows, H), **bf)
        d["leo"] = torch.randn((rows, H), device=dev).to(torch.bfloat16)
        d["out"] = torch.empty((T, H), **bf)
        sets.append(d)
    qT, nq, nk, hd = 8192, 32, 4, 128
    qk = [(torch.randn((qT, nq, hd), device=dev).to(torch.bfloat16),
           torch.randn((qT, nk, hd), device=dev).to(torch.bfloat16)) for _ in range(n_sets)]
    qkw = (torch.randn(hd, device=dev).to(torch.bfloat16), torch.randn(hd, device=dev).to(torch.bfloat16))

    def timed(fns):
        for f in fns:
            assert f() == 0
        torch.cuda.synchronize(dev)
        torch.cuda._sleep(4_000_000)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        for r in range(reps):
            assert fns[r % len(fns)]() == 0
        b.record()
        torch.cuda.synchronize(dev)
        return 1e3 * a.elapsed_time(b) / reps

    n_loc = int(sum(int(d["loc"].expert_counts.sum()) for d in sets) / n_sets)   # local slots per batch
    cases = {
        "swiglu_bf16": ([lambda d=d: lib.moe_swiglu(p(d["gate_up"]), S, I, p(d["act"]), sp) for d in sets],
                        6 * S * I),
        "swiglu_mxfp8": ([lambda d=d: lib.moe_swiglu_mxfp8(p(d["gate_up"]), S, I, p(d["act_c"]), p(d["act_s"]),
                                                           sp) for d in sets],
                         4 * S * I + S * I + S * I // 32),
        "expand_bf16": ([lambda d=d: lib.moe_expand(p(d["x"]), T, H, k, p(d["r"].inv_perm), p(d["ex"]), sp)
                         for d in sets], 2 * T * H + 2 * S * H + 4 * S),
        "combine_bf16": ([lambda d=d: lib.moe_combine(p(d["expert_out"]), T, H, k, p(d["r"].topk_weights),
                                                      p(d["r"].inv_perm), p(d["out"]), sp) for d in sets],
                         2 * S * H + 8 * S + 2 * T * H),
        "expand_mxfp8": ([lambda d=d: lib.moe_expand_mxfp8(p(d["x"]), T, H, k, p(d["r"].inv_perm), S,
                                                           p(d["ex_c"]), p(d["ex_s"]), sp) for d in sets],
                         2 * T * H + S * H + S * H // 32 + 4 * S),
        "swiglu_nvfp4": ([lambda d=d: lib.moe_swiglu_fp4(p(d["gate_up"]), S, I, 0, 64.0, p(d["act4"]),
                                                        p(d["act4_s"]), sp) for d in sets],
                         4 * S * I + S * I // 2 + S * I // 16),
        "swiglu_mxfp4": ([lambda d=d: lib.moe_swiglu_fp4(p(d["gate_up"]), S, I, 1, 0.0, p(d["act4"]),
                                                        p(d["act4_s"]), sp) for d in sets],
                         4 * S * I + S * I // 2 + S * I // 32),
        "expand_nvfp4": ([lambda d=d: lib.moe_expand_fp4(p(d["x"]), T, H, k, p(d["r"].inv_perm), S, 0, 64.0,
                                                        p(d["ex4"]), p(d["ex4_s"]), sp) for d in sets],
                         2 * T * H + S * H // 2 + S * H // 16 + 4 * S),
        "expand_mxfp4": ([lambda d=d: lib.moe_expand_fp4(p(d["x"]), T, H, k, p(d["r"].inv_perm), S, 1, 0.0,
                                                        p(d["ex4"]), p(d["ex4_s"]), sp) for d in sets],
                         2 * T * H + S * H // 2 + S * H // 32 + 4 * S),
        "route_local_rank0of4": ([lambda d=d: lib.moe_route_local(
            p(d["logits"]), T, E, k, 1, e0, e1, pad, p(d["loc"].topk_ids), p(d["loc"].topk_weights),
            p(d["loc"].expert_counts), p(d["loc"].expert_offsets), p(d["loc"].perm), p(d["loc"].inv_perm),
            p(ws), ws.numel(), sp) for d in sets], 4 * T * E + 12 * S + 4 * rows),
        "expand_rows_rank0of4": ([lambda d=d: lib.moe_expand_rows(p(d["x"]), T, H, k, p(d["loc"].inv_perm), rows,
                                                                    p(d["lex"]), sp) for d in sets],
                                 2 * T * H + 2 * n_loc * H + 4 * S),
        "combine_rows_rank0of4": ([lambda d=d: lib.moe_combine_rows(p(d["leo"]), rows, T, H, k,
                                                                      p(d["loc"].topk_weights), p(d["loc"].inv_perm),
                                                                      p(d["out"]), sp) for d in sets],
                                  2 * n_loc * H + 8 * S + 2 * T * H),
        "qk_rmsnorm_qwen3": ([lambda q=q, kk=kk: lib.moe_qk_rmsnorm(p(q), p(kk), qT, nq, nk, hd, p(qkw[0]),
                                                                       p(qkw[1]), 1.0, 1e-6, sp)
                              for q, kk in qk], 2 * 2 * qT * (nq + nk) * hd),
    }
    res = {"workload": w.describe(), "local_rank": f"experts [{e0},{e1}) of {E}, pad {pad}, {n_loc} local slots",
           "qk_rmsnorm": f"T={qT} q_heads={nq} k_heads={nk} head_dim={hd}, in place",
           "timing": f"{reps} back-to-back launches over {n_sets} sets of inputs and outputs"}
    for name, (fns, nbytes) in cases.items():
        us = timed(fns)
        gbs = nbytes / (us * 1e-6) / 1e9
        res[name] = {"us": round(us, 3), "GBps": round(gbs, 1), "frac": round(gbs / peak, 4)}
    return res


# ---------------------------------------------------------------------------
# the CPU oracle (baseline and reference arm)
# ---------------------------------------------------------------------------

def _oracle_batches(w, inputs, n_tokens, parts):
    """The first n_tokens tokens of the batch cut into `parts` contiguous
    token ranges, each an independent sub-batch (its logits and x rows and
    its k slots' rows of gate_up / expert_out) as C-contiguous numpy arrays."""
    import numpy as np
    from memory_bound_moe_gb300.workloads import as_u16
    n = max(1, min(n_tokens, w.T))
    parts = max(1, min(parts, n))
    logits = inputs["logits"].numpy()
    x, gu, eo = as_u16(inputs["x"]), as_u16(inputs["gate_up"]), as_u16(inputs["expert_out"])
    cuts = [n * i // parts for i in range(parts + 1)]
    out = []
    for a, b in zip(cuts[:-1], cuts[1:]):
        out.append((np.ascontiguousarray(logits[a:b]), np.ascontiguousarray(x[a:b]),
                    np.ascontiguousarray(gu[a * w.k:b * w.k]), np.ascontiguousarray(eo[a * w.k:b * w.k])))
    return n, out


def oracle_steps(w, batch):
    """The oracle's four steps on one sub-batch, each timed on its own;
    returns {step: seconds}."""
    from oracle import oracle
    logits, x, gu, eo = batch
    t = {}
    t0 = time.perf_counter()
    r = oracle.route(logits, w.k, w.renorm)
    t1 = time.perf_counter()
    oracle.expand(x, w.k, r["perm"])
    t2 = time.perf_counter()
    oracle.swiglu(gu)
    t3 = time.perf_counter()
    oracle.combine(eo, r["topk_weights"], r["inv_perm"])
    t4 = time.perf_counter()
    t["route"], t["expand"], t["swiglu"], t["combine"] = t1 - t0, t2 - t1, t3 - t2, t4 - t3
    return t


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover - non-Linux
        return os.cpu_count() or 1


def oracle_pass(w, batches, threads):
    """One pass of the oracle over the sub-batches, `threads` at a time
    (the C oracle runs outside the interpreter lock, so threads run it in
    parallel). Returns (seconds, summed per-step seconds)."""
    import concurrent.futures as cf
    t0 = time.perf_counter()
    if threads == 1:
        per = [oracle_steps(w, b) for b in batches]
    else:
        with cf.ThreadPoolExecutor(max_workers=threads) as ex:
            per = list(ex.map(lambda b: oracle_steps(w, b), batches))
    dt = time.perf_counter() - t0
    return dt, {s: sum(p[s] for p in per) for s in KERNELS}


def cpu_baseline(w, inputs, budget_s):
    """The unchanged oracle on this machine's host cores: single-threaded, then
    one thread per core over independent token sub-batches, each for about
    half of `budget_s`. Reports tokens/s for both and the per-step split."""
    from oracle import oracle
    oracle.build()
    cores = host_cores()
    _, warm = _oracle_batches(w, inputs, 16, 1)
    oracle_steps(w, warm[0])                                   # load + warm
    probe = oracle_pass(w, _oracle_batches(w, inputs, 256, 1)[1], 1)[0] / min(256, w.T)
    res = {}
    for label, threads in (("1core", 1), ("all_cores", cores)):
        n_tok = int(max(16, min(w.T, budget_s / 2 * threads / max(probe, 1e-9) / 3)))
        n, batches = _oracle_batches(w, inputs, n_tok, threads)
        spent, tokens, passes = 0.0, 0, 0
        steps = {s: 0.0 for s in KERNELS}
        while passes < 1 or (spent < budget_s / 2 and passes < 20):
            dt, per = oracle_pass(w, batches, threads)
            spent += dt
            tokens += n
            passes += 1
            for s in KERNELS:
                steps[s] += per[s]
        tot = sum(steps.values())
        res[label] = {"value": tokens / spent, "threads": threads, "tokens": tokens, "seconds": round(spent, 3),
                      "step_share": {s: round(steps[s] / tot, 4) for s in KERNELS},
                      "step_us_per_token": {s: round(1e6 * steps[s] / tokens, 3) for s in KERNELS}}
    one, allc = res["1core"], res["all_cores"]
    return {"value": allc["value"], "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "value_1core": one["value"], "per_step": res,
            "sample": f"{one['tokens']} tokens on 1 thread and {allc['tokens']} tokens on {cores} threads "
                      f"(token sub-batches of the {w.describe()} batch, each routed, expanded, activated "
                      "and combined on its own); plain C oracle in float64, unchanged; per-step split "
                      "summed over the threads' own step times"}


def reference_arm(args, rank, world):
    """The oracle as the reference implementation, timed on host cores on
    rank 0 only: each step is one pass over a bounded sample of the workload,
    cut into one independent token sub-batch per core."""
    if rank != 0:
        return
    from memory_bound_moe_gb300.workloads import WORKLOADS, generate
    w = WORKLOADS[args.workload]
    inputs = generate(w, seed=0)
    from oracle import oracle
    oracle.build()
    cores = host_cores()
    _, warm = _oracle_batches(w, inputs, 16, 1)
    oracle_steps(w, warm[0])
    t_probe = oracle_pass(w, _oracle_batches(w, inputs, 64, 1)[1], 1)[0] / min(64, w.T)  # s per token, 1 thread
    budget = 90.0                                          # whole run, seconds
    per_step = budget / max(1, args.steps + args.warmup)
    n_tok = int(max(1, min(w.T, per_step * cores / 2 / max(t_probe, 1e-9))))
    n, batches = _oracle_batches(w, inputs, n_tok, cores)
    for _ in range(args.warmup):
        oracle_pass(w, batches, cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_pass(w, batches, cores)
    dt = time.perf_counter() - t0
    value = n * args.steps / dt
    sample = (f"first {n} of {w.T} tokens of the {w.describe()} batch per step, as {len(batches)} "
              f"token sub-batches on {cores} threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_dict(w),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# process group
# ---------------------------------------------------------------------------

_PG = {"on": False}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and args.impl == "ours":
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        _PG["on"] = True
    return rank, world, local


def barrier():
    if _PG["on"]:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(v: float) -> float:
    """Max of a per-rank float over all ranks (identity without a group)."""
    if not _PG["on"]:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, tokens_per_rank: int, ms_step_max: float) -> float:
    """Whole-job tokens/s: every rank processes its own batch each step, and
    the job's step time is the slowest rank's."""
    return world * tokens_per_rank / (ms_step_max * 1e-3)


def step_bytes(w) -> tuple:
    """(algorithmic bytes of one step, bytes of its inputs: logits, x,
    gate_up, expert_out)."""
    ab = algorithmic_bytes(w)
    inputs = 4 * w.T * w.E + 2 * w.T * w.H + 4 * w.S * w.I + 2 * w.S * w.H
    return sum(ab.values()), inputs


L2_BYTES = 129 * 10 ** 6


def l2_note(w) -> str:
    total, inputs = step_bytes(w)
    if inputs > L2_BYTES:
        return (f"no flush: steps run back to back and one step streams {total / 1e6:.0f} MB "
                f"(inputs {inputs / 1e6:.0f} MB) through the 129 MB L2, so every input is evicted "
                "between its uses")
    return (f"no flush: a latency workload whose inputs ({inputs / 1e6:.1f} MB) stay in the 129 MB L2 "
            "between steps")


def config_dict(w):
    return {"workload": w.describe(), "T": w.T, "H": w.H, "E": w.E, "k": w.k, "renorm": w.renorm,
            "I": w.I, "storage": "bf16 activations, fp32 logits/weights", "l2": l2_note(w),
            "parallelism": "replicas (one independent batch per GPU)"}


# ---------------------------------------------------------------------------

def kernel_split(w, per_kernel, peak) -> dict:
    """Mean event duration, algorithmic bytes, GB/s and fraction of peak of
    each of the four calls."""
    ab = algorithmic_bytes(w)
    kern = {}
    for name in KERNELS:
        us = 1e3 * sum(per_kernel[name]) / len(per_kernel[name])
        gbs = ab[name] / (us * 1e-6) / 1e9
        kern[name] = {"us": round(us, 3), "algorithmic_bytes": ab[name], "GBps": round(gbs, 1),
                      "frac": round(gbs / peak, 4)}
    kern["sum_of_kernels_us"] = round(sum(kern[n]["us"] for n in KERNELS), 3)
    return kern


def time_alone(step, name, reps, dev):
    """One of the step's calls launched `reps` times back to back on the
    step's own buffers (after one untimed launch); mean microseconds per
    launch. Only meaningful where the call's inputs exceed L2, so that every
    launch reads them from HBM."""
    torch = step.torch
    sp = torch.cuda.current_stream(dev).cuda_stream
    fn = {"expand": lambda: step.lib.moe_expand(*step.expand_args, sp),
          "swiglu": lambda: step.lib.moe_swiglu(*step.swiglu_args, sp),
          "combine": lambda: step.lib.moe_combine(*step.combine_args, sp)}[name]
    assert fn() == 0
    torch.cuda.synchronize(dev)
    torch.cuda._sleep(4_000_000)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        assert fn() == 0
    b.record()
    torch.cuda.synchronize(dev)
    return 1e3 * a.elapsed_time(b) / reps


def measure_side(w, dev, scratch, steps, peak, seed):
    """A whole-path step on another workload: back-to-back device-resident
    steps (value) and the per-kernel event split."""
    from memory_bound_moe_gb300.workloads import generate
    step = Step(w, generate(w, seed=seed), dev)
    ms, _ = time_device_resident(step, steps, 20, dev, scratch)
    ms = reduce_max(ms)
    total, _ = step_bytes(w)
    kern = kernel_split(w, time_per_kernel(step, min(steps, 500), dev, scratch), peak)
    res = {"workload": w.describe(), "steps": steps, "ms_per_step": round(ms, 5),
           "tokens_per_s": round(job_throughput(_world(), w.T, ms), 1),
           "step_bytes": total, "path_GBps": round(total / (ms * 1e-3) / 1e9, 1),
           "path_frac": round(total / (ms * 1e-3) / 1e9 / peak, 4), "l2": l2_note(w), "kernels": kern}
    del step
    return res


def _world() -> int:
    return int(os.environ.get("WORLD_SIZE", "1"))


def main():
    args = parse_args()
    rank, world, local = dist_setup(args)
    if args.impl == "reference":
        reference_arm(args, rank, world)
        return
    import torch
    from memory_bound_moe_gb300 import build as cuda_build
    if rank == 0 or not _PG["on"]:
        cuda_build.build()
    barrier()
    cuda_build.build()
    from memory_bound_moe_gb300.workloads import WORKLOADS, generate
    w = WORKLOADS[args.workload]
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    inputs = generate(w, seed=rank)
    step = Step(w, inputs, dev)
    scratch = (torch.empty((L2_FLUSH_BYTES,), dtype=torch.uint8, device=dev),
               torch.ones((L2_FLUSH_BYTES // 4,), dtype=torch.float32, device=dev))

    remeasured = False
    for attempt in range(2):
        clocks = ClockSampler(str(torch.cuda.get_device_properties(dev).uuid))
        clocks.start()
        ms_step_local, wall = time_device_resident(step, args.steps, args.warmup, dev, scratch)
        clk = clocks.stop()
        if not (set(clk["reasons"]) & BAD_REASONS) or attempt == 1:
            break
        remeasured = True

    ms_step = reduce_max(ms_step_local)
    value = job_throughput(world, w.T, ms_step)
    per_kernel = time_per_kernel(step, min(max(args.steps, 200), 1000), dev, scratch)

    peak, peak_src = peak_hbm()
    kern = kernel_split(w, per_kernel, peak)
    dominant = max(KERNELS, key=lambda n: kern[n]["us"])
    total_bytes, input_bytes = step_bytes(w)
    roofline = {"bound": "hbm", "kernel": dominant, "achieved": kern[dominant]["GBps"], "peak": peak,
                "unit": "GB/s", "frac": kern[dominant]["frac"],
                "traffic": traffic_from_profiles(dominant, w.name),
                "algorithmic_bytes": kern[dominant]["algorithmic_bytes"],
                "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
                else "fallback 6.8 TB/s",
                "path_GBps": round(total_bytes / (ms_step * 1e-3) / 1e9, 1),
                "path_frac": round(total_bytes / (ms_step * 1e-3) / 1e9 / peak, 4)}
    # the dominant kernel alone, back to back on the step's own buffers when
    # its inputs exceed L2 (every launch then reads them from HBM)
    if dominant != "route" and kern[dominant]["algorithmic_bytes"] > 2 * L2_BYTES:
        us = time_alone(step, dominant, 50, dev)
        gbs = kern[dominant]["algorithmic_bytes"] / (us * 1e-6) / 1e9
        roofline["alone_us"] = round(us, 3)
        roofline["alone_GBps"] = round(gbs, 1)
        roofline["alone_frac"] = round(gbs / peak, 4)

    e2e = None
    if not args.no_e2e:
        e2e_ms, h2d, d2h = time_e2e(w, inputs, min(args.steps, 200), min(args.warmup, 5), dev)
        e2e_ms = reduce_max(e2e_ms)
        e2e = {"value": job_throughput(world, w.T, e2e_ms), "unit": "tokens/s", "ms_per_step": e2e_ms,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "h2d_GBps": round(h2d / (e2e_ms * 1e-3) / 1e9, 1),
               "how": "pinned host inputs copied every step in 32 MB chunks over 4 copy streams into "
                      "double-buffered device sets; the C-ABI calls through the Python binding; "
                      "out copied back on a separate stream"}
    launches = step.launches_per_step * args.steps

    more = args.workload == WORKLOAD and not args.no_extras
    side = None
    if more:
        del step
        torch.cuda.empty_cache()
        side = {}
        for name in SIDE_WORKLOADS:
            side[name] = measure_side(WORKLOADS[name], dev, scratch, args.extra_reps or 2000, peak, rank)
            torch.cuda.empty_cache()
    decode = decode_latency(dev, reps=args.extra_reps or 2000) if more else None
    extras = extras_measurement(dev, reps=args.extra_reps or 240) if more else None

    cpu = None
    if rank == 0 and world == 1 and args.cpu_budget > 0:
        cpu = cpu_baseline(w, inputs, args.cpu_budget)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": config_dict(w),
            "roofline": roofline, "kernels": kern, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": launches,
            "workloads": side,
            "decode_latency": decode,
            "extras": extras,
            "clocks": clk, "remeasured": remeasured, "wall_s_timed_region": round(wall, 3),
            "device": torch.cuda.get_device_name(dev),
        }
        print(json.dumps(line), flush=True)
    if _PG["on"]:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
