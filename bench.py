"""Benchmark of the fused memory-bound chains on GB300.

One step = one call of each fused chain on its at-scale synthetic workload:

    pointwise_f32_4Mi          y = relu(x + b1) * 0.5 + b2, 4 Mi fp32 elements
    inductor_f32_1024x1024     the TorchInductor example chain, fp32
    ln_gelu_f32_8192x4096      residual + LayerNorm + GeLU-tanh, fp32
    ln_gelu_bf16_32768x8192    residual + LayerNorm + GeLU-tanh, bf16 I/O

value = the step's read-once/write-once bytes / the step's kernel time
(effective HBM GB/s) with every input resident in device memory.  Exactly K
whole steps are captured in one CUDA graph and replayed between CUDA events
on the launching stream; each chain cycles through copies of its buffers
whose footprint is at least twice the L2, so every call streams its inputs
from HBM and every call's deferred L2 write-backs are paid inside the timed
region.  Each chain is also timed alone over K back-to-back calls for the
per-kernel figures.  Per-kernel microseconds per call, GB/s and fraction of the
measured HBM copy bandwidth are reported alongside, with the single-call
latency after an L2 flush and the unfused eager PyTorch chain (back-to-back,
same buffers).  `e2e` repeats the measurement through the same public API
with the row tensors in pinned host memory: the kernels read and write them
over the host link inside the timed region (the copy-engine pipeline, H2D /
call / D2H over three streams, is reported beside it).
`cpu_baseline` times the CPU oracle on a sample of the same step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun every rank runs the full per-GPU workload (weak scaling) and
rank 0 prints one JSON line.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from synth import workloads as W  # noqa: E402

STEP = (W.POINTWISE_4M, W.INDUCTOR_1024, W.LN_F32, W.LN_BF16)
METRIC = "effective HBM GB/s per fused-chain step (read-once/write-once bytes / kernel time)"
UNIT = "GB/s"
WORKLOAD = ("fused_chains_step: pointwise_f32_4Mi + inductor_f32_1024x1024 + "
            "ln_gelu_f32_8192x4096 + ln_gelu_bf16_32768x8192")
FLUSH_BYTES = 1 << 30
PEAKS_FALLBACK = {"hbm_gbs": 6800.0}
NOMINAL_HBM_GBS = 8000.0


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-eager", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-next", action="store_true",
                    help="skip the further chains (softmax, LayerNorm family, bf16 Inductor)")
    return ap.parse_args(argv)


# --------------------------------------------------------------------------
# environment
# --------------------------------------------------------------------------

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": PEAKS_FALLBACK["hbm_gbs"], "source": "fallback"}


def source_hash():
    """Hash of the CUDA sources, to tell whether stored ncu counters still
    describe the kernels being timed."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "memory_bound_gb300", "csrc")
    for name in sorted(os.listdir(d)):
        with open(os.path.join(d, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def stored_traffic(kernel_key):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current sources; else None."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    try:
        lines = open(p).read().splitlines()
    except OSError:
        return None
    cur = source_hash()
    for ln in lines:
        parts = ln.split()
        if len(parts) >= 3 and not ln.startswith("#") and parts[0] == kernel_key and parts[1] == cur:
            return float(parts[2])
    return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index, enabled=True):
        self.index, self.proc, self.enabled = index, None, enabled

    def __enter__(self):
        if self.enabled:
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                     "--format=csv,noheader,nounits", "-lms", "20"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
                time.sleep(1.0)                 # let nvidia-smi start sampling
            except OSError:
                self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        if not self.enabled or self.proc is None:
            return None
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.out.splitlines():
            f = [c.strip() for c in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "samples": len(sm),
                "reasons": sorted(reasons)}


# --------------------------------------------------------------------------
# our arm
# --------------------------------------------------------------------------

def _dev(a, bf16, device):
    import torch
    if bf16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)


def _pinned(a, bf16):
    import torch
    t = torch.from_numpy(a.view(np.int16) if bf16 else a).pin_memory()
    return t.view(torch.bfloat16) if bf16 else t


class Case:
    """One workload: its host inputs, `nsets` device copies of its buffers
    (footprint >= 2x L2), and its calls (ours and eager)."""

    def __init__(self, w, device, l2_bytes):
        import torch
        self.w = w
        self.bf16 = w.dtype == "bf16"
        host = w.generate_all()
        self.host = host
        shape = (w.cols,) if w.chain == "add_relu_scale" else (w.rows, w.cols)
        dt = torch.bfloat16 if self.bf16 else torch.float32
        self.ideal = w.ideal_bytes()
        self.nsets = max(1, -(-2 * l2_bytes // self.ideal))
        first = {k: _dev(v, self.bf16, device) for k, v in host.items()}
        self.sets = [first] + [{k: v.clone() for k, v in first.items()}
                               for _ in range(self.nsets - 1)]
        self.outs = [torch.empty(shape, dtype=dt, device=device) for _ in range(self.nsets)]
        self.houts = ([torch.empty(shape, dtype=dt, device=device) for _ in range(self.nsets)]
                      if w.params.get("write_h") else None)
        self.dev, self.out = self.sets[0], self.outs[0]
        self.in_bytes = sum(v.nbytes for v in host.values())
        self.out_bytes = self.out.numel() * self.out.element_size()

    def call(self, k=0):
        import memory_bound_gb300 as mb
        d, out = self.sets[k % self.nsets], self.outs[k % self.nsets]
        p = self.w.params
        if self.w.chain in ("add_relu_scale", "add_relu_scale_bcast"):
            mb.fused_add_relu_scale(d["x"], d["b1"], d["b2"], p["scale"], out=out)
        elif self.w.chain == "inductor":
            mb.fused_bias_relu_branch_mean_epilogue(d["x"], d["bias"], d["gamma"], d["beta"],
                                                    p["x_scale"], p["branch_scale"], out=out)
        elif self.w.chain == "softmax":
            mb.fused_row_softmax(d["x"], out=out)
        elif self.w.chain == "softmax_mask":
            mb.fused_row_softmax(d["x"], out=out, scale=p["scale"], causal=p["causal"],
                                 period=p["period"], offset=p["offset"])
        elif self.w.chain == "lnact":
            mb.fused_layernorm_act(d["x"], d.get("r"), d["w"], d["b"], eps=p["eps"],
                                   act=p["act"], out=out,
                                   h_out=self.houts[k % self.nsets] if p["write_h"] else None,
                                   p=p.get("p", 0.0), seed=p.get("seed", 0),
                                   offset=p.get("offset", 0))
        else:
            mb.fused_residual_layernorm_gelu(d["x"], d["r"], d["w"], d["b"], p["eps"], out=out)

    def call_on(self, d, out, a, b):
        """The fused call on rows (elements) [a, b) of the buffers d / out."""
        import memory_bound_gb300 as mb
        p = self.w.params
        if self.w.chain == "add_relu_scale":
            mb.fused_add_relu_scale(d["x"][a:b], d["b1"][a:b], d["b2"][a:b], p["scale"],
                                    out=out[a:b])
        elif self.w.chain == "inductor":
            mb.fused_bias_relu_branch_mean_epilogue(d["x"][a:b], d["bias"], d["gamma"], d["beta"],
                                                    p["x_scale"], p["branch_scale"], out=out[a:b])
        else:
            mb.fused_residual_layernorm_gelu(d["x"][a:b], d["r"][a:b], d["w"], d["b"], p["eps"],
                                             out=out[a:b])

    def eager(self, k=0):
        """The unfused PyTorch eager chain (the pages' motivating baseline)."""
        import torch
        import torch.nn.functional as F
        d, p = self.sets[k % self.nsets], self.w.params
        if self.w.chain in ("add_relu_scale", "add_relu_scale_bcast"):
            return torch.relu(d["x"] + d["b1"]) * p["scale"] + d["b2"]
        if self.w.chain == "softmax":
            return torch.softmax(d["x"], dim=1)
        if self.w.chain == "softmax_mask":
            if not hasattr(self, "_mask"):
                q = torch.arange(self.w.rows, device=d["x"].device)[:, None] % p["period"]
                k = torch.arange(self.w.cols, device=d["x"].device)[None, :]
                self._mask = k > q + p["offset"]          # built once, outside the timing
            return torch.softmax((d["x"] * p["scale"]).masked_fill(self._mask, float("-inf")),
                                 dim=1)
        if self.w.chain == "lnact":
            v = d["x"] + d["r"] if "r" in d else d["x"]
            n = F.layer_norm(v, (self.w.cols,), d["w"], d["b"], p["eps"])
            a = torch.relu(n) if p["act"] == "relu" else F.gelu(n, approximate="tanh")
            return F.dropout(a, p["p"]) if p.get("p") else a
        if self.w.chain == "inductor":
            t = d["x"] * p["x_scale"] + d["bias"]
            a = torch.relu(t)
            s = a * a + a * p["branch_scale"]
            m = s.mean(dim=1, keepdim=True)
            return (s - m) * d["gamma"] + d["beta"]
        return F.gelu(F.layer_norm(d["x"] + d["r"], (self.w.cols,), d["w"], d["b"], p["eps"]),
                      approximate="tanh")


class CopyCase:
    """A plain device-to-device copy moving as many bytes as a workload's
    call (half read, half written), cycling through buffer sets like Case:
    the size-matched copy each kernel is compared with.  Copies are issued in
    pieces of at most 256 MiB: single copies above about 1 GB ran at half the
    speed on GB300, which would flatter the kernels."""

    PIECE = 64 << 20     # floats (256 MiB)

    def __init__(self, case, device):
        import torch
        from types import SimpleNamespace
        self.w = SimpleNamespace(name=case.w.name)
        n = (case.ideal // 2 // 4) & ~3      # whole 16-byte vectors: torch's vector copy path
        self.src = [torch.ones(n, dtype=torch.float32, device=device) for _ in range(case.nsets)]
        self.dst = [torch.empty(n, dtype=torch.float32, device=device) for _ in range(case.nsets)]

    def call(self, k=0):
        d, src = self.dst[k % len(self.dst)], self.src[k % len(self.src)]
        for a in range(0, d.numel(), self.PIECE):
            d[a:a + self.PIECE].copy_(src[a:a + self.PIECE])


def aggregate_ranks(step_ms, step_bytes, world, device=None):
    """Whole-job throughput: every rank processed `step_bytes` per step; the
    job's step time is the slowest rank's.  Returns (max step ms, GB/s).
    Host-side timing exchange only (one scalar), not a data-path collective."""
    if world > 1:
        import torch
        import torch.distributed as dist
        tt = torch.tensor([float(step_ms)], dtype=torch.float64,
                          device=device if device is not None else "cpu")
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        step_ms = float(tt.item())
    return step_ms, world * step_bytes / (step_ms * 1e-3) / 1e9


def time_steady(cases, fn, steps, warmup):
    """Per case: mean milliseconds per call over `steps` back-to-back calls
    cycling through its buffer sets (one event pair around the loop)."""
    import torch
    stream = torch.cuda.current_stream()
    for c in cases:
        for k in range(warmup):
            fn(c, k)
    torch.cuda.synchronize()
    ev = {}
    for c in cases:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for k in range(steps):
            fn(c, k)
        b.record(stream)
        ev[c.w.name] = (a, b)
    torch.cuda.synchronize()
    return {name: a.elapsed_time(b) / steps for name, (a, b) in ev.items()}


def time_graph(cases, fn, steps, warmup, replays=1):
    """Per case: milliseconds per call over `steps` back-to-back calls
    cycling through its buffer sets, captured once into a CUDA graph and
    replayed between CUDA events, so the GPU runs the calls back to back with
    no host launch gaps (the calls themselves are the library's ordinary
    entry points; it neither allocates nor synchronises, so it captures).
    With replays > 1 the graph is replayed that many times, each replay
    between its own event pair; a case then maps to the list of per-call
    means, one per replay (else to the one mean)."""
    import torch
    stream = torch.cuda.current_stream()
    out = {}
    for c in cases:
        for k in range(warmup):                 # W untimed calls
            fn(c, k)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()              # capture records, runs nothing
        with torch.cuda.graph(g, capture_error_mode="thread_local"):
            for k in range(steps):
                fn(c, k)
        g.replay()                              # untimed: the first launch uploads the graph
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(replays)]
        for a, b in ev:
            a.record(stream)
            g.replay()
            b.record(stream)
        torch.cuda.synchronize()
        ms = [a.elapsed_time(b) / steps for a, b in ev]
        out[c.w.name] = ms if replays > 1 else ms[0]
        del g
    return out


def spread(ms_list):
    """(mean, median, p10, p90) of per-call milliseconds, one per replay."""
    q = np.percentile(np.array(ms_list), [50, 10, 90])
    return float(np.mean(ms_list)), float(q[0]), float(q[1]), float(q[2])


def time_steps_graph(cases, steps, warmup, world=1):
    """Whole steps: one step calls every chain once (each on its next buffer
    set); `steps` steps are captured into one CUDA graph, replayed once
    untimed (graph upload), then replayed between CUDA events on the
    launching stream, bracketed by a barrier (under torchrun) and a
    synchronize on both sides.  Returns milliseconds per step."""
    import torch
    stream = torch.cuda.current_stream()
    for k in range(warmup):
        for c in cases:
            c.call(k)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="thread_local"):
        for k in range(steps):
            for c in cases:
                c.call(k)
    g.replay()
    torch.cuda.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    g.replay()
    b.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    del g
    return a.elapsed_time(b) / steps


def plan_chain(w):
    """The row-plan query name of a workload's chain (None for the pointwise
    chains, which have no row plan)."""
    p = w.params
    if w.chain == "ln_gelu":
        return "ln"
    if w.chain in ("inductor", "softmax", "softmax_mask"):
        return w.chain
    if w.chain == "lnact":
        if p.get("write_h"):
            return "lnact_res_h"
        name = "lnact_res" if p.get("residual") else "lnact"
        return name + "_dropout" if p.get("p") else name
    return None


def time_single_flushed(cases, fn, reps, flush):
    """Per case: (p10, median, p90) milliseconds of one call after an L2
    flush (a 1 GiB read, outside the events) -- the latency of an isolated
    call and its spread; ten untimed calls first."""
    import torch
    stream = torch.cuda.current_stream()
    out = {}
    for c in cases:
        for _ in range(10):
            fn(c, 0)
        ts = []
        for _ in range(reps):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn(c, 0)
            b.record(stream)
            b.synchronize()
            ts.append(a.elapsed_time(b))
        q = np.percentile(np.array(ts), [10, 50, 90])
        out[c.w.name] = tuple(float(v) for v in q)
    return out


def time_e2e(cases, steps, warmup, chunks=8):
    """Through the public API from pinned host buffers.  Per step and chain:
    H2D of every input, the fused call, D2H of the output, all inside the
    events.  The rows (elements for the pointwise chain) are split into
    `chunks` pieces pipelined over three streams -- H2D of piece c+1 and D2H
    of piece c-1 overlap the call on piece c -- chained by CUDA events."""
    import torch
    main = torch.cuda.current_stream()
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    items = []
    for c in cases:
        hin = {k: _pinned(v, c.bf16) for k, v in c.host.items()}
        hout = torch.empty(c.out.shape, dtype=c.out.dtype).pin_memory()
        lead = c.out.shape[0]
        bounds = [lead * i // chunks for i in range(chunks + 1)]
        items.append((c, hin, hout, bounds))

    def one_step():
        start = torch.cuda.Event()
        start.record(main)
        for st in (s_in, s_cmp, s_out):
            st.wait_event(start)
        for c, hin, hout, bounds in items:
            d, out = c.sets[0], c.outs[0]
            percol = {k for k, v in hin.items() if v.dim() == 1 and c.w.chain != "add_relu_scale"}
            with torch.cuda.stream(s_in):
                for k in percol:
                    d[k].copy_(hin[k], non_blocking=True)
            for i in range(len(bounds) - 1):
                a, b = bounds[i], bounds[i + 1]
                if a == b:
                    continue
                ev_in, ev_cmp = torch.cuda.Event(), torch.cuda.Event()
                with torch.cuda.stream(s_in):
                    for k, v in hin.items():
                        if k not in percol:
                            d[k][a:b].copy_(v[a:b], non_blocking=True)
                    ev_in.record(s_in)
                with torch.cuda.stream(s_cmp):
                    s_cmp.wait_event(ev_in)
                    c.call_on(d, out, a, b)
                    ev_cmp.record(s_cmp)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_cmp)
                    hout[a:b].copy_(out[a:b], non_blocking=True)
        for st in (s_in, s_cmp, s_out):
            done = torch.cuda.Event()
            done.record(st)
            main.wait_event(done)

    for _ in range(warmup):
        one_step()
    torch.cuda.synchronize()
    ms = []
    for _ in range(steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(main)
        one_step()
        b.record(main)
        torch.cuda.synchronize()
        ms.append(a.elapsed_time(b))
    bi = sum(c.in_bytes for c in cases)
    bo = sum(c.out_bytes for c in cases)
    return ms, bi, bo


def time_e2e_zero_copy(cases, steps, warmup):
    """Through the public API with the row tensors in pinned host memory: the
    kernels read the inputs and write the outputs over the host link (no
    staging copy); the per-column vectors are copied H2D each step, on the
    same stream, before the call that reads them.  One step = every chain
    once, back to back, between CUDA events."""
    import torch
    main = torch.cuda.current_stream()
    items = []
    for c in cases:
        rowk = [k for k, v in c.host.items() if v.ndim == 2 or c.w.chain == "add_relu_scale"]
        hrows = {k: _pinned(c.host[k], c.bf16) for k in rowk}
        hcols = {k: _pinned(v, c.bf16) for k, v in c.host.items() if k not in hrows}
        dcols = {k: c.sets[0][k] for k in hcols}
        hout = torch.empty(c.out.shape, dtype=c.out.dtype).pin_memory()
        items.append((c, hrows, hcols, dcols, hout))

    def one_step():
        for c, hrows, hcols, dcols, hout in items:
            for k, v in hcols.items():
                dcols[k].copy_(v, non_blocking=True)
            c.call_on({**hrows, **dcols}, hout, 0, hout.shape[0])

    for _ in range(warmup):
        one_step()
    torch.cuda.synchronize()
    ms = []
    for _ in range(steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(main)
        one_step()
        b.record(main)
        torch.cuda.synchronize()
        ms.append(a.elapsed_time(b))
    bi = sum(c.in_bytes for c in cases)
    bo = sum(c.out_bytes for c in cases)
    return ms, bi, bo


def host_info():
    """The CPU the oracle runs on: model and the cores this process may use."""
    import platform
    model = platform.processor() or platform.machine()
    arm_parts = {"0xd4f": "Arm Neoverse V2", "0xd40": "Arm Neoverse V1", "0xd0c": "Arm Neoverse N1",
                 "0xd49": "Arm Neoverse N2", "0xd8f": "Arm Neoverse V3"}
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                key = ln.split(":")[0].strip().lower()
                if key in ("model name", "cpu part"):
                    val = ln.split(":", 1)[1].strip()
                    model = f"{platform.machine()} {arm_parts.get(val, val)}"
                    break
    except OSError:
        pass
    try:
        avail = len(os.sched_getaffinity(0))
    except AttributeError:
        avail = os.cpu_count()
    return {"cpu": model, "cores_available": avail}


def cpu_sample(fraction):
    """The inputs of a `fraction` sample of the step: the first rows of each
    row workload, the first elements of the pointwise one."""
    out = []
    for w in STEP:
        if w.chain == "add_relu_scale":
            n = max(1, int(round(w.cols * fraction)))
            t = {k: np.ascontiguousarray(v[:n]) for k, v in w.generate_all().items()}
            out.append((w, t, 16 * n, f"{w.name}: {n} of {w.cols} elements"))
        else:
            rows = max(1, int(round(w.rows * fraction)))
            t = w.generate_all(rows=rows)
            out.append((w, t, w.ideal_bytes(rows), f"{w.name}: {rows} of {w.rows} rows"))
    return out


def cpu_baseline(sample):
    """The CPU oracle, as it stands, on a sample from cpu_sample().
    Returns (GB/s, seconds, sample description)."""
    import oracle
    tot_bytes, tot_s = 0, 0.0
    for w, t, nbytes, _ in sample:
        t0 = time.perf_counter()
        if w.chain == "add_relu_scale":
            oracle.add_relu_scale(t["x"], t["b1"], t["b2"], w.params["scale"])
        elif w.chain == "inductor":
            oracle.bias_relu_branch_mean_epilogue(t["x"], t["bias"], t["gamma"], t["beta"],
                                                  w.params["x_scale"], w.params["branch_scale"])
        else:
            oracle.residual_layernorm_gelu(t["x"], t["r"], t["w"], t["b"], w.params["eps"])
        tot_s += time.perf_counter() - t0
        tot_bytes += nbytes
    return tot_bytes / tot_s / 1e9, tot_s, "; ".join(d for *_, d in sample)


# --- the same oracle on every available core (row chunks, one process each) ---

_PAR = {}


def _par_init(barrier):
    sys.path.insert(0, ROOT)
    _PAR["barrier"] = barrier


def _par_load(chunks):
    """Worker: keep this worker's row chunks (outside the timing)."""
    import oracle
    oracle.load()
    _PAR["chunks"] = chunks
    return os.getpid()


def _par_run(_):
    """Worker: wait for every worker, then run the oracle on its chunks."""
    import oracle
    _PAR["barrier"].wait()
    t0 = time.perf_counter()
    for chain, params, t in _PAR["chunks"]:
        if chain == "add_relu_scale":
            oracle.add_relu_scale(t["x"], t["b1"], t["b2"], params["scale"])
        elif chain == "inductor":
            oracle.bias_relu_branch_mean_epilogue(t["x"], t["bias"], t["gamma"], t["beta"],
                                                  params["x_scale"], params["branch_scale"])
        else:
            oracle.residual_layernorm_gelu(t["x"], t["r"], t["w"], t["b"], params["eps"])
    return time.perf_counter() - t0


def cpu_baseline_all_cores(sample, workers):
    """The unchanged oracle on `workers` processes at once, each on a
    contiguous slice of every workload's rows (elements for the pointwise
    chain), started together at a barrier.  Returns (GB/s, seconds of the
    slowest worker).  Processes are spawned, never forked."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    barrier = ctx.Barrier(workers)
    per = [[] for _ in range(workers)]
    tot_bytes = 0
    for w, t, nbytes, _ in sample:
        tot_bytes += nbytes
        lead = next(iter(v for v in t.values() if w.chain == "add_relu_scale" or v.ndim == 2)).shape[0]
        for i in range(workers):
            a, b = lead * i // workers, lead * (i + 1) // workers
            part = {k: (v[a:b] if (w.chain == "add_relu_scale" or v.ndim == 2) else v)
                    for k, v in t.items()}
            per[i].append((w.chain, dict(w.params), part))
    with ctx.Pool(workers, initializer=_par_init, initargs=(barrier,)) as pool:
        # one chunk set per worker process (the pool may not spread plain map
        # calls evenly, so each task pins its chunks by a blocking barrier)
        pids = pool.map(_par_load_one, [(i, per[i]) for i in range(workers)], chunksize=1)
        assert len(set(pids)) == workers
        secs = pool.map(_par_run, range(workers), chunksize=1)
    wall = max(secs)
    return tot_bytes / wall / 1e9, wall


def _par_load_one(item):
    """Worker: take one chunk set, then hold until every worker has one, so
    that each process ends up with exactly one."""
    _, chunks = item
    pid = _par_load(chunks)
    _PAR["barrier"].wait()
    return pid


def run_ours(args):
    import torch
    import torch.distributed as dist

    import memory_bound_gb300 as mb
    from memory_bound_gb300 import build as lib_build

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if rank == 0 or world > 1:
        lib_build.build()
    if world > 1:
        dist.barrier()
    mb.load_library()
    mb.set_row_path("auto")

    # CPU baseline first (rank 0, N=1 only), before any GPU work is timed
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        gbs, secs, sample = cpu_baseline(cpu_sample(0.25))
        host = host_info()
        cpu = {"value": round(gbs, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
               "host": host,
               "sample": f"first quarter of each workload ({sample}); {secs:.1f} s single-threaded"}
        n_par = min(16, host["cores_available"] or 1)
        if n_par > 1:
            try:
                pg, ps = cpu_baseline_all_cores(cpu_sample(0.25), n_par)
                cpu["all_cores"] = {"value": round(pg, 4), "unit": UNIT, "cores": n_par,
                                    "kind": "oracle",
                                    "sample": f"the same sample split into {n_par} row slices, "
                                              f"one spawned process each; {ps:.2f} s for the "
                                              "slowest"}
            except Exception as e:          # a reported baseline, never a reason to fail
                cpu["all_cores"] = {"unavailable": f"{type(e).__name__}: {e}"[:200]}

    props = torch.cuda.get_device_properties(device)
    l2_bytes = int(getattr(props, "L2_cache_size", 0) or (132 << 20))
    cases = [Case(w, device, l2_bytes) for w in STEP]
    flush_buf = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=device).fill_(1.0)

    def flush():
        flush_buf.sum()

    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    # per-kernel figures: the K-call graph replayed until at least 100 calls
    # (and 10 replays) are timed; median and spread over the replays
    replays = max(10, -(-100 // args.steps))
    with ClockSampler(local, enabled=not args.no_clocks) as clk:
        t_wall0 = time.perf_counter()
        step_region_ms = time_steps_graph(cases, args.steps, args.warmup, world)
        t_wall = time.perf_counter() - t_wall0
        ours = time_graph(cases, lambda c, k: c.call(k), args.steps, args.warmup, replays)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = clk.summary()

    copies = [CopyCase(c, device) for c in cases]
    copy_ms = time_graph(copies, lambda c, k: c.call(k), args.steps, 2)
    del copies
    stream_api = time_steady(cases, lambda c, k: c.call(k), args.steps, 2)
    single = time_single_flushed(cases, lambda c, k: c.call(k), 100, flush)
    eager = None
    if not args.no_eager:
        eager = time_graph(cases, lambda c, k: c.eager(k), max(5, args.steps // 5), 2)

    e2e = e2e_copy = None
    if not args.no_e2e:
        ms, bi, bo = time_e2e_zero_copy(cases, max(5, args.steps // 5), 3)
        e2e = (statistics.mean(ms), bi, bo)
        ms, _, _ = time_e2e(cases, max(5, args.steps // 5), 3)
        e2e_copy = statistics.mean(ms)

    peaks = measured_peaks()
    per_kernel = {}
    step_ms = 0.0
    step_bytes = 0
    for c in cases:
        mean_ms, med_ms, p10_ms, p90_ms = spread(ours[c.w.name])
        step_ms += mean_ms
        step_bytes += c.ideal
        gbs = c.ideal / (med_ms * 1e-3) / 1e9
        entry = {"us_per_call": round(med_ms * 1e3, 3),
                 "us_per_call_p10_p90": [round(p10_ms * 1e3, 3), round(p90_ms * 1e3, 3)],
                 "us_per_call_mean": round(mean_ms * 1e3, 3),
                 "calls_timed": replays * args.steps,
                 "ideal_bytes": c.ideal, "gbs": round(gbs, 1),
                 "frac_of_measured_hbm": round(gbs / peaks["hbm_gbs"], 4),
                 "frac_of_nominal_8tbs": round(gbs / NOMINAL_HBM_GBS, 4),
                 "buffer_sets": c.nsets,
                 "us_per_call_python_stream": round(stream_api[c.w.name] * 1e3, 3),
                 "us_single_call_l2_flushed": round(single[c.w.name][1] * 1e3, 3),
                 "us_single_call_l2_flushed_p10_p90": [round(single[c.w.name][0] * 1e3, 3),
                                                       round(single[c.w.name][2] * 1e3, 3)],
                 "size_matched_copy_us": round(copy_ms[c.w.name] * 1e3, 3),
                 "frac_of_size_matched_copy": round(copy_ms[c.w.name] / med_ms, 4)}
        if plan_chain(c.w):
            entry["launch"] = mb.row_plan(plan_chain(c.w), c.w.dtype, c.w.rows, c.w.cols)
        if eager:
            em = eager[c.w.name]
            entry["eager_us_per_call"] = round(em * 1e3, 3)
            entry["speedup_vs_eager"] = round(em / mean_ms, 2)
        per_kernel[c.w.name] = entry

    # The scope table's further chains, measured the same way (not part of
    # the step or its value).
    next_rows = None
    if not args.no_next:
        nxt = [Case(w, device, l2_bytes) for w in W.NEXT]
        t_next = time_graph(nxt, lambda c, k: c.call(k), args.steps, args.warmup, replays)
        e_next = (time_graph(nxt, lambda c, k: c.eager(k), max(5, args.steps // 5), 2)
                  if not args.no_eager else None)
        cp_next = {}
        for c in nxt:                       # one chain's copies at a time (memory)
            cc = CopyCase(c, device)
            cp_next.update(time_graph([cc], lambda x, k: x.call(k), args.steps, 2))
            del cc
        next_rows = {}
        for c in nxt:
            mean_ms, ms, p10_ms, p90_ms = spread(t_next[c.w.name])
            gbs = c.ideal / (ms * 1e-3) / 1e9
            ent = {"us_per_call": round(ms * 1e3, 3),
                   "us_per_call_p10_p90": [round(p10_ms * 1e3, 3), round(p90_ms * 1e3, 3)],
                   "us_per_call_mean": round(mean_ms * 1e3, 3), "ideal_bytes": c.ideal,
                   "gbs": round(gbs, 1), "frac_of_measured_hbm": round(gbs / peaks["hbm_gbs"], 4),
                   "size_matched_copy_us": round(cp_next[c.w.name] * 1e3, 3),
                   "frac_of_size_matched_copy": round(cp_next[c.w.name] / ms, 4)}
            if plan_chain(c.w):
                ent["launch"] = mb.row_plan(plan_chain(c.w), c.w.dtype, c.w.rows, c.w.cols)
            if e_next:
                ent["eager_us_per_call"] = round(e_next[c.w.name] * 1e3, 3)
                ent["speedup_vs_eager"] = round(e_next[c.w.name] / ms, 2)
            next_rows[c.w.name] = ent
        del nxt

    # The launch-bound configs (the 4096-element pointwise chain and the
    # Inductor chain) back to back on a single buffer set: their inputs stay
    # in the L2, so this is the call rate of a small chain, labelled hot-L2.
    hot_l2 = {}
    for w in (W.POINTWISE_TINY, W.INDUCTOR_1024):
        hc = Case(w, device, 0)
        ms = time_graph([hc], lambda c, k: c.call(k), max(100, args.steps), args.warmup)[w.name]
        hot_l2[w.name] = {"us_per_call": round(ms * 1e3, 3), "ideal_bytes": hc.ideal,
                          "l2": "hot: one buffer set, calls back to back in one graph"}
        del hc

    kernels_sum_ms = step_ms
    step_ms, value = aggregate_ranks(step_region_ms, step_bytes, world, device)

    dominant = max(cases, key=lambda c: per_kernel[c.w.name]["us_per_call"])
    dk = per_kernel[dominant.w.name]
    achieved = dominant.ideal / (dk["us_per_call_mean"] * 1e-6) / 1e9   # average launch
    roofline = {"bound": "hbm", "kernel": dominant.w.name,
                "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4),
                "peak_source": f"{peaks['source']} (MEASURED_PEAKS.json hbm_gbs, copy burst)",
                "traffic": stored_traffic(dominant.w.name),
                "algorithmic_bytes_per_launch": dominant.ideal}

    line = {"metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "io_dtypes": ["f32", "bf16"],
            "data": "synthetic (seeded SplitMix64/Box-Muller)",
            "config": {"workload": WORKLOAD,
                       "l2": f"inputs larger than L2: each chain cycles through buffer copies "
                             f"totalling >= 2x the {l2_bytes >> 20} MiB L2",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "timing": "W warmup steps; exactly K whole steps (each chain once, on "
                                 "its next buffer set) captured in one CUDA graph, one untimed "
                                 "replay (graph upload), then one replay between CUDA events on "
                                 "the launching stream, bracketed by a barrier and a synchronize "
                                 "on both sides: ms_per_step = that time / K. Per-kernel "
                                 "figures: each chain's K calls in a graph of their own, timed "
                                 "the same way; eager timed the same way"},
            "kernels": per_kernel, "roofline": roofline,
            "ms_per_step_sum_of_kernels": round(kernels_sum_ms, 4),
            "gpu_launches": args.steps * len(cases),
            "wall_s_timed_region": round(t_wall, 3)}
    if clocks:
        line["clocks"] = clocks
    if next_rows:
        line["next_rows"] = next_rows
    line["hot_l2"] = hot_l2
    if e2e:
        e_ms, bi, bo = e2e
        e2e_ms = aggregate_ranks(e_ms, step_bytes, world, device)[0]
        cp_ms = aggregate_ranks(e2e_copy, step_bytes, world, device)[0]
        line["e2e"] = {"value": round(world * step_bytes / (e2e_ms * 1e-3) / 1e9, 1),
                       "unit": UNIT, "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
                       "ms_per_step": round(e2e_ms, 3),
                       "mode": "zero copy: each chain called on pinned host row tensors; its "
                               "kernel reads the inputs and writes the output over the host "
                               "link (NVLink-C2C); per-column vectors copied H2D each step",
                       "copy_engine_pipelined": {
                           "value": round(world * step_bytes / (cp_ms * 1e-3) / 1e9, 1),
                           "ms_per_step": round(cp_ms, 3),
                           "note": "same step with device-resident buffers: H2D, fused call, "
                                   "D2H, each chain in 8 row chunks pipelined over 3 streams"}}
    if cpu:
        line["cpu_baseline"] = cpu
    line["per_kernel_summary"] = kernel_summary(per_kernel, next_rows, hot_l2)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def kernel_summary(per_kernel, next_rows, hot_l2):
    """Every measured kernel in a few characters each, printed as the last key
    of the JSON line so that a reader keeping only the end of the line still
    has them: per workload [median us/call, p10, p90, GB/s, fraction of the
    measured HBM copy peak, fraction of a size-matched copy]."""
    out = {"fields": ["us_median", "us_p10", "us_p90", "GB/s", "frac_of_measured_hbm",
                      "frac_of_size_matched_copy"]}
    for table in (per_kernel, next_rows or {}):
        for name, e in table.items():
            p10, p90 = e["us_per_call_p10_p90"]
            out[name] = [e["us_per_call"], p10, p90, e["gbs"], e["frac_of_measured_hbm"],
                         e["frac_of_size_matched_copy"]]
    out["hot_l2_us_per_call"] = {k: v["us_per_call"] for k, v in hot_l2.items()}
    return out


# --------------------------------------------------------------------------
# reference arm: the CPU oracle, timed on the host cores
# --------------------------------------------------------------------------

def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from oracle import build as oracle_build
    oracle_build.build()
    full_cpu_s = 32.0                   # whole step on one core, measured order
    total = args.steps + args.warmup
    fraction = min(0.125, 120.0 / (total * full_cpu_s))
    inputs = cpu_sample(fraction)
    for _ in range(args.warmup):
        cpu_baseline(inputs)
    vals, secs = [], []
    sample = ""
    for _ in range(args.steps):
        gbs, s, sample = cpu_baseline(inputs)
        vals.append(gbs)
        secs.append(s)
    value = sum(vals) / len(vals)
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * statistics.mean(secs), 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "dtype_note": "the oracle: fp32 op by op for the pointwise steps, "
                                                "double for the statistics and the transcendentals",
            "data": "synthetic (seeded SplitMix64/Box-Muller)",
            "config": {"workload": WORKLOAD,
                       "sample": f"{fraction:.4f} of each workload per step"},
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": 1,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
