"""Benchmark of the multi-LoRA linear layer on one GB300 (or N replicas).

A step is one pass of the whole hot path over one batch: the plan of the
batch's token slot ids, then for every adapted target the layer (shrink +
tensor-core GEMM with the fused expand). The headline workload is the largest
one: the full Llama-3-8B decoder-layer sweep over its seven targets at T=4096
rows (50 resident rank-16 adapters per target). The same JSON line carries a
`per_config` block with every configuration of the parity set (the tiny case,
the q_proj decode step, the gate/up prefill, the mixed-rank down projection,
and the layer sweep at T = 1, 8, 64, 512, 4096).

Steps form a dependent chain wherever the shapes allow one: step j + 1's x is
step j's output (the layer's own output for a square projection; the down
projection's output for the layer sweep, as in a decoder), so no step can
overlap the next. Where no shape-compatible chain exists the steps reuse one
resident x; a call's first kernel still waits for the kernel ahead of it
before it reads x, so those steps are serialised the same way.

Prints one JSON line. `value` is tokens/s over all ranks with inputs resident
in HBM; `e2e` is the same through the public API with inputs copied from
pinned host memory and the outputs copied back inside the timed region;
`roofline` rates the dominant kernel against the measured peaks (the burst
bf16 figure, as the kernel is timed in isolation); `cpu_baseline` is the fp64
CPU oracle on a bounded sample of the same batch.

Weight copies rotate between steps so the working set exceeds twice the L2.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "tokens/s and % of roofline for base GEMM + multi-LoRA SGMV per linear layer"
DEFAULT_CONFIG = "layer_sweep_T4096"
# The five configurations: tiny, q_proj decode, gate/up prefill, mixed-rank
# down projection, and the layer sweep at every batch size.
PER_CONFIGS = ("tiny", "q_decode", "gateup_prefill", "mixed_down", "layer_sweep_T1", "layer_sweep_T8",
               "layer_sweep_T64", "layer_sweep_T512", "layer_sweep_T4096")


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--per-config", default=",".join(PER_CONFIGS),
                    help="comma-separated workloads measured for the per_config block ('' for none)")
    ap.add_argument("--config-seconds", type=float, default=0.3,
                    help="timed GPU time of each per_config entry")
    ap.add_argument("--no-graph", action="store_true", help="launch steps eagerly instead of replaying graphs")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--reference-seconds", type=float, default=60.0,
                    help="total CPU time of the reference arm (warm-up + timed steps)")
    ap.add_argument("--kernel-steps", type=int, default=40)
    ap.add_argument("--profile-steps", type=int, default=0,
                    help="run this many eager steps of --config after 3 warm-up steps, untimed, and exit: "
                         "the launch sequence of one step, for an external profiler's launch list")
    return ap.parse_args(argv)


def peaks():
    """(HBM GB/s, bf16 TFLOP/s burst, bf16 TFLOP/s sustained, source)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


# The files a kernel's DRAM traffic depends on: its own source, the shared
# headers and the host code that picks its launch shape.
KERNEL_SOURCES = {
    "gemm_skinny_kernel": "gemm_skinny.cu",
    "gemm_wide_kernel": "gemm_wide.cu",
    "gemm_wide_pair_kernel": "gemm_wide_pair.cu",
    "shrink_tc_kernel": "shrink.cu",
    "plan_kernel": "plan.cu",
}


def src_digest(kernel: str) -> str:
    """Digest of the CUDA sources a kernel's traffic depends on, with comments
    and blank lines dropped, so a comment-only edit (or a change to another
    kernel) keeps the recorded ncu traffic valid."""
    import re
    h = hashlib.sha256()
    d = os.path.join(ROOT, "adapter_gemm_gb300", "csrc")
    for f in sorted([KERNEL_SOURCES[kernel], "kernels.h", "ptx.cuh", "api.cu"]):
        text = open(os.path.join(d, f), encoding="utf-8").read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        lines = [ln.rstrip() for ln in text.splitlines() if ln.strip()]
        h.update(f.encode())
        h.update("\n".join(lines).encode())
    return h.hexdigest()[:16]


def ncu_traffic(config: str):
    """dram read+write bytes per launch of the dominant kernel from a committed
    ncu summary, if it was taken on that kernel's current sources."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(config)
    if not d or d.get("src_sha") != src_digest(d["kernel"]):
        return None
    return float(d["dram_bytes_per_launch"])


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None
        self.spans = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thr = threading.Thread(target=self._read, daemon=True)
            self.thr.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), line.strip()))

    def span(self, t0: float, t1: float):
        """Mark [t0, t1] (time.time()) as a timed region."""
        self.spans.append((t0, t1))

    def stop(self):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, spans=None):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        spans = self.spans if spans is None else spans
        inside = [r for t, r in self.rows if any(a - 0.2 <= t <= b + 0.2 for a, b in spans)]
        use = inside or [self.rows[-1][1]]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in use:
            f = [v.strip() for v in r.split(",")]
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(use)}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(ms: float, device=None) -> float:
    """The largest of the ranks' times (a whole job ends with its slowest
    replica); the value itself on a single process. `device` is where the
    process group's backend keeps tensors (a CUDA device for NCCL, None for
    gloo)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(ms)
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: int, steps: int, world: int, ms: float) -> float:
    """Units all replicas processed per second: every rank runs the same
    per-GPU workload (weak scaling), and the job takes the slowest rank's
    time `ms` for `steps` steps."""
    return units_per_rank * steps * world / (ms / 1e3)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# --------------------------------------------------------------- oracle leg --

def oracle_tokens_per_s(w, seconds: float):
    """Time the CPU oracle, as it stands, on whole steps of the workload until
    `seconds` of work is done; returns (tokens/s, threads, sample text)."""
    from oracle import lora_oracle as O
    from adapter_gemm_gb300 import workloads as WL
    try:
        from threadpoolctl import threadpool_info
        threads = max([i.get("num_threads", 1) for i in threadpool_info()] or [os.cpu_count()])
    except ImportError:
        threads = os.cpu_count()
    prep = []
    for t in w.targets:
        x = WL.rows_input(w, t).double().numpy()
        prep.append((x, t.W.double().numpy(), t.A.double().numpy(), t.B.double().numpy(), t.rank, t.alpha))
    T = w.T
    # bounded sample: whole steps if one is cheap, else a subset of rows
    rows = None
    t0 = time.perf_counter()
    x, W_, A_, B_, r_, a_ = prep[0]
    O.lora_linear(x[:1], W_, A_, B_, r_, a_, w.ids[:1])
    one_row = time.perf_counter() - t0
    est_step = one_row * T * len(prep)
    if est_step > seconds / 3:
        n = max(1, int(T * (seconds / 3) / est_step))
        rows = np.linspace(0, T - 1, n).astype(np.int64)
    done_rows = 0
    t0 = time.perf_counter()
    reps = 0
    while True:
        for (x, W_, A_, B_, r_, a_) in prep:
            O.lora_linear(x, W_, A_, B_, r_, a_, w.ids, rows=rows)
        done_rows += T if rows is None else len(rows)
        reps += 1
        if time.perf_counter() - t0 >= seconds:
            break
    el = time.perf_counter() - t0
    what = "whole steps" if rows is None else f"{len(rows)} of {T} rows per step"
    sample = f"{reps} x ({what}) of {w.name}, all {len(prep)} target(s), fp64 numpy/BLAS"
    return done_rows / el, threads, sample


# --------------------------------------------------------------- GPU leg ----

class Runner:
    """One workload on the device: weights and pools in rotating copies, one
    plan per copy, and the step as a chain of library calls."""

    def __init__(self, w, dev, use_graph=True):
        import torch
        from adapter_gemm_gb300 import lora as L, workloads as WL
        self.torch, self.L, self.WL = torch, L, WL
        self.w, self.dev, self.use_graph = w, dev, use_graph
        T = w.T
        props = torch.cuda.get_device_properties(dev)
        l2 = int(getattr(props, "L2_cache_size", 126 * 2**20))

        # ---- device copies: rotate weights so the working set exceeds 2x L2
        per_copy = 0
        for t in w.targets:
            per_copy += t.W.numel() * 2 + t.A.numel() * 2 + t.B.numel() * 2
        n_copies = max(2, int(np.ceil(2.0 * l2 / max(per_copy, 1))) + 1)
        self.n_copies = n_copies = min(n_copies, 64)
        self.per_copy = per_copy

        self.xs = {}
        for t in w.targets:
            k = id(WL.input_for(w, t))
            if k not in self.xs:
                self.xs[k] = WL.input_for(w, t).to(dev)
        self.x0_key = id(w.x)
        self.ids = torch.from_numpy(w.ids).to(dev)
        # The step's calls: a target on its own, or targets that share x as
        # one call over their output slices (W stacked by rows, one pool per
        # slice).
        self.units = units = w.units()
        self.u_name = ["+".join(w.targets[i].name for i in u) for u in units]
        self.u_dout = [[w.targets[i].d_out for i in u] for u in units]
        self.u_key = [id(WL.input_for(w, w.targets[u[0]])) for u in units]
        base_units = []
        for u in units:
            W = torch.cat([w.targets[i].W for i in u], 0).to(dev)
            pools = []
            for i in u:
                t = w.targets[i]
                pool = L.Pool(w.S, w.R_max, t.d_in, t.d_out, device=dev)
                pool.load_padded(t.A, t.B, t.rank, t.alpha)
                pools.append(pool)
            base_units.append((W, pools))
        self.copies = [base_units]
        for _ in range(n_copies - 1):
            c = []
            for (W, pools) in base_units:
                p2s = []
                for pool in pools:
                    p2 = L.Pool(w.S, w.R_max, pool.d_in, pool.d_out, device=dev)
                    p2.A.copy_(pool.A); p2.B.copy_(pool.B); p2.scale.copy_(pool.scale); p2.rank.copy_(pool.rank)
                    p2s.append(p2)
                c.append((W.clone(), p2s))
            self.copies.append(c)
        self.d_cap = max(t.d_in for t in w.targets)
        self.plans = [L.Plan(T, w.S, w.R_max, self.d_cap, device=dev) for _ in range(n_copies)]
        self.ys = [torch.empty((T, sum(d)), dtype=torch.bfloat16, device=dev) for d in self.u_dout]
        # The chain: the call whose output has x's width feeds the next step's
        # x (the last such call: the down projection in the layer sweep).
        self.chain_unit = None
        if w.sel is None:
            for j, d in enumerate(self.u_dout):
                if sum(d) == w.x.shape[1]:
                    self.chain_unit = j
        self.ychain = [torch.empty_like(self.ys[self.chain_unit]) for _ in range(2)] \
            if self.chain_unit is not None else None
        self.sel_dev = torch.from_numpy(w.sel).to(dev) if w.sel is not None else None
        self.x_rows = [torch.empty((T, w.targets[u[0]].d_in), dtype=torch.bfloat16, device=dev) for u in units] \
            if w.sel is not None else None
        torch.cuda.synchronize()
        self.G = n_copies * max(1, -(-16 // n_copies))
        self.big, self.singles = None, []

        # library kernels per step and per call
        for i in range(3):
            self.step(i, 0)
        torch.cuda.synchronize()
        n0 = L.launch_count()
        self.step(0, 0)
        self.launches_per_step = L.launch_count() - n0
        self.u_launch = []
        for j in range(len(units)):
            n0 = L.launch_count()
            W, pools = self.copies[0][j]
            self.call(j, self.xs[self.u_key[j]], W, pools, self.plans[0], self.ys[j])
            self.u_launch.append(L.launch_count() - n0)
        torch.cuda.synchronize()

    def call(self, j, x, W, pools, plan, y):
        L = self.L
        if self.sel_dev is not None:
            L.linear_rows(x, self.sel_dev, W, pools[0], plan, self.x_rows[j], y)
        elif len(pools) == 1:
            L.linear(x, W, pools[0], plan, y)
        else:
            L.linear_sliced(x, W, self.u_dout[j], pools, plan, y)

    def step(self, i, j):
        """Step i of the weight rotation, j-th of its chain (j = 0 reads the
        resident x; j > 0 reads step j - 1's chained output)."""
        c = i % self.n_copies
        self.plans[c].build(self.ids)
        x_step = self.xs[self.x0_key] if (j == 0 or self.ychain is None) else self.ychain[(j - 1) % 2]
        for u, (W, pools) in enumerate(self.copies[c]):
            x = x_step if self.u_key[u] == self.x0_key else self.xs[self.u_key[u]]
            y = self.ychain[j % 2] if u == self.chain_unit else self.ys[u]
            self.call(u, x, W, pools, self.plans[c], y)

    def capture(self, fn):
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream(self.dev)
        s.wait_stream(torch.cuda.current_stream(self.dev))
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                fn()
        torch.cuda.current_stream(self.dev).wait_stream(s)
        return g

    def graphs(self):
        """One graph of a G-step chain over the copies in rotation, and a
        one-step graph per copy for the remainder: the host launches one graph
        per G steps and never starves the GPU."""
        if not self.use_graph or self.big is not None:
            return
        self.big = self.capture(lambda: [self.step(i, i) for i in range(self.G)])
        self.singles = [self.capture(lambda c=c: self.step(c, 0)) for c in range(self.n_copies)]
        self.big.replay()
        for g in self.singles:
            g.replay()
        self.torch.cuda.synchronize()

    def run_steps(self, k):
        if not self.use_graph:
            for i in range(k):
                self.step(i, i % self.G)
            return
        for _ in range(k // self.G):
            self.big.replay()
        for i in range(k % self.G):
            self.singles[i % self.n_copies].replay()

    def time_steps(self, k, world=1):
        """ms for k steps, device time on this stream, max over ranks."""
        torch = self.torch
        barrier(world)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        t0 = time.time()
        e0.record()
        self.run_steps(k)
        e1.record()
        torch.cuda.synchronize()
        t1 = time.time()
        barrier(world)
        return max_over_ranks(e0.elapsed_time(e1), self.dev), (t0, t1)

    def kernel_times(self, ksteps):
        """Per call, the mean time of its GEMM launch (of all kernels of a
        sliced call that runs per slice), from a pair of events the library
        records on the launch stream right around it. The launches are queued
        behind a sleep kernel, so the GPU runs them back to back and the
        intervals hold GPU time only; a chunk whose sleep ended before the
        host finished queueing is redone with a longer sleep."""
        torch, L = self.torch, self.L
        nt = len(self.units)
        per = np.zeros(nt)
        evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in self.units] for _ in range(ksteps)]
        for row in evs:            # torch times only events it has recorded once itself;
            for a, b in row:       # the library's later records on the same handles win
                a.record()
                b.record()
        torch.cuda.synchronize()
        sleep_cycles = int(4e7)
        chunk, i0, starved = 8, 0, 0
        while i0 < ksteps:
            n_ch = min(chunk, ksteps - i0)
            torch.cuda._sleep(sleep_cycles)
            slept = torch.cuda.Event()
            slept.record()
            for i in range(i0, i0 + n_ch):
                c = i % self.n_copies
                self.plans[c].build(self.ids)
                for j, (W, pools) in enumerate(self.copies[c]):
                    a, b = evs[i][j]
                    L.profile_gemm_events(a, b)
                    self.call(j, self.xs[self.u_key[j]], W, pools, self.plans[c], self.ys[j])
            L.profile_gemm_events(None, None)
            if slept.query():                 # the GPU caught up with the host
                starved += 1
                torch.cuda.synchronize()
                if sleep_cycles < int(2e9):
                    sleep_cycles *= 4
                    continue
            i0 += n_ch
        torch.cuda.synchronize()
        for i in range(ksteps):
            for j in range(nt):
                a, b = evs[i][j]
                per[j] += a.elapsed_time(b)
        return per / ksteps, starved

    def roofline(self, per_ms, config_name):
        """The dominant call's kernel against its roof, and the step's roof."""
        from adapter_gemm_gb300 import cost
        w, L = self.w, self.L
        T = w.T
        hbm, tf_burst, tf_sus, src = peaks()
        j = int(np.argmax(per_ms))
        u = self.units[j]
        td = w.targets[u[0]]
        ranks = [w.targets[i].rank for i in u]
        n_dom = sum(self.u_dout[j])
        all_kernels = len(u) > 1 and self.u_launch[j] > 1
        if self.u_launch[j] == 1 or all_kernels:
            # one kernel does the whole layer (shrink fused in), or the timing
            # brackets every kernel of the call: the layer's work
            work = cost.sliced_layer(T, td.d_in, self.u_dout[j], w.ids, ranks)
        else:
            work = cost.sliced_gemm_kernel(T, td.d_in, self.u_dout[j], w.ids, ranks)
        t_k = per_ms[j] / 1e3
        _, bound = cost.roofline_time(work, tf_burst, hbm)
        if bound == "hbm":
            achieved, peak, unit = work.bytes / t_k / 1e9, hbm, "GB/s"
        else:
            achieved, peak, unit = work.flops / t_k / 1e12, tf_burst, "TFLOP/s"
        kname = ("gemm_skinny_kernel", "gemm_wide_kernel", "gemm_wide_pair_kernel")[
            L.kernel_for(T, td.d_in, n_dom, self.copies[0][j][1][0])]
        if all_kernels:
            kname = f"all {self.u_launch[j]} kernels of the per-slice calls"
        roof = {"bound": bound, "achieved": round(achieved, 1), "peak": peak, "unit": unit,
                "frac": round(achieved / peak, 4), "traffic": ncu_traffic(config_name),
                "kernel": kname, "target": self.u_name[j], "kernel_us": round(t_k * 1e6, 3),
                "per_target_us": {nm: round(v * 1e3, 3) for nm, v in zip(self.u_name, per_ms)},
                "algorithmic_bytes": work.bytes, "algorithmic_flops": work.flops,
                "work": "whole layer (shrink + GEMM + expand)" if (self.u_launch[j] == 1 or all_kernels)
                        else "GEMM with the fused expand",
                "timing": "events around each launch, queued behind a sleep kernel (no host gaps, no overlap)",
                "peak_source": f"{src} ({'hbm_gbs' if bound == 'hbm' else 'bf16_tflops, burst: timed in isolation'})"}
        t_roof = 0.0
        for uu, d in zip(self.units, self.u_dout):
            lw = cost.sliced_layer(T, w.targets[uu[0]].d_in, d, w.ids, [w.targets[i].rank for i in uu])
            t_roof += cost.roofline_time(lw, tf_burst, hbm)[0]
        total_flops = sum(cost.layer(T, t.d_in, t.d_out, w.ids, t.rank).flops for t in w.targets)
        return roof, t_roof, total_flops

    def timing_label(self):
        if self.ychain is not None:
            return (f"chained: step j+1 reads step j's {self.u_name[self.chain_unit]} output as x "
                    f"(graphs of {self.G}-step chains)")
        return ("independent steps on one resident x (no shape-compatible chain); each call's first "
                "kernel waits for the kernel ahead before reading x")

    def e2e(self, steps, world):
        """End to end with host buffers: every step copies its inputs in from
        pinned host memory and its outputs back out, inside the timed region.
        Steps rotate over four streams, each with its own staging buffers and
        plan, so one step's copies overlap the others' kernels; all streams
        are captured in the same graphs. A workload of one call goes through
        the C ABI's host-buffer entry point (lora_linear_host); others copy
        with torch and call the device entry points."""
        torch, L, w, dev = self.torch, self.L, self.w, self.dev
        T = w.T
        NP = 4
        estreams = [torch.cuda.Stream(dev) for _ in range(NP)]
        eplans = [L.Plan(T, w.S, w.R_max, self.d_cap, device=dev) for _ in range(NP)]
        hx = {k: v.cpu().pin_memory() for k, v in self.xs.items()}
        hids = torch.from_numpy(w.ids).pin_memory()
        hy = [[torch.empty_like(y, device="cpu").pin_memory() for y in self.ys] for _ in range(NP)]
        dx = [{k: torch.empty_like(v) for k, v in self.xs.items()} for _ in range(NP)]
        dids = [torch.empty_like(self.ids) for _ in range(NP)]
        dy = [[torch.empty_like(y) for y in self.ys] for _ in range(NP)]
        host_api = len(self.units) == 1 and len(self.units[0]) == 1 and w.sel is None

        def e2e_step(i):
            b, c = i % NP, i % self.n_copies
            st = estreams[b]
            if host_api:
                W, pools = self.copies[c][0]
                L.linear_host(hx[self.u_key[0]], W, hy[b][0], dx[b][self.u_key[0]], dy[b][0], pools[0], eplans[b],
                              hids, dids[b], stream=st)
                return
            with torch.cuda.stream(st):
                for k in hx:
                    dx[b][k].copy_(hx[k], non_blocking=True)
                dids[b].copy_(hids, non_blocking=True)
                eplans[b].build(dids[b])
                for j, (W, pools) in enumerate(self.copies[c]):
                    self.call(j, dx[b][self.u_key[j]], W, pools, eplans[b], dy[b][j])
                    hy[b][j].copy_(dy[b][j], non_blocking=True)

        def capture_e2e(n):
            g = torch.cuda.CUDAGraph()
            s0 = torch.cuda.Stream(dev)
            s0.wait_stream(torch.cuda.current_stream(dev))
            with torch.cuda.stream(s0):
                with torch.cuda.graph(g, stream=s0):
                    for es in estreams:
                        es.wait_stream(s0)
                    for i in range(n):
                        e2e_step(i)
                    for es in estreams:
                        s0.wait_stream(es)
            torch.cuda.current_stream(dev).wait_stream(s0)
            return g

        for es in estreams:
            es.wait_stream(torch.cuda.current_stream(dev))
        for i in range(3):
            e2e_step(i)
        for es in estreams:
            torch.cuda.current_stream(dev).wait_stream(es)
        torch.cuda.synchronize()
        G = self.G
        esteps = G * max(1, min(steps, 512) // G)
        ebig = None
        if self.use_graph:
            ebig = capture_e2e(G)
            ebig.replay()
            torch.cuda.synchronize()
        f0 = torch.cuda.Event(enable_timing=True)
        f1 = torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        f0.record()
        if ebig is not None:
            for _ in range(esteps // G):
                ebig.replay()
        else:
            for es in estreams:
                es.wait_stream(torch.cuda.current_stream(dev))
            for i in range(esteps):
                e2e_step(i)
            for es in estreams:
                torch.cuda.current_stream(dev).wait_stream(es)
        f1.record()
        torch.cuda.synchronize()
        barrier(world)
        ems = max_over_ranks(f0.elapsed_time(f1), dev)
        bi = sum(v.numel() * v.element_size() for v in hx.values()) + hids.numel() * 4
        bo = sum(v.numel() * v.element_size() for v in hy[0])
        return {"value": round(job_throughput(T, esteps, world, ems), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": int(bi), "d2h_bytes_per_step": int(bo), "steps": esteps,
                "ms_per_step": round(ems / esteps, 6),
                "api": "lora_linear_host" if host_api else "host copies + lora_plan / lora_linear",
                "pipelines": NP}


def measure_config(name, args, dev, world, clocks, seconds):
    """A per_config entry: the step (chained where possible), its roofline,
    and the dominant kernel timed in isolation."""
    import torch
    from adapter_gemm_gb300 import workloads as WL
    w = WL.by_name(name)
    r = Runner(w, dev, use_graph=not args.no_graph)
    r.graphs()
    r.run_steps(max(args.warmup, 3))
    ms1, _ = r.time_steps(r.G, 1)
    est = max(ms1 / r.G, 1e-3)
    k = int(np.clip(seconds * 1e3 / est, 2 * r.G, 20000)) // r.G * r.G
    ms, span = r.time_steps(k, world)
    clocks.span(*span)
    per_ms, _ = r.kernel_times(min(args.kernel_steps, 40))
    roof, t_roof, flops = r.roofline(per_ms, name)
    ms_step = ms / k
    out = {"T": w.T, "us_per_step": round(ms_step * 1e3, 3),
           "tokens_per_s": round(job_throughput(w.T, k, world, ms), 1),
           "tflops": round(flops / (ms_step / 1e3) / 1e12, 2),
           "step_roofline_frac": round(t_roof / (ms_step / 1e3), 4),
           "kernel": roof["kernel"], "kernel_target": roof["target"], "kernel_us": roof["kernel_us"],
           "kernel_frac": roof["frac"], "kernel_bound": roof["bound"], "traffic": roof["traffic"],
           "kernels_per_step": r.launches_per_step, "steps": k, "timing": r.timing_label()}
    del r
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def main(argv=None):
    args = parse(argv)
    rank, world, local = dist_env()
    import torch

    if args.impl == "reference":
        return run_reference(args, rank, world)

    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(dev)

    from adapter_gemm_gb300 import build as B
    B.build()
    from adapter_gemm_gb300 import lora as L, workloads as WL

    if args.profile_steps > 0:
        # The steps the timed run replays as graphs, launched eagerly (the
        # same kernels, one launch each), with no timing around them.
        w = WL.by_name(args.config)
        r = Runner(w, dev, use_graph=False)
        n0 = L.launch_count()
        r.run_steps(3 + args.profile_steps)
        torch.cuda.synchronize()
        assert L.last_device_error() == 0, "a kernel gave up a bounded wait"
        if rank == 0:
            print(json.dumps({"profile_steps": args.profile_steps, "warmup": 3, "workload": w.name,
                              "launches": L.launch_count() - n0,
                              "launches_per_step": r.launches_per_step}), flush=True)
        return 0

    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    clocks.start()
    time.sleep(0.3)

    # ---- headline workload
    w = WL.by_name(args.config)
    T = w.T
    r = Runner(w, dev, use_graph=not args.no_graph)
    r.graphs()
    r.run_steps(max(args.warmup, 3))
    torch.cuda.synchronize()
    ms, span = r.time_steps(args.steps, world)
    clocks.span(*span)
    head_clock = clocks.summary([span])
    ms_per_step = ms / args.steps
    value = job_throughput(T, args.steps, world, ms)
    per_ms, starved = r.kernel_times(max(10, min(args.kernel_steps, args.steps)))
    roof, t_roof, total_flops = r.roofline(per_ms, args.config)
    roof["starved_chunks_redone"] = starved
    e2e = r.e2e(args.steps, world)
    assert L.last_device_error() == 0, "a kernel gave up a bounded wait"
    head = {"T": T, "us_per_step": round(ms_per_step * 1e3, 3), "tokens_per_s": round(value, 1),
            "tflops": round(total_flops / (ms_per_step / 1e3) / 1e12, 2),
            "step_roofline_frac": round(t_roof / (ms_per_step / 1e3), 4), "kernel": roof["kernel"],
            "kernel_target": roof["target"], "kernel_us": roof["kernel_us"], "kernel_frac": roof["frac"],
            "kernel_bound": roof["bound"], "traffic": roof["traffic"], "kernels_per_step": r.launches_per_step,
            "steps": args.steps, "timing": r.timing_label()}
    groups = [r.u_name[j] for j, u in enumerate(r.units) if len(u) > 1]
    config = {"workload": w.name, "T": T, "targets": [[t.name, t.d_in, t.d_out] for t in w.targets],
              "sliced_calls": groups, "slots": w.S, "R_max": w.R_max, "parallelism": f"replicas x{world}",
              "l2": f"{r.n_copies} rotating weight/pool copies ({r.n_copies * r.per_copy / 2**20:.0f} MiB > 2x L2)",
              "launch": f"CUDA graphs of {r.G} steps" if not args.no_graph else "eager",
              "timing": r.timing_label()}
    launches_per_step = r.launches_per_step
    del r
    torch.cuda.synchronize()
    torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1:
        v, cores, sample = oracle_tokens_per_s(w, args.cpu_seconds)
        cpu = {"value": round(v, 2), "unit": "tokens/s", "cores": int(cores), "kind": "oracle", "sample": sample}
    del w

    # ---- every configuration of the parity set
    per_config = {}
    for name in [n for n in args.per_config.split(",") if n]:
        if name == args.config:
            per_config[name] = head
            continue
        per_config[name] = measure_config(name, args, dev, world, clocks, args.config_seconds)
    assert L.last_device_error() == 0, "a kernel gave up a bounded wait"
    clocks.stop()

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; random-init weights and adapters)",
        "config": config,
        "tflops": head["tflops"],
        "step_roofline_frac": head["step_roofline_frac"],
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": head_clock,
        "clocks_all_timed_regions": clocks.summary(),
        "per_config": per_config,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_reference(args, rank, world):
    """The reference arm is the CPU oracle, timed as it stands.

    Each step runs the oracle on a bounded sample of the batch's rows (every
    target), sized so that warm-up plus timed steps take about
    --reference-seconds in all; value = sampled rows / time."""
    if rank != 0:
        return
    from oracle import lora_oracle as O
    from adapter_gemm_gb300 import workloads as WL
    w = WL.by_name(args.config)
    prep = []
    for t in w.targets:
        x = WL.rows_input(w, t).double().numpy()
        prep.append((x, t.W.double().numpy(), t.A.double().numpy(), t.B.double().numpy(), t.rank, t.alpha))
    T = w.T

    def run_rows(rows):
        for (x, W_, A_, B_, r_, a_) in prep:
            O.lora_linear(x, W_, A_, B_, r_, a_, w.ids, rows=rows)

    run_rows(np.arange(1))                      # first call pays one-off costs
    probe = np.arange(min(T, 4))
    t0 = time.perf_counter()
    run_rows(probe)
    per_row = max((time.perf_counter() - t0) / len(probe), 1e-6)
    per_step = max(0.005, args.reference_seconds / max(1, args.steps + args.warmup))
    n = int(max(1, min(T, per_step / per_row)))
    rows = np.linspace(0, T - 1, n).astype(np.int64)
    for _ in range(args.warmup):
        run_rows(rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run_rows(rows)
    el = time.perf_counter() - t0
    value = n * args.steps / el
    try:
        from threadpoolctl import threadpool_info
        cores = max([i.get("num_threads", 1) for i in threadpool_info()] or [os.cpu_count()])
    except ImportError:
        cores = os.cpu_count()
    sample = (f"{n} of {T} rows per step of {w.name}, all {len(prep)} target(s), "
              f"fp64 numpy/BLAS, {args.steps} timed steps")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * el / max(1, args.steps), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)", "config": {"workload": w.name, "T": T},
        "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": int(cores), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
