#!/usr/bin/env python
"""Benchmark of the owner-local optimizer step (MatrixFSDP: Communication-Free
Matrix Optimizers Under ZeRO-3 Parameter Sharding -- Abstract).

One step = one pass of the whole hot path over one owner set: the momentum /
segment-view / norm phase, five Newton-Schulz iterations (Gram, polynomial,
update products on tcgen05 tensor cores) and AdamW over the rank's packed tail,
all through the C ABI (libmfsdp.so) on one stream.  Default workload: the
Llama-3-8B-shaped owner set (one rank of eight: 28 matrices, 872.4M bf16
gradient elements with Student-t(3) entries, 32,768-element RMSNorm tail).

Prints one JSON line.  `value` is the device-timed owner-step latency in ms
(inputs resident in HBM; every input is larger than L2, so no flush is needed),
`e2e` the same latency through the same API with the gradient copied in from
pinned host memory and the update copied back every step.  The supplementary
block times, in the same process, the momentum phase alone, the owner-segment
reduce, AdamW over a 50M-element tail and the other four workloads' owner sets
(owner-step ms, Newton-Schulz TFLOP/s, momentum and AdamW GB/s, each against
its measured peak).  `cpu_baseline` is the fp64 oracle on the host cores: one
matrix of every shape of the owner set timed, times its count, plus the whole
tail.  `--impl reference` times that oracle instead, one shape per step.

Under torchrun (N > 1) each GPU runs the owner set of a different simulated
rank (weak scaling: no collective on the data path; a barrier and a max over
ranks bracket the timed region).
"""
from __future__ import annotations

import argparse
import gc
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from matrix_optimizers_under_gb300 import workloads as W  # noqa: E402

METRIC = "owner-step ms; Newton–Schulz TFLOP/s (% BF16 peak); AdamW-tail GB/s (% HBM)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM bytes (read + write) of one Newton-Schulz kernel launch per owner set,
# from an ncu capture of dram__bytes_read.sum + dram__bytes_write.sum, keyed
# by a digest of the kernel's sources (ns_source_digest): a kernel changed
# since its capture reports null traffic until it is captured again.
NS_GEMM_TRAFFIC = {("26400a1bdf0b290e", "llama3_8b_rank"): 28.58e9, ("26400a1bdf0b290e", "llama_1p3b_rank"): 5.48e9}
# Share of the same launch's elapsed cycles with the tensor pipe active
# (sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_elapsed), keyed alike.
NS_TENSOR_ACTIVE = {("26400a1bdf0b290e", "llama3_8b_rank"): 0.9134, ("26400a1bdf0b290e", "llama_1p3b_rank"): 0.8354}

# The sources that make up the Newton-Schulz kernel.
NS_SOURCES = ("ns_gemm.cu", "ptx.cuh", "mfsdp_internal.h")


# --------------------------------------------------------------------------- helpers
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def strip_code(text: str) -> str:
    """C/C++ source without comments and with whitespace runs collapsed, so that
    editing a comment does not change what the digest says about the code."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def ns_source_digest(sources=None) -> str:
    """First 16 hex digits of the SHA-256 of the Newton-Schulz kernel's sources
    (comments and layout ignored).  `sources`: {name: text}, default the files."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "matrix_optimizers_under_gb300", "csrc")
    for name in NS_SOURCES:
        if sources is not None:
            text = sources[name]
        else:
            with open(os.path.join(csrc, name)) as f:
                text = f.read()
        h.update(strip_code(text).encode())
    return h.hexdigest()[:16]


def ns_flops(rows: int, cols: int, steps: int) -> int:
    s, l = min(rows, cols), max(rows, cols)
    return steps * (4 * s * s * l + 2 * s ** 3)


def simulated_rank(heavy: int, rank: int, planner_world: int) -> int:
    """Owner set a GPU benches under torchrun: the heaviest planner rank on GPU 0,
    the next ones on the other GPUs (weak scaling: one owner set per GPU)."""
    return (heavy + rank) % planner_world


def max_over_ranks(value: float, device=None) -> float:
    """The slowest rank's figure (the step ends when every owner set is done)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def heaviest_rank(plan) -> int:
    world = len(plan.rank_matrix_elems)
    cost, tail = [0] * world, [0] * world
    for s in plan.matrix_shards:
        cost[s.owner] += s.cost
    for s in plan.tail_shards:
        tail[s.owner] += s.numel
    return min(range(world), key=lambda r: (-cost[r], tail[r], r))


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max((num(r[3]) or 0.0) for r in rows)}


# --------------------------------------------------------------------------- CPU oracle
def shape_groups(shards):
    """The owner set's distinct (rows, cols), each with its count and the
    lowest param id of that shape (the one timed), largest work first."""
    groups = {}
    for s in shards:
        g = groups.setdefault((s.rows, s.cols), [0, s.param_id])
        g[0] += 1
        g[1] = min(g[1], s.param_id)
    return sorted(((rc, c, pid) for rc, (c, pid) in groups.items()),
                  key=lambda x: (-ns_flops(x[0][0], x[0][1], 5), x[0]))


def oracle_matrix_seconds(w, rows, cols, param_id):
    """Wall-clock of the fp64 oracle's owner step (momentum, Frobenius
    normalisation, Newton-Schulz) on one matrix held in a flat buffer as
    stored (bf16 bits or fp32), from zero momentum."""
    from oracle.muon import muon_owner_step_ref
    a, b, c = w.ns_coeffs
    flat = W.grad_storage(w, param_id).reshape(-1)
    shard = [dict(param_id=param_id, offset=0, rows=rows, cols=cols)]
    t0 = time.perf_counter()
    muon_owner_step_ref(shard, flat, w.grad_dtype, np.zeros(rows * cols), w.beta, w.nesterov, w.ns_steps,
                        a, b, c, w.ns_eps)
    return time.perf_counter() - t0


def oracle_tail_seconds(w, tail_n):
    """Wall-clock of the fp64 oracle's AdamW over a whole tail of tail_n elements."""
    from oracle import adamw_ref
    if not tail_n:
        return 0.0
    rng = np.random.default_rng(0)
    p = rng.standard_normal(tail_n) * w.tail_scale
    g = rng.standard_normal(tail_n) * w.tail_scale
    t0 = time.perf_counter()
    adamw_ref(p, g, np.zeros(tail_n), np.zeros(tail_n), w.lr, w.betas[0], w.betas[1], w.adam_eps,
              w.weight_decay, w.step)
    return time.perf_counter() - t0


def oracle_owner_step_estimate(w, shards, tail_n):
    """The fp64 oracle's owner step on the host cores, per shape: one matrix of
    every distinct shape timed once, each time multiplied by that shape's count
    (the oracle's work and time per matrix depend on the shape alone), plus
    AdamW over the whole tail, timed.  Returns (ms, description, seconds spent)."""
    t_all = time.perf_counter()
    groups = shape_groups(shards)
    per = []
    ms = 0.0
    for (rows, cols), count, pid in groups:
        sec = oracle_matrix_seconds(w, rows, cols, pid)
        per.append(f"{rows}x{cols}: {sec * 1e3:.0f} ms x {count}")
        ms += sec * 1e3 * count
    tail_sec = oracle_tail_seconds(w, tail_n)
    ms += tail_sec * 1e3
    desc = (f"fp64 NumPy oracle: one matrix of each of the {len(groups)} shapes of the {len(shards)}-matrix owner "
            f"set timed once (momentum + normalisation + Newton-Schulz from a flat buffer) and multiplied by the "
            f"shape's count [{'; '.join(per)}], plus AdamW over the whole {tail_n}-element tail ({tail_sec * 1e3:.0f} ms)")
    return ms, desc, time.perf_counter() - t_all


def oracle_owner_step_full(w, shards, tail_n):
    """The fp64 oracle's whole owner step on the host cores: every matrix of the
    owner set (momentum, normalisation, Newton-Schulz from one flat buffer, as
    stored) and AdamW over the whole tail, timed once.  Minutes for the large
    owner sets.  Returns (ms, description, seconds spent)."""
    from oracle.muon import muon_owner_step_ref
    a, b, c = w.ns_coeffs
    numel = max(s.offset + s.rows * s.cols for s in shards) if shards else 0
    flat = np.zeros(numel, np.uint16 if w.grad_dtype == "bf16" else np.float32)
    for s in shards:
        flat[s.offset:s.offset + s.rows * s.cols] = W.grad_storage(w, s.param_id).reshape(-1)
    table = [dict(param_id=s.param_id, offset=s.offset, rows=s.rows, cols=s.cols) for s in shards]
    t0 = time.perf_counter()
    muon_owner_step_ref(table, flat, w.grad_dtype, np.zeros(numel), w.beta, w.nesterov, w.ns_steps, a, b, c, w.ns_eps)
    sec = time.perf_counter() - t0
    tail_sec = oracle_tail_seconds(w, tail_n)
    ms = (sec + tail_sec) * 1e3
    desc = (f"fp64 NumPy oracle: the whole {len(shards)}-matrix owner step from one flat buffer "
            f"({sec:.1f} s) plus AdamW over the whole {tail_n}-element tail ({tail_sec * 1e3:.0f} ms), measured once")
    return ms, desc, sec + tail_sec


def cpu_threads():
    try:
        from threadpoolctl import threadpool_info
        info = threadpool_info()
        if info:
            return int(max(i.get("num_threads", 1) for i in info))
    except Exception:
        pass
    return os.cpu_count() or 1


def blas_info():
    """BLAS library and thread count NumPy uses (for the CPU-baseline record):
    from threadpoolctl where it is installed, else NumPy's build configuration
    and the usual thread-count variables."""
    try:
        from threadpoolctl import threadpool_info
        info = [i for i in threadpool_info() if i.get("user_api") == "blas"]
        if info:
            return {"blas": info[0].get("internal_api"), "threads": info[0].get("num_threads")}
    except Exception:
        pass
    blas = None
    try:
        blas = np.show_config(mode="dicts")["Build Dependencies"]["blas"]["name"]
    except Exception:
        pass
    threads = None
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            threads = int(os.environ[var])
            break
    return {"blas": blas, "threads": threads if threads is not None else os.cpu_count()}


# --------------------------------------------------------------------------- reference arm
def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1 and rank != 0:
        return 0
    w = W.get(args.workload)
    from oracle.planner import plan_owners_ref, heaviest_rank_ref
    plan = plan_owners_ref(w.param_table(), w.world, w.ns_steps, w.align_elems)
    r = heaviest_rank_ref(plan)

    class S:  # adapter with attribute access
        def __init__(self, d):
            self.__dict__.update(d)
    shards = [S(d) for d in plan["matrix_shards"] if d["owner"] == r]
    tail_n = plan["rank_tail_numel"][r]
    groups = shape_groups(shards)
    # Step i times one shape (in rotation) and the tail; the owner-step figure is
    # every shape's mean time times its count, plus the tail's.
    times = {g[0]: [] for g in groups}
    tails = []
    t_total = time.perf_counter()
    for i in range(args.warmup + args.steps):
        (rows, cols), count, pid = groups[i % len(groups)]
        sec = oracle_matrix_seconds(w, rows, cols, pid)
        tsec = oracle_tail_seconds(w, tail_n)
        if i >= args.warmup:
            times[(rows, cols)].append(sec)
            tails.append(tsec)
    for (rows, cols), count, pid in groups:         # fewer timed steps than shapes
        if not times[(rows, cols)]:
            times[(rows, cols)].append(oracle_matrix_seconds(w, rows, cols, pid))
    value = sum(statistics.mean(times[rc]) * 1e3 * count for rc, count, _ in groups) + \
        (statistics.mean(tails) * 1e3 if tails else 0.0)
    cores = cpu_threads()
    desc = (f"fp64 NumPy oracle, one shape of the {len(shards)}-matrix owner set per step in rotation "
            f"({', '.join(f'{rc[0]}x{rc[1]} x {c}' for rc, c, _ in groups)}) plus AdamW over the whole "
            f"{tail_n}-element tail; the owner-step figure is each shape's mean time times its count plus "
            f"the tail's")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "ms", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(value, 3), "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "matrices": len(shards),
                       "elements": sum(s.rows * s.cols for s in shards), "ns_steps": w.ns_steps},
            "cpu_baseline": {"value": round(value, 3), "unit": "ms", "cores": cores, "kind": "oracle",
                             "estimated": True, "method": "per shape: measured time x count",
                             "sample": desc, "seconds": round(time.perf_counter() - t_total, 1),
                             **blas_info()},
            "e2e": {"value": round(value, 3), "unit": "ms", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------- our arm
class OwnerStep:
    """Device buffers of one owner set and its step through the C ABI: the
    momentum phase, the Newton-Schulz phase and AdamW over the packed tail, on
    the current stream (events between the phases when asked)."""

    def __init__(self, mfsdp, w, shards, numel, tail_numel, grad_np, dev, pin=False):
        import torch
        self.mfsdp, self.w, self.shards, self.tail_numel = mfsdp, w, shards, tail_numel
        self.stream = torch.cuda.current_stream()
        bf16 = w.grad_dtype == "bf16"
        host = torch.from_numpy(grad_np.view(np.int16) if bf16 else grad_np)
        self.grad_host = host.pin_memory() if pin else host
        if bf16:
            self.grad_host = self.grad_host.view(torch.bfloat16)
        self.grad = self.grad_host.to(dev)
        self.mom = torch.zeros(numel, dtype=torch.float32, device=dev)
        self.upd = torch.zeros(numel, dtype=torch.bfloat16, device=dev)
        self.ws = torch.empty(max(mfsdp.muon_workspace_bytes(shards), 1), dtype=torch.uint8, device=dev)
        rng = np.random.default_rng(w.seed)
        n = max(tail_numel, 1)
        self.tp = torch.from_numpy((rng.standard_normal(n) * w.tail_scale).astype(np.float32)).to(dev)
        tg = torch.from_numpy((rng.standard_normal(n) * w.tail_scale).astype(np.float32))
        self.tg_host = tg.pin_memory() if pin else tg
        self.tg = self.tg_host.to(dev)
        self.tm, self.tv = torch.zeros_like(self.tp), torch.zeros_like(self.tp)
        self.kw = dict(beta=w.beta, nesterov=w.nesterov, ns_steps=w.ns_steps, coeffs=w.ns_coeffs, eps=w.ns_eps)
        self.count = 0
        batches = math.ceil(len(shards) / 128) if shards else 0
        self.batches = batches
        # per batch of 128 matrices: momentum, norm finalise, one Newton-Schulz launch
        self.launches = 3 * batches + (1 if tail_numel else 0)

    def adamw(self, stream=None):
        w = self.w
        self.mfsdp.adamw_tail_step(self.tp, self.tg, self.tm, self.tv, lr=w.lr, beta1=w.betas[0], beta2=w.betas[1],
                                   eps=w.adam_eps, wd=w.weight_decay, step=self.count, stream=stream)

    def step(self, ev=None, stream=None):
        """One owner step on self.stream, or on `stream` (a capture stream)."""
        m = self.mfsdp
        s = stream or self.stream
        self.count += 1
        if ev:
            ev[0].record(s)
        if self.shards:
            m.muon_owner_step(self.shards, self.grad, self.mom, self.upd, self.ws, phases=m.PHASE_MOMENTUM,
                              stream=s, **self.kw)
        if ev:
            ev[1].record(s)
        if self.shards:
            m.muon_owner_step(self.shards, self.grad, self.mom, self.upd, self.ws, phases=m.PHASE_NEWTON_SCHULZ,
                              stream=s, **self.kw)
        if ev:
            ev[2].record(s)
        if self.tail_numel:
            self.adamw(stream=s)
        if ev:
            ev[3].record(s)

    def check_status(self, when):
        if not self.shards:
            return
        st, detail = self.mfsdp.muon_device_status(self.ws)
        if st != self.mfsdp.OK:
            raise RuntimeError(f"device status {when}: {self.mfsdp.status_string(st)} ({detail})")


def figures(mfsdp, step, ms, peaks):
    """Algorithmic rates of one owner set's phases (ms: mean phase times).
    Matrices whose gradient is all zero (the MoE set's unrouted experts) keep
    a zero momentum and skip every Newton-Schulz product, so their FLOPs are
    left out of both counts."""
    w, shards = step.w, step.shards
    active = [s for s in shards if s.param_id not in w.zero_params]
    flops, flops_exec = mfsdp.muon_step_flops(active, w.ns_steps) if active else (0, 0)
    elems = sum(s.rows * s.cols for s in shards)
    gsz = 2 if w.grad_dtype == "bf16" else 4
    mom_bytes = elems * (gsz + 4 + 4 + 2)
    peak_tf, hbm = peaks["bf16_tflops_sustained"], peaks["hbm_gbs"]
    ns_tf = flops / (ms["ns"] * 1e-3) / 1e12 if ms["ns"] > 0 else 0.0
    ns_tf_exec = flops_exec / (ms["ns"] * 1e-3) / 1e12 if ms["ns"] > 0 else 0.0
    mom_gbs = mom_bytes / (ms["momentum"] * 1e-3) / 1e9 if ms["momentum"] > 0 else 0.0
    adam_gbs = 28 * step.tail_numel / (ms["adamw"] * 1e-3) / 1e9 if ms["adamw"] > 0 and step.tail_numel else 0.0
    return {"momentum_ms": round(ms["momentum"], 4), "momentum_gbs": round(mom_gbs, 1),
            "momentum_frac_hbm": round(mom_gbs / hbm, 4), "momentum_bytes": mom_bytes,
            "newton_schulz_ms": round(ms["ns"], 4),
            "newton_schulz_tflops_executed": round(ns_tf_exec, 1),
            "newton_schulz_frac_bf16_executed": round(ns_tf_exec / peak_tf, 4),
            # The standard iteration's dense FLOPs over the measured time: the rate
            # a dense evaluation would need to match it.  Not executed work (the
            # symmetric products skip half their tiles and wide matrices iterate on
            # their Gram matrix), so it is not compared with the tensor peak.
            "newton_schulz_tflops_dense_equivalent": round(ns_tf, 1),
            "flops_dense": flops, "flops_executed": flops_exec,
            "flops_dense_definition": "T (4 s^2 l + 2 s^3) per s x l matrix (standard iteration, dense)",
            "adamw_ms": round(ms["adamw"], 4), "adamw_gbs": round(adam_gbs, 1),
            "adamw_frac_hbm": round(adam_gbs / hbm, 4)}


def time_resident(step, steps, warmup, sampler=None, barrier=None):
    """W untimed steps, then K steps timed with CUDA events on the launching
    stream (a synchronize on both sides); returns the total ms, per-phase mean
    ms and the per-step times."""
    import torch
    for _ in range(warmup):
        step.step()
    torch.cuda.synchronize()
    step.check_status("after warm-up")
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if sampler:
        sampler.start()
        time.sleep(0.4)
    if barrier:
        barrier()
    torch.cuda.synchronize()
    gc.collect()
    gc.disable()            # no collector pause while the host enqueues the timed steps
    t0.record(step.stream)
    for k in range(steps):
        step.step(evs[k])
    t1.record(step.stream)
    torch.cuda.synchronize()
    gc.enable()
    if barrier:
        barrier()
    clocks = sampler.stop() if sampler else None
    step.check_status("after the timed region")
    ms = {"momentum": sum(e[0].elapsed_time(e[1]) for e in evs) / steps,
          "ns": sum(e[1].elapsed_time(e[2]) for e in evs) / steps,
          "adamw": sum(e[2].elapsed_time(e[3]) for e in evs) / steps}
    per_step = sorted(e[0].elapsed_time(e[3]) for e in evs)
    return t0.elapsed_time(t1), ms, per_step, clocks


def time_graph(step, steps):
    """The same owner step captured once in a CUDA graph and replayed `steps`
    times back to back (3 untimed replays first): the device time of the step
    without the host's per-call work between its launches, which a small owner
    set's step is short enough to expose.  Returns ms per step."""
    import torch
    graph = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        step.step(stream=torch.cuda.current_stream())
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    stream = torch.cuda.current_stream()
    e0.record(stream)
    for _ in range(steps):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    step.check_status("after the graph replays")
    ms = e0.elapsed_time(e1) / steps
    del graph
    return ms


def run_ours(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    w = W.get(args.workload)

    from matrix_optimizers_under_gb300 import _build
    _build.ensure_built()
    from matrix_optimizers_under_gb300 import binding as mfsdp

    def owner_set(wl, r_offset):
        plan = mfsdp.plan_owners(wl.param_table(), wl.world, wl.ns_steps, wl.align_elems)
        heavy = heaviest_rank(plan)
        sim = simulated_rank(heavy, r_offset, wl.world)
        return plan, sim, plan.rank_matrices(sim), plan.rank_matrix_elems[sim], plan.rank_tail_elems[sim]

    plan, sim_rank, shards, numel, tail_numel = owner_set(w, rank)
    supp_names = [] if (rank != 0 or args.no_supplementary) else [n for n in W.ORDER if n != w.name]

    # The headline's gradient buffer is generated before the first CUDA call
    # (a spawn pool); the other owner sets' only after the headline's timed
    # regions, so that no host memory but the headline's own is held while
    # they run.
    t_gen = time.time()
    grad_np = W.owner_grad_buffer(w, shards, numel)
    t_gen = time.time() - t_gen

    import torch
    import torch.distributed as dist
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    peaks, peak_src = load_peaks()
    barrier = dist.barrier if world > 1 else None

    # ---------------------------------------------------------- timed region
    step = OwnerStep(mfsdp, w, shards, numel, tail_numel, grad_np, dev, pin=True)
    grad_bytes = grad_np.nbytes
    del grad_np                                  # the step holds a pinned copy
    total_ms, phase_ms, steps_ms, clocks = time_resident(step, args.steps, args.warmup, ClockSampler(local_rank),
                                                         barrier)
    step_ms = max_over_ranks(total_ms / args.steps, dev)
    phases = figures(mfsdp, step, phase_ms, peaks)
    phases.update({"step_ms_median": round(statistics.median(steps_ms), 4), "step_ms_min": round(steps_ms[0], 4),
                   "step_ms_max": round(steps_ms[-1], 4)})

    # ---------------------------------------------------------- end to end
    # Through the host-buffer entry point: each step copies the gradient in from
    # pinned host memory and the update back out, shard group by shard group,
    # overlapped with the compute of the neighbouring groups; the AdamW tail's
    # gradient comes in and its parameters go back out too.
    stream = step.stream
    e2e_steps = max(1, args.steps)           # the same K steps as the device-resident region
    e2e_groups = mfsdp.host_step_groups(shards, step.grad.dtype, step.upd.dtype, args.e2e_groups)[0]
    upd_host = torch.empty(numel, dtype=torch.bfloat16).pin_memory()
    tp_host = torch.empty_like(step.tg_host).pin_memory()
    h2d = step.grad_host.numel() * step.grad_host.element_size() + (step.tg_host.numel() * 4 if tail_numel else 0)
    d2h = upd_host.numel() * 2 + (tp_host.numel() * 4 if tail_numel else 0)

    def one_step_host():
        step.count += 1
        mfsdp.muon_owner_step_host(shards, step.grad_host, step.grad, step.mom, step.upd, upd_host, step.ws,
                                   groups=args.e2e_groups, **step.kw)
        if tail_numel:
            step.tg.copy_(step.tg_host, non_blocking=True)
            step.adamw()
            tp_host.copy_(step.tp, non_blocking=True)

    # As many untimed warm-up steps as the device-resident measurement: with a
    # single one, the first timed step sometimes took ~200 ms more (a one-off
    # on the host-memory side) and dominated the mean.
    # No clock sampler runs in this region (nvidia-smi's polling is kept away
    # from the host-buffer copies); the clocks of the resident region, just
    # before, stand for the box.
    for _ in range(max(args.warmup, 1)):
        one_step_host()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    step_ev = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps + 1)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    gc.collect()
    gc.disable()
    # The host's time to enqueue each step: when it approaches the step's device
    # time, the host runs in lockstep with the device and any host stall becomes
    # device idle time inside that step.
    host_ms = []
    e0.record(stream)
    step_ev[0].record(stream)
    for k in range(e2e_steps):
        t_enq = time.perf_counter()
        one_step_host()
        step_ev[k + 1].record(stream)
        host_ms.append(round((time.perf_counter() - t_enq) * 1e3, 3))
    e1.record(stream)
    torch.cuda.synchronize()
    gc.enable()
    step.check_status("after the end-to-end region")
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, dev)
    e2e_steps_ms = [round(step_ev[k].elapsed_time(step_ev[k + 1]), 3) for k in range(e2e_steps)]

    # The same step as one CUDA graph, timed after the end-to-end region, so
    # that nothing the graph leaves behind (its memory pool, its instantiated
    # launches) is released while that region runs.
    if rank == 0 and not args.no_supplementary:
        phases["step_ms_graph"] = round(time_graph(step, min(args.steps, 10)), 4)

    sup = {}
    # ---------------------------------------------------------- supplementary: momentum phase alone
    # The momentum phase of this owner set back to back, with no Newton-Schulz launch
    # before it: inside the step it runs at the SM clock the power cap leaves after
    # the GEMMs, here at the clock the memory-bound kernel itself allows.
    if rank == 0 and not args.no_supplementary and shards:
        for _ in range(2):
            mfsdp.muon_owner_step(shards, step.grad, step.mom, step.upd, step.ws, phases=mfsdp.PHASE_MOMENTUM,
                                  **step.kw)
        torch.cuda.synchronize()
        time.sleep(0.2)
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 5
        s0.record(stream)
        for _ in range(reps):
            mfsdp.muon_owner_step(shards, step.grad, step.mom, step.upd, step.ws, phases=mfsdp.PHASE_MOMENTUM,
                                  **step.kw)
        s1.record(stream)
        torch.cuda.synchronize()
        mb_ms = s0.elapsed_time(s1) / reps
        gbs = phases["momentum_bytes"] / (mb_ms * 1e-3) / 1e9
        sup["momentum_back_to_back"] = {"ms": round(mb_ms, 4), "gbs": round(gbs, 1),
                                        "frac_hbm": round(gbs / peaks["hbm_gbs"], 4)}

    # ---------------------------------------------------------- supplementary: owner-segment reduce
    # The reduce that lands every owned matrix on this owner before the step:
    # w.world simulated ranks' local gradients (bf16, unsharded model layout)
    # summed in rank order into this rank's flat gradient buffer.  The sources
    # are left uninitialised; only the time is taken.
    if rank == 0 and not args.no_supplementary and w.world > 1:
        model = mfsdp.model_placements(w.param_table(), w.align_elems)
        _, model_total = mfsdp.model_layout(w.param_table(), w.align_elems)
        mp, _ = mfsdp.placements(plan)
        segs = mfsdp.placement_segments(model, mp, sim_rank)
        srcs = [torch.empty(model_total, dtype=torch.bfloat16, device=dev) for _ in range(w.world)]
        red_dst = torch.empty(numel, dtype=torch.bfloat16, device=dev)
        for _ in range(2):
            mfsdp.segment_copy(srcs, segs, mfsdp.SEGMENT_REDUCE, red_dst)
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 5
        torch.cuda.synchronize()
        s0.record(stream)
        for _ in range(reps):
            mfsdp.segment_copy(srcs, segs, mfsdp.SEGMENT_REDUCE, red_dst)
        s1.record(stream)
        torch.cuda.synchronize()
        r_ms = s0.elapsed_time(s1) / reps
        moved = sum(g.numel for g in segs) * 2 * (w.world + 1)
        sup["owner_segment_reduce"] = {"ranks": w.world, "ms": round(r_ms, 4),
                                       "gbs": round(moved / r_ms / 1e6, 1), "bytes": moved,
                                       "frac_hbm": round(moved / r_ms / 1e6 / peaks["hbm_gbs"], 4)}
        del srcs, red_dst

    # ---------------------------------------------------------- supplementary: a large AdamW tail
    if rank == 0 and not args.no_supplementary:
        n_big = 50_000_000
        bp = torch.randn(n_big, device=dev) * 1e-3
        bg = torch.randn(n_big, device=dev) * 1e-3
        bm, bv = torch.zeros_like(bp), torch.zeros_like(bp)
        for i in range(3):
            mfsdp.adamw_tail_step(bp, bg, bm, bv, lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, wd=0.1, step=i + 1)
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 10
        torch.cuda.synchronize()
        s0.record(stream)
        for i in range(reps):
            mfsdp.adamw_tail_step(bp, bg, bm, bv, lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, wd=0.1, step=4 + i)
        s1.record(stream)
        torch.cuda.synchronize()
        a_ms = s0.elapsed_time(s1) / reps
        gbs = 28 * n_big / a_ms / 1e6
        sup["adamw_50M"] = {"ms": round(a_ms, 4), "gbs": round(gbs, 1), "frac_hbm": round(gbs / peaks["hbm_gbs"], 4)}
        del bp, bg, bm, bv

    # ---------------------------------------------------------- supplementary: the other owner sets
    # Each of the other workloads' owner sets (the heaviest planner rank),
    # device-resident, timed the same way as the headline (fewer steps).
    if supp_names:
        del step
        torch.cuda.empty_cache()
        sup["workloads"] = {}
        for name in supp_names:
            ws_ = W.get(name)
            _, _, sh, nm, tn = owner_set(ws_, 0)
            g_np = W.owner_grad_buffer(ws_, sh, nm)      # a spawn pool: safe after CUDA work
            st_ = OwnerStep(mfsdp, ws_, sh, nm, tn, g_np, dev)
            del g_np
            k = args.supp_steps
            tot, pms, sms, clk = time_resident(st_, k, max(args.warmup, 3), ClockSampler(local_rank))
            graph_ms = time_graph(st_, max(k, 10))
            fig = figures(mfsdp, st_, pms, peaks)
            fig.pop("momentum_bytes")
            sup["workloads"][name] = {"owner_step_ms": round(tot / k, 4),
                                      "owner_step_ms_median": round(statistics.median(sms), 4),
                                      "owner_step_ms_graph": round(graph_ms, 4),
                                      "steps": k, "matrices": len(sh), "elements": sum(s.rows * s.cols for s in sh),
                                      "tail_elems": tn, **fig,
                                      "sm_mhz": clk.get("sm_mhz"), "reasons": clk.get("reasons")}
            del st_
            torch.cuda.empty_cache()

    # ---------------------------------------------------------- figures
    ns_launches = math.ceil(len(shards) / 128) if shards else 0
    flops_exec = phases["flops_executed"]
    ns_ms = phases["newton_schulz_ms"]
    ns_tflops_exec = phases["newton_schulz_tflops_executed"]
    peak_tf = peaks["bf16_tflops_sustained"]
    digest = ns_source_digest()
    traffic = NS_GEMM_TRAFFIC.get((digest, w.name))
    tensor_active = NS_TENSOR_ACTIVE.get((digest, w.name))

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        if args.cpu_baseline == "full":
            ms_, desc, sec = oracle_owner_step_full(w, shards, tail_numel)
            cpu = {"value": round(ms_, 1), "unit": "ms", "cores": cpu_threads(), "kind": "oracle",
                   "estimated": False, "measured": True, "method": "the whole owner step, timed once",
                   "sample": desc, "seconds": round(sec, 1), **blas_info()}
        else:
            est_ms, desc, sec = oracle_owner_step_estimate(w, shards, tail_numel)
            cpu = {"value": round(est_ms, 1), "unit": "ms", "cores": cpu_threads(), "kind": "oracle",
                   "estimated": True, "method": "per shape: measured time x count", "sample": desc,
                   "seconds": round(sec, 1), **blas_info()}

    elems = sum(s.rows * s.cols for s in shards)
    phases.pop("momentum_bytes")
    line = {
        "metric": METRIC, "value": round(step_ms, 4), "unit": "ms", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 4), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "simulated_rank": sim_rank, "planner_world": w.world,
                   "matrices": len(shards), "elements": elems, "ns_steps": w.ns_steps,
                   "grad_dtype": w.grad_dtype, "update_dtype": "bf16", "tail_elems": tail_numel,
                   "grad_dist": w.grad_dist,
                   "l2": f"no flush: inputs {(grad_bytes + 4 * numel) / 1e9:.1f} GB > 129 MB L2",
                   "parallelism": f"owner sets x{world}"},
        "phases": phases,
        "roofline": {"kernel": "ns_kernel", "bound": "tensor", "achieved": ns_tflops_exec,
                     "peak": peak_tf, "unit": "TFLOP/s", "frac": round(ns_tflops_exec / peak_tf, 4),
                     "traffic": traffic, "tensor_pipe_active_ncu": tensor_active, "kernel_digest": digest,
                     "peak_source": f"{peak_src} bf16_tflops_sustained",
                     "flops": ("executed tensor-core FLOPs (symmetric products: upper-triangle blocks only; "
                               "matrices with l >= 2s iterate on their s x s Gram matrix)"),
                     "flops_per_launch": round(flops_exec / max(ns_launches, 1)), "launches_per_step": ns_launches,
                     "ms_per_launch": round(ns_ms / max(ns_launches, 1), 4)},
        "clocks": clocks,
        "e2e": {"value": round(e2e_ms, 4), "unit": "ms", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "api": "mfsdp_muon_owner_step_host",
                "pipeline_groups": e2e_groups, "steps_ms": e2e_steps_ms, "host_enqueue_ms": host_ms,
                "median_ms": round(statistics.median(e2e_steps_ms), 3),
                "clocks": "not sampled in this region (see the top-level clocks)"},
        "gpu_launches": step_launches(shards, tail_numel) * args.steps,
        "cpu_baseline": cpu,
        "supplementary": sup,
        "input_generation_s": round(t_gen, 1),
        "library": mfsdp.version(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def step_launches(shards, tail_numel):
    """Kernels one owner step launches: per batch of 128 matrices the momentum
    kernel, the norm finalise and one Newton-Schulz launch; one AdamW launch."""
    batches = math.ceil(len(shards) / 128) if shards else 0
    return 3 * batches + (1 if tail_numel else 0)


def run_kernel_case(args):
    """One memory-bound kernel alone, on a case small enough for a full ncu
    capture (a few GB on the device) but larger than L2: K timed launches after
    W warm-up ones, CUDA events on the launching stream.  Prints one JSON line
    with the kernel's algorithmic GB/s against the measured HBM peak.

    adamw:          the fused AdamW kernel over a 50M-element fp32 tail (the
                    skewed MoE owner set's tail), 28 bytes per element.
    segment_reduce: the owner-segment reduce of a three-layer Llama-1.3B-shaped
                    stack (d = 2048, ffn = 5504) planned over 8 simulated ranks:
                    the heaviest owner's matrix segments summed in rank order
                    from the 8 ranks' bf16 model-layout buffers, 2 bytes per
                    element per source plus 2 written.
    """
    from matrix_optimizers_under_gb300 import _build
    _build.ensure_built()
    from matrix_optimizers_under_gb300 import binding as mfsdp
    import torch
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    gen = torch.Generator(device=dev)
    gen.manual_seed(5)
    if args.kernel == "adamw":
        n = 50_000_000
        bp = torch.randn(n, device=dev, generator=gen) * 1e-3
        bg = torch.randn(n, device=dev, generator=gen) * 1e-3
        bm, bv = torch.zeros_like(bp), torch.zeros_like(bp)
        count = [0]

        def launch():
            count[0] += 1
            mfsdp.adamw_tail_step(bp, bg, bm, bv, lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, wd=0.1, step=count[0])
        moved = 28 * n
        case = {"kernel": "adamw_kernel", "elements": n, "dtype": "f32"}
    else:
        world = 8
        table = W.llama_param_table(3, 2048, 5504, 2048)
        plan = mfsdp.plan_owners(table, world, 5, 128)
        owner = heaviest_rank(plan)
        model = mfsdp.model_placements(table, 128)
        _, model_total = mfsdp.model_layout(table, 128)
        mp, _ = mfsdp.placements(plan)
        segs = mfsdp.placement_segments(model, mp, owner)
        srcs = [(torch.randn(model_total, device=dev, generator=gen) * 1e-3).to(torch.bfloat16)
                for _ in range(world)]
        dst = torch.empty(plan.rank_matrix_elems[owner], dtype=torch.bfloat16, device=dev)

        def launch():
            mfsdp.segment_copy(srcs, segs, mfsdp.SEGMENT_REDUCE, dst)
        owned = sum(g.numel for g in segs)
        moved = owned * 2 * (world + 1)
        case = {"kernel": "segment_kernel", "mode": "reduce", "ranks": world, "segments": len(segs),
                "elements": owned, "model_elements": model_total, "dtype": "bf16"}
    for _ in range(args.warmup):
        launch()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(0)
    sampler.start()
    time.sleep(0.4)
    e0.record(stream)
    for _ in range(args.steps):
        launch()
    e1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    ms = e0.elapsed_time(e1) / args.steps
    peaks, peak_src = load_peaks()
    gbs = moved / (ms * 1e-3) / 1e9
    print(json.dumps({"kernel_case": args.kernel, "metric": "algorithmic HBM GB/s", "value": round(gbs, 1),
                      "unit": "GB/s", "ms_per_launch": round(ms, 4), "launches": args.steps, "warmup": args.warmup,
                      "bytes_per_launch": moved, "frac_hbm": round(gbs / peaks["hbm_gbs"], 4),
                      "peak_gbs": peaks["hbm_gbs"], "peak_source": peak_src, "config": case,
                      "l2": f"no flush: {moved / 1e9:.2f} GB moved per launch > 129 MB L2",
                      "clocks": clocks, "library": mfsdp.version()}))
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="llama3_8b_rank", choices=W.ORDER)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-baseline", choices=("per-shape", "full"), default="per-shape",
                    help="CPU oracle leg: one matrix of each shape timed x its count (default, ~30 s), or the "
                         "whole owner step timed once (minutes on the large owner sets)")
    ap.add_argument("--no-supplementary", action="store_true")
    ap.add_argument("--supp-steps", type=int, default=10,
                    help="timed steps of each other workload's owner set in the supplementary lines")
    ap.add_argument("--e2e-groups", type=int, default=0,
                    help="shard groups the host-buffer step overlaps copies with (1 = no overlap, "
                         "0 = the library's choice for the owner set)")
    ap.add_argument("--kernel", choices=("adamw", "segment_reduce"), default=None,
                    help="time one memory-bound kernel alone on a small case instead of the owner step")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.kernel:
        return run_kernel_case(args)
    return run_reference(args) if args.impl == "reference" else run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
