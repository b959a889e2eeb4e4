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
pinned host memory and the update copied back every step.  `--impl reference`
times the fp64 CPU oracle on a bounded sample of the same workload instead.

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

# DRAM bytes (read + write) per Newton-Schulz kernel launch on the llama3_8b_rank owner set
# (0.5/0.6: the mean over one owner step's 15 per-product launches; 0.7: the one launch that
# runs all of a step's products), from the ncu capture summarised in
# profiles/launches_llama3_8b_rank.md; keyed by the library version it was taken on, so
# that a changed kernel reports null until it is captured again.
NS_GEMM_TRAFFIC = {("0.5.0", "llama3_8b_rank"): 3.359e9, ("0.6.0", "llama3_8b_rank"): 3.401e9,
                   ("0.7.0", "llama3_8b_rank"): 50.17e9, ("0.8.1", "llama3_8b_rank"): 50.02e9,
                   ("0.8.2", "llama3_8b_rank"): 50.02e9, ("0.8.3", "llama3_8b_rank"): 50.02e9,
                   ("0.8.4", "llama3_8b_rank"): 50.02e9,
                   ("0.8.5", "llama3_8b_rank"): 50.58e9, ("0.8.6", "llama3_8b_rank"): 50.08e9,
                   # 0.8.7-0.8.9 changed only host code (the host-buffer entry's grouping, argument
                   # checks): ns_kernel is 0.8.6's
                   ("0.8.7", "llama3_8b_rank"): 50.08e9, ("0.8.8", "llama3_8b_rank"): 50.08e9,
                   ("0.8.9", "llama3_8b_rank"): 50.08e9}


# --------------------------------------------------------------------------- helpers
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


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
def oracle_sample(w, shards, tail_n, sample_ids, threads_note=""):
    """Times the fp64 oracle on the sample matrices (momentum + Newton-Schulz)
    and on the AdamW tail; returns (seconds, sample NS FLOPs, sample elements)."""
    from oracle import adamw_ref, muon_matrix_ref
    a, b, c = w.ns_coeffs
    t0 = time.perf_counter()
    flops = 0
    elems = 0
    for s in shards:
        if s.param_id not in sample_ids:
            continue
        g = W.grad_storage(w, s.param_id)
        G = ((g.astype(np.uint32) << 16).view(np.float32) if g.dtype == np.uint16 else g).astype(np.float64)
        muon_matrix_ref(G, np.zeros_like(G), w.beta, w.nesterov, w.ns_steps, a, b, c, w.ns_eps)
        flops += ns_flops(s.rows, s.cols, w.ns_steps)
        elems += s.rows * s.cols
    if tail_n:
        rng = np.random.default_rng(0)
        p = rng.standard_normal(tail_n)
        adamw_ref(p, p, np.zeros(tail_n), np.zeros(tail_n), w.lr, w.betas[0], w.betas[1], w.adam_eps,
                  w.weight_decay, w.step)
    return time.perf_counter() - t0, flops, elems


def cpu_threads():
    try:
        from threadpoolctl import threadpool_info
        info = threadpool_info()
        if info:
            return int(max(i.get("num_threads", 1) for i in info))
    except Exception:
        pass
    return os.cpu_count() or 1


def pick_sample(shards):
    """A bounded sample of the owner set: its smallest matrix plus one square one
    (about 10-30 s of fp64 CPU work for the transformer owner sets)."""
    by_size = sorted(shards, key=lambda s: (s.rows * s.cols, s.param_id))
    ids = [by_size[0].param_id]
    sq = [s for s in shards if s.rows == s.cols]
    if sq and sq[0].param_id not in ids:
        ids.append(sq[0].param_id)
    return ids


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
    total_flops = sum(ns_flops(s.rows, s.cols, w.ns_steps) for s in shards)
    sample = [min(shards, key=lambda s: (s.rows * s.cols, s.param_id)).param_id]
    ms = []
    for i in range(args.warmup + args.steps):
        sec, fl, el = oracle_sample(w, shards, tail_n, sample)
        if i >= args.warmup:
            ms.append(sec * 1e3 * total_flops / fl)
    value = statistics.mean(ms)
    cores = cpu_threads()
    desc = (f"fp64 NumPy oracle on param {sample[0]} "
            f"({[(s.rows, s.cols) for s in shards if s.param_id == sample[0]][0]}) + the {tail_n}-element tail "
            f"per step, scaled by dense Newton-Schulz FLOPs to the {len(shards)}-matrix owner set")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "ms", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(value, 3), "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "matrices": len(shards),
                       "elements": sum(s.rows * s.cols for s in shards), "ns_steps": w.ns_steps},
            "cpu_baseline": {"value": round(value, 3), "unit": "ms", "cores": cores, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": round(value, 3), "unit": "ms", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------- our arm
def run_ours(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    w = W.get(args.workload)

    from matrix_optimizers_under_gb300 import _build
    _build.ensure_built()
    from matrix_optimizers_under_gb300 import binding as mfsdp

    plan = mfsdp.plan_owners(w.param_table(), w.world, w.ns_steps, w.align_elems)
    heavy = heaviest_rank(plan)
    sim_rank = simulated_rank(heavy, rank, w.world)
    shards = plan.rank_matrices(sim_rank)
    tails = plan.rank_tails(sim_rank)
    numel = plan.rank_matrix_elems[sim_rank]
    tail_numel = plan.rank_tail_elems[sim_rank]

    t_gen = time.time()
    grad_np = W.owner_grad_buffer(w, shards, numel)   # before any CUDA call (spawn pool)
    t_gen = time.time() - t_gen

    import torch
    import torch.distributed as dist
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream()

    bf16 = w.grad_dtype == "bf16"
    grad_host = torch.from_numpy(grad_np.view(np.int16) if bf16 else grad_np).pin_memory()
    grad_host = grad_host.view(torch.bfloat16) if bf16 else grad_host
    grad = grad_host.to(dev)
    mom = torch.zeros(numel, dtype=torch.float32, device=dev)
    upd = torch.zeros(numel, dtype=torch.bfloat16, device=dev)
    ws = torch.empty(mfsdp.muon_workspace_bytes(shards), dtype=torch.uint8, device=dev)
    rng = np.random.default_rng(w.seed)
    tp = torch.from_numpy((rng.standard_normal(max(tail_numel, 1)) * w.tail_scale).astype(np.float32)).to(dev)
    tg_host = torch.from_numpy((rng.standard_normal(max(tail_numel, 1)) * w.tail_scale)
                               .astype(np.float32)).pin_memory()
    tg = tg_host.to(dev)
    tm, tv = torch.zeros_like(tp), torch.zeros_like(tp)
    upd_host = torch.empty(numel, dtype=torch.bfloat16).pin_memory()
    tp_host = torch.empty_like(tg_host).pin_memory()
    a, b, c = w.ns_coeffs
    kw = dict(beta=w.beta, nesterov=w.nesterov, ns_steps=w.ns_steps, coeffs=w.ns_coeffs, eps=w.ns_eps)
    batches = math.ceil(len(shards) / 128) if shards else 0
    # per batch of 128 matrices: momentum, norm finalise, one Newton-Schulz launch (or the T = 0 emit)
    launches_per_step = 3 * batches + (1 if tail_numel else 0)

    step_counter = [0]

    def one_step(ev=None):
        step_counter[0] += 1
        if ev:
            ev[0].record(stream)
        mfsdp.muon_owner_step(shards, grad, mom, upd, ws, phases=mfsdp.PHASE_MOMENTUM, **kw)
        if ev:
            ev[1].record(stream)
        mfsdp.muon_owner_step(shards, grad, mom, upd, ws, phases=mfsdp.PHASE_NEWTON_SCHULZ, **kw)
        if ev:
            ev[2].record(stream)
        if tail_numel:
            mfsdp.adamw_tail_step(tp, tg, tm, tv, lr=w.lr, beta1=w.betas[0], beta2=w.betas[1], eps=w.adam_eps,
                                  wd=w.weight_decay, step=step_counter[0])
        if ev:
            ev[3].record(stream)

    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize()
    st, detail = mfsdp.muon_device_status(ws)
    if st != mfsdp.OK:
        raise RuntimeError(f"device status after warm-up: {mfsdp.status_string(st)} ({detail})")

    # ---------------------------------------------------------- timed region
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.4)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    gc.collect()
    gc.disable()            # no collector pause while the host enqueues the timed steps
    t_start.record(stream)
    for k in range(args.steps):
        one_step(evs[k])
    t_end.record(stream)
    torch.cuda.synchronize()
    gc.enable()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    total_ms = t_start.elapsed_time(t_end)
    mom_ms = sum(e[0].elapsed_time(e[1]) for e in evs) / args.steps
    ns_ms = sum(e[1].elapsed_time(e[2]) for e in evs) / args.steps
    adam_ms = sum(e[2].elapsed_time(e[3]) for e in evs) / args.steps
    steps_ms = sorted(e[0].elapsed_time(e[3]) for e in evs)
    step_ms = max_over_ranks(total_ms / args.steps, dev)
    st, detail = mfsdp.muon_device_status(ws)
    if st != mfsdp.OK:
        raise RuntimeError(f"device status after timed region: {mfsdp.status_string(st)} ({detail})")

    # ---------------------------------------------------------- end to end
    # Through the host-buffer entry point: each step copies the gradient in from
    # pinned host memory and the update back out, shard group by shard group,
    # overlapped with the compute of the neighbouring groups; the AdamW tail's
    # gradient comes in and its parameters go back out too.
    e2e_steps = max(1, min(args.steps, 10))
    e2e_groups = mfsdp.host_step_groups(shards, grad.dtype, upd.dtype, args.e2e_groups)[0]
    h2d = grad_host.numel() * grad_host.element_size() + (tg_host.numel() * 4 if tail_numel else 0)
    d2h = upd_host.numel() * 2 + (tp_host.numel() * 4 if tail_numel else 0)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def one_step_host():
        step_counter[0] += 1
        mfsdp.muon_owner_step_host(shards, grad_host, grad, mom, upd, upd_host, ws, groups=args.e2e_groups, **kw)
        if tail_numel:
            tg.copy_(tg_host, non_blocking=True)
            mfsdp.adamw_tail_step(tp, tg, tm, tv, lr=w.lr, beta1=w.betas[0], beta2=w.betas[1], eps=w.adam_eps,
                                  wd=w.weight_decay, step=step_counter[0])
            tp_host.copy_(tp, non_blocking=True)

    # As many untimed warm-up steps as the device-resident measurement: with a
    # single one, the first timed step sometimes took ~200 ms more (a one-off
    # on the host-memory side) and dominated the mean.
    e2e_sampler = ClockSampler(local_rank)      # clocks and throttle reasons of the e2e region too
    e2e_sampler.start()
    for _ in range(max(args.warmup, 1)):
        one_step_host()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    step_ev = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps + 1)]
    gc.collect()
    gc.disable()
    e0.record(stream)
    step_ev[0].record(stream)
    for k in range(e2e_steps):
        one_step_host()
        step_ev[k + 1].record(stream)
    e1.record(stream)
    torch.cuda.synchronize()
    gc.enable()
    e2e_clocks = e2e_sampler.stop()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, dev)
    e2e_steps_ms = [round(step_ev[k].elapsed_time(step_ev[k + 1]), 3) for k in range(e2e_steps)]

    # ---------------------------------------------------------- supplementary: a large AdamW tail
    sup = {}
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
        sup["adamw_50M"] = {"ms": round(a_ms, 4), "gbs": round(28 * n_big / a_ms / 1e6, 1)}
        del bp, bg, bm, bv

    # ---------------------------------------------------------- supplementary: momentum phase alone
    # The momentum phase of this owner set back to back, with no Newton-Schulz launch
    # before it: inside the step it runs at the SM clock the power cap leaves after
    # the GEMMs, here at the clock the memory-bound kernel itself allows.
    if rank == 0 and not args.no_supplementary and shards:
        for _ in range(2):
            mfsdp.muon_owner_step(shards, grad, mom, upd, ws, phases=mfsdp.PHASE_MOMENTUM, **kw)
        torch.cuda.synchronize()
        time.sleep(0.2)
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 5
        s0.record(stream)
        for _ in range(reps):
            mfsdp.muon_owner_step(shards, grad, mom, upd, ws, phases=mfsdp.PHASE_MOMENTUM, **kw)
        s1.record(stream)
        torch.cuda.synchronize()
        sup["momentum_back_to_back"] = {"ms": round(s0.elapsed_time(s1) / reps, 4)}

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
                                       "gbs": round(moved / r_ms / 1e6, 1), "bytes": moved}
        del srcs, red_dst

    # ---------------------------------------------------------- figures
    peaks, peak_src = load_peaks()
    flops, flops_exec = mfsdp.muon_step_flops(shards, w.ns_steps)
    elems = sum(s.rows * s.cols for s in shards)
    gsz = 2 if bf16 else 4
    mom_bytes = elems * (gsz + 4 + 4 + 2)
    ns_tflops = flops / (ns_ms * 1e-3) / 1e12 if ns_ms > 0 else 0.0           # dense-equivalent
    ns_tflops_exec = flops_exec / (ns_ms * 1e-3) / 1e12 if ns_ms > 0 else 0.0  # executed MMA work
    mom_gbs = mom_bytes / (mom_ms * 1e-3) / 1e9 if mom_ms > 0 else 0.0
    adam_gbs = 28 * tail_numel / (adam_ms * 1e-3) / 1e9 if adam_ms > 0 and tail_numel else 0.0
    peak_tf = peaks["bf16_tflops_sustained"]
    hbm = peaks["hbm_gbs"]
    ns_launches = batches
    if "adamw_50M" in sup:
        sup["adamw_50M"]["frac_hbm"] = round(sup["adamw_50M"]["gbs"] / hbm, 4)
    if "momentum_back_to_back" in sup:
        mb = sup["momentum_back_to_back"]
        mb["gbs"] = round(mom_bytes / (mb["ms"] * 1e-3) / 1e9, 1)
        mb["frac_hbm"] = round(mb["gbs"] / hbm, 4)
    if "owner_segment_reduce" in sup:
        sup["owner_segment_reduce"]["frac_hbm"] = round(sup["owner_segment_reduce"]["gbs"] / hbm, 4)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        sample = pick_sample(shards)
        sec, fl, el = oracle_sample(w, shards, 0, sample)
        est_ms = sec * 1e3 * flops / fl
        desc = (f"fp64 NumPy oracle (momentum + Newton-Schulz) on params {sample} "
                f"{[(s.rows, s.cols) for s in shards if s.param_id in sample]} of the benched owner set, "
                f"{sec:.1f} s, scaled by dense Newton-Schulz FLOPs to all {len(shards)} matrices")
        cpu = {"value": round(est_ms, 1), "unit": "ms", "cores": cpu_threads(), "kind": "oracle", "sample": desc}

    line = {
        "metric": METRIC, "value": round(step_ms, 4), "unit": "ms", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 4), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "simulated_rank": sim_rank, "planner_world": w.world,
                   "matrices": len(shards), "elements": elems, "ns_steps": w.ns_steps,
                   "grad_dtype": w.grad_dtype, "update_dtype": "bf16", "tail_elems": tail_numel,
                   "grad_dist": w.grad_dist,
                   "l2": f"no flush: inputs {(grad_np.nbytes + 4 * numel + ws.numel()) / 1e9:.1f} GB > 129 MB L2",
                   "parallelism": f"owner sets x{world}"},
        "phases": {"momentum_ms": round(mom_ms, 4), "momentum_gbs": round(mom_gbs, 1),
                   "momentum_frac_hbm": round(mom_gbs / hbm, 4),
                   "newton_schulz_ms": round(ns_ms, 4),
                   "newton_schulz_tflops_executed": round(ns_tflops_exec, 1),
                   "newton_schulz_frac_bf16_executed": round(ns_tflops_exec / peak_tf, 4),
                   "newton_schulz_tflops_dense_equivalent": round(ns_tflops, 1),
                   "newton_schulz_frac_bf16_dense_equivalent": round(ns_tflops / peak_tf, 4),
                   "flops_dense": flops, "flops_executed": flops_exec,
                   "adamw_ms": round(adam_ms, 4), "adamw_gbs": round(adam_gbs, 1),
                   "step_ms_median": round(statistics.median(steps_ms), 4),
                   "step_ms_min": round(steps_ms[0], 4), "step_ms_max": round(steps_ms[-1], 4)},
        "roofline": {"kernel": "ns_kernel", "bound": "tensor", "achieved": round(ns_tflops_exec, 1),
                     "peak": peak_tf, "unit": "TFLOP/s", "frac": round(ns_tflops_exec / peak_tf, 4),
                     "traffic": NS_GEMM_TRAFFIC.get((mfsdp.version(), w.name)),
                     "peak_source": f"{peak_src} bf16_tflops_sustained",
                     "flops": "executed tensor-core FLOPs (symmetric Gram/polynomial: upper-triangle blocks only)",
                     "flops_per_launch": round(flops_exec / max(ns_launches, 1)), "launches_per_step": ns_launches},
        "clocks": clocks,
        "e2e": {"value": round(e2e_ms, 4), "unit": "ms", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "api": "mfsdp_muon_owner_step_host",
                "pipeline_groups": e2e_groups, "steps_ms": e2e_steps_ms,
                "median_ms": round(statistics.median(e2e_steps_ms), 3), "clocks": e2e_clocks},
        "gpu_launches": launches_per_step * args.steps,
        "cpu_baseline": cpu,
        "supplementary": sup,
        "input_generation_s": round(t_gen, 1),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


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
    ap.add_argument("--no-supplementary", action="store_true")
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
