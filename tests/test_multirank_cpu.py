"""The multi-GPU bench path on CPU: two gloo ranks on 127.0.0.1.

Owner sets shard with no data-path collective (MatrixFSDP -- Abstract: no
optimizer-step matrix collective), so under torchrun each GPU benches a
different simulated rank's owner set and only the timings are reduced (max over
ranks).  This checks that the ranks pick distinct, complete owner sets of the
same plan, that the plan is identical on every rank (the deterministic planner
runs locally everywhere), and that the max-reduce returns the slowest rank.
"""
import os
import socket

import pytest
import torch.multiprocessing as tmp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from matrix_optimizers_under_gb300 import _build, workloads as W
    _build.ensure_built()
    from matrix_optimizers_under_gb300 import binding as mfsdp
    w = W.get("llama3_8b_rank")
    plan = mfsdp.plan_owners(w.param_table(), w.world, w.ns_steps, w.align_elems)
    heavy = bench.heaviest_rank(plan)
    sim = bench.simulated_rank(heavy, rank, w.world)
    ids = sorted(s.param_id for s in plan.rank_matrices(sim))
    slowest = bench.max_over_ranks(10.0 + rank)
    digest = hash(tuple((s.param_id, s.owner, s.offset) for s in plan.matrix_shards))
    gathered = [None] * world
    dist.all_gather_object(gathered, (sim, ids, digest))
    out[rank] = (slowest, gathered)
    dist.destroy_process_group()


def test_two_gloo_ranks_bench_distinct_owner_sets(mfsdp):
    world = 2
    port = _free_port()
    mgr = tmp.get_context("spawn").Manager()
    out = mgr.dict()
    tmp.start_processes(_worker, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
    assert sorted(out.keys()) == [0, 1]
    for r in range(world):
        slowest, gathered = out[r]
        assert slowest == 11.0
        sims = [g[0] for g in gathered]
        assert len(set(sims)) == world                     # distinct owner sets
        assert len({g[2] for g in gathered}) == 1          # same plan on every rank
        for g in gathered:
            assert len(g[1]) == 28                         # each a complete 8B owner set
        assert not set(gathered[0][1]) & set(gathered[1][1])
