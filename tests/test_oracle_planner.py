"""Pins for the oracle planner (MatrixFSDP -- Abstract: balance-aware owner
planner, whole-matrix ownership, tail owners; Section 1: no rank keeps a full
model copy).  Checked against a hand-worked layout, brute-force enumeration of
all assignments on tiny layouts (Graham's LPT bound and its optimality case),
and structural invariants of the segment map."""
import itertools
import json
import os

import numpy as np
import pytest

from oracle.planner import plan_owners_ref, ns_cost, heaviest_rank_ref
from matrix_optimizers_under_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_hand_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "planner_hand_example.json")))
    plan = plan_owners_ref([tuple(p) for p in g["params"]], g["world"], g["ns_steps"], g["align_elems"])
    for k in ("matrix_shards", "tail_shards", "rank_matrix_elems", "rank_tail_elems", "rank_cost"):
        assert plan[k] == g[k], k


def check_layout(params, plan, world, align):
    mats = [i for i, p in enumerate(params) if p[2] == 0]
    tails = [i for i, p in enumerate(params) if p[2] == 1]
    assert sorted(s["param_id"] for s in plan["matrix_shards"]) == mats
    assert sorted(s["param_id"] for s in plan["tail_shards"]) == tails
    for key, ext, size in (("matrix_shards", plan["rank_matrix_elems"], lambda s: s["rows"] * s["cols"]),
                           ("tail_shards", plan["rank_tail_elems"], lambda s: s["numel"])):
        for r in range(world):
            segs = sorted((s for s in plan[key] if s["owner"] == r), key=lambda s: s["offset"])
            ids = [s["param_id"] for s in segs]
            assert ids == sorted(ids)      # declaration order inside a rank
            end = 0
            for s in segs:
                assert s["offset"] % align == 0 and s["offset"] >= end
                end = s["offset"] + size(s)
            assert ext[r] >= end and ext[r] % align == 0 and ext[r] - end < align
    for s in plan["matrix_shards"]:
        p = params[s["param_id"]]
        assert (s["rows"], s["cols"]) == (p[0], p[1])
        assert s["transposed"] == int(p[0] > p[1])


def brute_force_opt(costs, world):
    best, best_two = None, None
    for assign in itertools.product(range(world), repeat=len(costs)):
        load = [0] * world
        cnt = [0] * world
        for c, r in zip(costs, assign):
            load[r] += c
            cnt[r] += 1
        mk = max(load)
        if best is None or mk < best:
            best = mk
        if max(cnt) <= 2 and (best_two is None or mk < best_two):
            best_two = mk
    return best, best_two


@pytest.mark.parametrize("seed", range(40))
def test_lpt_against_brute_force(seed):
    rng = np.random.default_rng(seed)
    world = int(rng.integers(1, 4))
    n = int(rng.integers(1, 8))
    dims = [int(d) for d in rng.choice([8, 16, 24, 32, 48, 64], size=2 * n)]
    params = [(dims[2 * i], dims[2 * i + 1], 0) for i in range(n)]
    plan = plan_owners_ref(params, world, 5, 128)
    check_layout(params, plan, world, 128)
    costs = [ns_cost(r, c, 5) for r, c, _ in params]
    mk = max(plan["rank_cost"])
    opt, opt_two = brute_force_opt(costs, world)
    # Graham 1969: LPT makespan <= (4/3 - 1/(3W)) OPT
    assert 3 * world * mk <= (4 * world - 1) * opt
    # and LPT is optimal when some optimal schedule has at most two jobs per rank
    if opt_two == opt:
        assert mk == opt
    assert sum(plan["rank_cost"]) == sum(costs)


@pytest.mark.parametrize("seed", range(10))
def test_ragged_layout_invariants(seed):
    params = W.ragged_params(seed, 60)
    for world in (1, 2, 3, 8, 64):
        for align in (1, 8, 128):
            plan = plan_owners_ref(params, world, 5, align)
            check_layout(params, plan, world, align)


def test_empty_and_degenerate():
    plan = plan_owners_ref([], 4, 5, 128)
    assert plan["matrix_shards"] == [] and plan["rank_matrix_elems"] == [0] * 4
    # more ranks than matrices: the extra ranks hold empty shards
    plan = plan_owners_ref([(8, 8, 0), (4, 4, 0)], 5, 5, 128)
    assert [s["owner"] for s in plan["matrix_shards"]] == [0, 1]
    assert plan["rank_matrix_elems"] == [128, 128, 0, 0, 0]
    with pytest.raises(ValueError):
        plan_owners_ref([(8, 8, 0)], 0, 5, 128)


@pytest.mark.parametrize("name", W.ORDER)
def test_workload_plans(name):
    w = W.get(name)
    params = w.param_table()
    plan = plan_owners_ref(params, w.world, w.ns_steps, w.align_elems)
    check_layout(params, plan, w.world, w.align_elems)
    # no rank keeps a full model copy when there is more than one rank
    total = sum(p[0] * p[1] for p in params if p[2] == 0)
    if w.world > 1:
        assert max(plan["rank_matrix_elems"]) < total


def test_transformer_ranks_balance_exactly():
    # 8B: 224 matrices over 8 ranks come out as 12 MLP + 8 q/o + 8 k/v per rank.
    w = W.get("llama3_8b_rank")
    plan = plan_owners_ref(w.param_table(), 8, 5, 128)
    assert len(set(plan["rank_cost"])) == 1
    big = 5 * (4 * 4096 ** 2 * 14336 + 2 * 4096 ** 3)
    sq = 5 * 6 * 4096 ** 3
    kv = 5 * (4 * 1024 ** 2 * 4096 + 2 * 1024 ** 3)
    assert plan["rank_cost"][0] == 12 * big + 8 * sq + 8 * kv
    r = heaviest_rank_ref(plan)
    mine = [s for s in plan["matrix_shards"] if s["owner"] == r]
    assert len(mine) == 28 and sum(s["rows"] * s["cols"] for s in mine) == 872_415_232
    w = W.get("llama_1p3b_rank")
    plan = plan_owners_ref(w.param_table(), 8, 5, 128)
    assert len(set(plan["rank_cost"])) == 1
    r = heaviest_rank_ref(plan)
    mine = [s for s in plan["matrix_shards"] if s["owner"] == r]
    assert len(mine) == 21 and plan["rank_tail_numel"][r] == 8 * 2048
