"""Pins for the owner-segment reduce and resharding oracle (MatrixFSDP --
Abstract: the backward reduction lands each whole matrix on its owner;
owner-shard checkpoint resharding).  Checked against properties that any
correct reduce-scatter / remap has: one source copies exactly, x + (-x)
cancels, the sum over owners of the owners' segments is the total of the
sources, a reshard to a new plan and back is the identity, and every
parameter of a model lands exactly once."""
import numpy as np
import pytest

from oracle import (model_layout_ref, placement_segments_ref, segment_gather_ref, segment_reduce_ref,
                    plan_owners_ref)
from matrix_optimizers_under_gb300 import workloads as W


def placements(plan, params):
    m = [dict(param_id=s["param_id"], owner=s["owner"], offset=s["offset"], numel=s["rows"] * s["cols"])
         for s in plan["matrix_shards"]]
    t = [dict(param_id=s["param_id"], owner=s["owner"], offset=s["offset"], numel=s["numel"])
         for s in plan["tail_shards"]]
    return m, t


def test_model_layout_hand_example():
    offs, total = model_layout_ref([(3, 5, 0), (7, 1, 1), (2, 2, 0)], 8)
    assert offs == [0, 16, 24] and total == 32


@pytest.mark.parametrize("world", [1, 2, 3, 8])
def test_reduce_properties(world):
    params = W.ragged_params(world, 30, max_dim=40)
    offs, total = model_layout_ref(params, 16)
    model = [dict(param_id=i, owner=0, offset=o, numel=p[0] * p[1]) for i, (o, p) in enumerate(zip(offs, params))]
    plan = plan_owners_ref(params, world, 5, 16)
    mp, tp = placements(plan, params)
    rng = np.random.default_rng(world)
    srcs = [rng.standard_normal(total) for _ in range(world)]
    grand = sum(s for s in srcs)
    seen = 0
    for r in range(world):
        for pl, ext in ((mp, plan["rank_matrix_elems"][r]), (tp, plan["rank_tail_elems"][r])):
            segs = placement_segments_ref(model, pl, r)
            out = segment_reduce_ref(srcs, segs, ext)
            for g in segs:
                np.testing.assert_allclose(out[g["dst_offset"]:g["dst_offset"] + g["numel"]],
                                           grand[g["src_offset"]:g["src_offset"] + g["numel"]], rtol=1e-13)
                seen += g["numel"]
    assert seen == sum(p[0] * p[1] for p in params)   # every element lands exactly once
    segs = placement_segments_ref(model, mp, 0)
    one = segment_reduce_ref(srcs[:1], segs, plan["rank_matrix_elems"][0])
    assert np.array_equal(np.nan_to_num(one, nan=7.0), np.nan_to_num(segment_gather_ref(srcs[:1], segs, len(one)), nan=7.0))
    zero = segment_reduce_ref([srcs[0], -srcs[0]], segs, len(one))
    assert np.all(np.nan_to_num(zero) == 0.0)


@pytest.mark.parametrize("worlds", [(8, 3), (2, 5), (4, 1)])
def test_reshard_round_trip(worlds):
    wa, wb = worlds
    params = [p for p in W.ragged_params(11, 80, max_dim=48) if p[2] == 0]
    a = plan_owners_ref(params, wa, 5, 128)
    b = plan_owners_ref(params, wb, 5, 128)
    am, _ = placements(a, params)
    bm, _ = placements(b, params)
    # one number per parameter, repeated over its segment: one number per parameter, repeated over its segment
    bufs_a = []
    for r in range(wa):
        buf = np.full(a["rank_matrix_elems"][r], np.nan)
        for e in am:
            if e["owner"] == r:
                buf[e["offset"]:e["offset"] + e["numel"]] = e["param_id"]
        bufs_a.append(buf)
    bufs_b = [segment_gather_ref(bufs_a, placement_segments_ref(am, bm, r), b["rank_matrix_elems"][r])
              for r in range(wb)]
    for e in bm:
        assert np.all(bufs_b[e["owner"]][e["offset"]:e["offset"] + e["numel"]] == e["param_id"])
    back = [segment_gather_ref(bufs_b, placement_segments_ref(bm, am, r), a["rank_matrix_elems"][r])
            for r in range(wa)]
    for r in range(wa):
        assert np.array_equal(np.nan_to_num(back[r], nan=-1), np.nan_to_num(bufs_a[r], nan=-1))
