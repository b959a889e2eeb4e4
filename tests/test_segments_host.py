"""Host side of the owner-segment reduce and resharding (no GPU): the C++
layout and segment mapping reproduce the oracle exactly, and bad segment
tables are rejected before anything is queued (fake pointers; nothing runs)."""
import ctypes

import pytest

from oracle import model_layout_ref, placement_segments_ref, plan_owners_ref
from matrix_optimizers_under_gb300 import workloads as W


def _ref_placements(plan):
    m = [dict(param_id=s["param_id"], owner=s["owner"], offset=s["offset"], numel=s["rows"] * s["cols"])
         for s in plan["matrix_shards"]]
    t = [dict(param_id=s["param_id"], owner=s["owner"], offset=s["offset"], numel=s["numel"])
         for s in plan["tail_shards"]]
    return m, t


@pytest.mark.parametrize("name", ["gpt2_block", "llama_1p3b_rank", "llama3_8b_rank", "moe_skewed"])
def test_model_layout_matches_oracle(mfsdp, name):
    params = W.get(name).param_table()
    for align in (1, 128):
        assert mfsdp.model_layout(params, align) == model_layout_ref(params, align)


@pytest.mark.parametrize("seed", range(6))
def test_segments_match_oracle(mfsdp, seed):
    params = W.ragged_params(seed, 50, max_dim=64)
    model_ref = [dict(param_id=i, owner=0, offset=o, numel=p[0] * p[1])
                 for i, (o, p) in enumerate(zip(model_layout_ref(params, 16)[0], params))]
    model = mfsdp.model_placements(params, 16)
    for wa, wb in ((3, 5), (8, 2)):
        pa, pb = mfsdp.plan_owners(params, wa, 5, 16), mfsdp.plan_owners(params, wb, 5, 16)
        ra, rb = plan_owners_ref(params, wa, 5, 16), plan_owners_ref(params, wb, 5, 16)
        (am, at), (bm, bt) = mfsdp.placements(pa), mfsdp.placements(pb)
        (ram, rat), (rbm, rbt) = _ref_placements(ra), _ref_placements(rb)
        for r in range(wa):   # reduce: model layout -> owner buffers
            assert [g.as_dict() for g in mfsdp.placement_segments(model, am, r)] == \
                placement_segments_ref(model_ref, ram, r)
            assert [g.as_dict() for g in mfsdp.placement_segments(model, at, r)] == \
                placement_segments_ref(model_ref, rat, r)
        for r in range(wb):   # reshard: plan a -> plan b
            assert [g.as_dict() for g in mfsdp.placement_segments(am, bm, r)] == placement_segments_ref(ram, rbm, r)
            assert [g.as_dict() for g in mfsdp.placement_segments(at, bt, r)] == placement_segments_ref(rat, rbt, r)


def test_segment_errors(mfsdp):
    lib = mfsdp.raw_lib()
    A, B, D = 0x10000000, 0x20000000, 0x30000000

    def seg(so, do, n, si=0):
        g = mfsdp.Segment()
        g.src_offset, g.dst_offset, g.numel, g.src_index = so, do, n, si
        return g

    def call(segs, srcs=(A, B), sizes=(1000, 1000), mode=0, dst=D, dn=1000, sdt=1, ddt=1):
        ptrs = (ctypes.c_void_p * len(srcs))(*srcs)
        sz = (ctypes.c_int64 * len(sizes))(*sizes)
        arr = (mfsdp.Segment * max(len(segs), 1))(*segs)
        return lib.mfsdp_segment_copy(ptrs, sz, len(srcs), sdt, arr, len(segs), mode, dst, ddt, dn, None)
    assert call([]) == mfsdp.OK
    assert call([seg(0, 0, 10)], mode=2) == mfsdp.ERR_INVALID_ARG
    assert call([seg(0, 0, 10)], sdt=3) == mfsdp.ERR_UNSUPPORTED_DTYPE
    assert call([seg(0, 0, 10)], dst=D + 8) == mfsdp.ERR_MISALIGNED
    assert call([seg(0, 0, 10)], srcs=(A + 2, B)) == mfsdp.ERR_MISALIGNED
    assert call([seg(995, 0, 10)]) == mfsdp.ERR_OUT_OF_BOUNDS
    assert call([seg(0, 995, 10)]) == mfsdp.ERR_OUT_OF_BOUNDS
    assert call([seg(0, 0, 10)], sizes=(1000, 5)) == mfsdp.ERR_OUT_OF_BOUNDS      # reduce reads every source
    assert call([seg(0, 0, 10, si=2)], mode=1) == mfsdp.ERR_INVALID_ARG
    assert call([seg(0, 0, 10), seg(20, 5, 10)]) == mfsdp.ERR_OVERLAP
    assert call([seg(0, 0, 10)], dst=A + 64) == mfsdp.ERR_OVERLAP                  # dst inside a source
    assert call([seg(0, 0, 10)], srcs=tuple([A] * 65), sizes=tuple([1000] * 65)) == mfsdp.ERR_INVALID_ARG
    # placement mapping: a parameter missing from the source, or placed twice
    p = mfsdp.Placement(); p.param_id, p.owner, p.offset, p.numel = 3, 0, 0, 10
    q = mfsdp.Placement(); q.param_id, q.owner, q.offset, q.numel = 4, 0, 16, 10
    with pytest.raises(mfsdp.MfsdpError):
        mfsdp.placement_segments([p], [q], 0)
    with pytest.raises(mfsdp.MfsdpError):
        mfsdp.placement_segments([p, p], [p], 0)
