"""Owner-shard checkpoints on the host (no GPU): the file layout the header
documents, written out here byte by byte with struct and FNV-1a-64 from its
definition; round trips of ragged ranks (every float bit pattern kept);
damaged, truncated and foreign files refused; and resharding a W = 8 plan to
W = 3 through the library's placement segments, checked parameter by
parameter against the oracle's gather.

MatrixFSDP -- Abstract: "owner-shard checkpoint resharding"; FAQ: MatrixShard
metadata carries the owner plan through optimizer routing and resharding.
"""
import struct

import numpy as np
import pytest

from oracle import segment_gather_ref
from matrix_optimizers_under_gb300 import workloads as W


def fnv1a64(data: bytes) -> int:
    h = 0xCBF29CE484222325
    for b in data:
        h ^= b
        h = (h * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF
    return h


def rank_state(plan, r, seed):
    rng = np.random.default_rng(seed)
    mom = rng.standard_normal(plan.rank_matrix_elems[r]).astype(np.float32)
    tail = [rng.standard_normal(plan.rank_tail_elems[r]).astype(np.float32) for _ in range(3)]
    return mom, tail


def test_file_layout_is_the_documented_one(mfsdp, tmp_path):
    s = mfsdp.make_shard(128, 3, 5, param_id=7, owner=1)
    s.cost = 0x0102030405060708
    t = mfsdp.TailShard()
    t.param_id, t.owner, t.offset, t.numel = 2, 1, 4, 3
    mom = np.arange(128 + 15, dtype=np.float32) * np.float32(0.5)
    mom[0], mom[1], mom[2] = -0.0, np.inf, np.float32(1e-45)
    tp, tm, tv = (np.arange(8, dtype=np.float32) + k for k in (1, 10, 100))
    path = str(tmp_path / "r1.ck")
    mfsdp.checkpoint_save(path, 3, 1, 5, 128, [s], [t], mom, tp, tm, tv, adam_step=42)
    raw = open(path, "rb").read()
    body = b"MFSDPCK1" + struct.pack("<I", 1) + struct.pack("<5i", 3, 1, 5, 1, 1) + struct.pack("<4q", 128, 143, 8, 42)
    body += struct.pack("<iiqqqiiQ", 7, 1, 128, 3, 5, 0, 0, 0x0102030405060708)
    body += struct.pack("<iiqq", 2, 1, 4, 3)
    body += mom.astype("<f4").tobytes() + b"".join(x.astype("<f4").tobytes() for x in (tp, tm, tv))
    assert raw == body + struct.pack("<Q", fnv1a64(body))
    h = mfsdp.CheckpointHeader()
    h.world, h.rank, h.ns_steps, h.n_matrix, h.n_tail = 3, 1, 5, 1, 1
    h.align_elems, h.matrix_elems, h.tail_elems, h.adam_step = 128, 143, 8, 42
    assert mfsdp.raw_lib().mfsdp_checkpoint_bytes(h) == len(raw)
    ck = mfsdp.checkpoint_load(path)
    assert np.array_equal(ck.momentum.view(np.uint32), mom.view(np.uint32))   # -0, inf, subnormal kept
    assert (ck.header.world, ck.header.rank, ck.header.adam_step) == (3, 1, 42)
    assert ck.matrix_shards[0].as_dict() == s.as_dict() and ck.tail_shards[0].as_dict() == t.as_dict()


def test_round_trip_ragged_ranks(mfsdp, tmp_path):
    params = W.ragged_params(9, 40)
    plan = mfsdp.plan_owners(params, 3, 5, 128)
    for r in range(3):
        mom, tail = rank_state(plan, r, r)
        path = str(tmp_path / f"r{r}.ck")
        mfsdp.checkpoint_save(path, 3, r, 5, 128, plan.rank_matrices(r), plan.rank_tails(r), mom, *tail,
                              adam_step=3)
        ck = mfsdp.checkpoint_load(path)
        assert [s.as_dict() for s in ck.matrix_shards] == [s.as_dict() for s in plan.rank_matrices(r)]
        assert [s.as_dict() for s in ck.tail_shards] == [s.as_dict() for s in plan.rank_tails(r)]
        assert np.array_equal(ck.momentum, mom)
        for a, b in zip((ck.tail_p, ck.tail_m, ck.tail_v), tail):
            assert np.array_equal(a, b)


def test_damaged_and_foreign_files_are_refused(mfsdp, tmp_path):
    import ctypes
    params = W.ragged_params(10, 12)
    plan = mfsdp.plan_owners(params, 2, 5, 128)
    mom, tail = rank_state(plan, 0, 1)
    path = str(tmp_path / "r0.ck")
    mfsdp.checkpoint_save(path, 2, 0, 5, 128, plan.rank_matrices(0), plan.rank_tails(0), mom, *tail, adam_step=1)
    good = open(path, "rb").read()

    def status(data):
        p = str(tmp_path / "bad.ck")
        open(p, "wb").write(data)
        with pytest.raises(mfsdp.MfsdpError) as e:
            mfsdp.checkpoint_load(p)
        return e.value.status

    flipped = bytearray(good)
    flipped[len(good) // 2] ^= 0x10                       # one bit of the payload
    assert status(bytes(flipped)) == mfsdp.ERR_FORMAT
    assert status(good[:-1]) == mfsdp.ERR_FORMAT          # truncated
    assert status(good + b"\0") == mfsdp.ERR_FORMAT       # trailing bytes
    assert status(b"MFSDPCK2" + good[8:]) == mfsdp.ERR_FORMAT
    assert status(good[:8] + struct.pack("<I", 2) + good[12:]) == mfsdp.ERR_FORMAT
    with pytest.raises(mfsdp.MfsdpError) as e:
        mfsdp.checkpoint_load(str(tmp_path / "missing.ck"))
    assert e.value.status == mfsdp.ERR_IO
    # capacities below the file's counts
    lib = mfsdp.raw_lib()
    h = mfsdp.CheckpointHeader()
    assert lib.mfsdp_checkpoint_read_header(path.encode(), ctypes.byref(h)) == mfsdp.OK
    buf = np.empty(h.matrix_elems, np.float32)
    tb = [np.empty(h.tail_elems, np.float32) for _ in range(3)]
    marr = (mfsdp.MatrixShard * max(h.n_matrix, 1))()
    tarr = (mfsdp.TailShard * max(h.n_tail, 1))()
    assert lib.mfsdp_checkpoint_read(path.encode(), ctypes.byref(h), marr, h.n_matrix - 1, tarr, h.n_tail,
                                     buf.ctypes.data, h.matrix_elems, *[t.ctypes.data for t in tb],
                                     h.tail_elems) == mfsdp.ERR_WORKSPACE_TOO_SMALL
    # a table that does not belong to the rank, or leaves its buffer
    other = plan.rank_matrices(1)
    with pytest.raises(mfsdp.MfsdpError) as e:
        mfsdp.checkpoint_save(path, 2, 0, 5, 128, other, [], mom, *[t[:0] for t in tail], adam_step=1)
    assert e.value.status == mfsdp.ERR_OUT_OF_BOUNDS
    with pytest.raises(mfsdp.MfsdpError) as e:
        mfsdp.checkpoint_save(path, 2, 0, 5, 128, plan.rank_matrices(0), [], mom[:-200], *[t[:0] for t in tail],
                              adam_step=1)
    assert e.value.status == mfsdp.ERR_OUT_OF_BOUNDS


def test_reshard_eight_ranks_to_three_on_host(mfsdp, tmp_path):
    """W = 8 checkpoints reloaded under W = 3: the library's placement
    segments, applied with the oracle's gather on the host buffers, put every
    parameter's state at its new owner and offset unchanged."""
    params = W.llama_param_table(2, 512, 1376, 128)
    old = mfsdp.plan_owners(params, 8, 5, 128)
    states = {}
    for r in range(8):
        mom, tail = rank_state(old, r, 100 + r)
        states[r] = (mom, tail)
        mfsdp.checkpoint_save(str(tmp_path / f"w8r{r}.ck"), 8, r, 5, 128, old.rank_matrices(r), old.rank_tails(r),
                              mom, *tail, adam_step=1)
    cks = [mfsdp.checkpoint_load(str(tmp_path / f"w8r{r}.ck")) for r in range(8)]

    def placements(shards, key):
        out = []
        for s in shards:
            p = mfsdp.Placement()
            p.param_id, p.owner, p.offset = s.param_id, s.owner, s.offset
            p.numel = s.rows * s.cols if key == "m" else s.numel
            out.append(p)
        return out
    src_m = placements([s for ck in cks for s in ck.matrix_shards], "m")
    src_t = placements([s for ck in cks for s in ck.tail_shards], "t")
    new = mfsdp.plan_owners(params, 3, 5, 128)
    dst_m = placements(new.matrix_shards, "m")
    dst_t = placements(new.tail_shards, "t")
    for r in range(3):
        seg_m = [g.as_dict() for g in mfsdp.placement_segments(src_m, dst_m, r)]
        seg_t = [g.as_dict() for g in mfsdp.placement_segments(src_t, dst_t, r)]
        mom = segment_gather_ref([ck.momentum for ck in cks], seg_m, new.rank_matrix_elems[r])
        tails = [segment_gather_ref([getattr(ck, f) for ck in cks], seg_t, new.rank_tail_elems[r])
                 for f in ("tail_p", "tail_m", "tail_v")]
        for s in new.rank_matrices(r):
            o = next(x for x in old.matrix_shards if x.param_id == s.param_id)
            n = s.rows * s.cols
            assert np.array_equal(mom[s.offset:s.offset + n], states[o.owner][0][o.offset:o.offset + n])
        for s in new.rank_tails(r):
            o = next(x for x in old.tail_shards if x.param_id == s.param_id)
            for k in range(3):
                assert np.array_equal(tails[k][s.offset:s.offset + s.numel],
                                      states[o.owner][1][k][o.offset:o.offset + s.numel])
