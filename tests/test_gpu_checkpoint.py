"""Owner-shard checkpoint resharding on the GPU (MatrixFSDP -- Abstract:
"owner-shard checkpoint resharding"; FAQ: MatrixShard metadata carries the
owner plan through optimizer routing and resharding).

A two-layer Llama-shaped stack is planned over 8 simulated ranks; each rank
takes one optimizer step (owner step and AdamW tail) and saves its state and
tables to a checkpoint.  The 8 files are reloaded under a 3-rank plan: each
new rank's momentum and tail state are gathered from the old ranks' buffers by
the library's segment kernel along the placement segments, and each new rank
takes the second step.  Every matrix's momentum and update, and every tail
element, match the fp64 oracle continuing from the original state; the
gathered state equals the saved one bit for bit.
"""
import numpy as np
import pytest

from oracle import adamw_ref, bf16_bits_to_f64, muon_matrix_ref
from matrix_optimizers_under_gb300 import workloads as W
from tests import helpers as H

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

A, B, C = W.NS_COEFFS
LR, BETAS, EPS, WD = 1e-3, (0.9, 0.95), 1e-8, 0.1


def _grad_bits(pid, rows, cols, step):
    rng = np.random.default_rng([77, pid, step])
    return W.f32_to_bf16_bits((rng.standard_normal(rows * cols) * 1e-3).astype(np.float32))


def _tail_vals(pid, n, salt):
    rng = np.random.default_rng([78, pid, salt])
    return (rng.standard_normal(n) * 1e-3).astype(np.float32)


def _flat_grads(shards, numel, step):
    buf = np.zeros(numel, np.uint16)
    for s in shards:
        buf[s.offset:s.offset + s.rows * s.cols] = _grad_bits(s.param_id, s.rows, s.cols, step)
    return buf


def _flat_tail(tails, numel, salt):
    buf = np.zeros(numel, np.float32)
    for t in tails:
        buf[t.offset:t.offset + t.numel] = _tail_vals(t.param_id, t.numel, salt)
    return buf


def _placements(mfsdp, shards, matrix):
    out = []
    for s in shards:
        p = mfsdp.Placement()
        p.param_id, p.owner, p.offset = s.param_id, s.owner, s.offset
        p.numel = s.rows * s.cols if matrix else s.numel
        out.append(p)
    return out


def test_reshard_eight_ranks_to_three_and_continue(mfsdp, tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda:0")
    params = W.llama_param_table(2, 512, 1376, 128)
    kw = dict(beta=0.95, ns_steps=5, coeffs=W.NS_COEFFS, eps=W.NS_EPS)

    def to_dev_bits(bits):
        return torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)

    # ---- step 1 on 8 ranks, then save
    old = mfsdp.plan_owners(params, 8, 5, 128)
    for r in range(8):
        sh, tl = old.rank_matrices(r), old.rank_tails(r)
        n, nt = old.rank_matrix_elems[r], old.rank_tail_elems[r]
        mom = torch.zeros(max(n, 1), dtype=torch.float32, device=dev)[:n]
        if sh:
            g = to_dev_bits(_flat_grads(sh, n, 1))
            upd = torch.zeros(n, dtype=torch.bfloat16, device=dev)
            ws = torch.empty(mfsdp.muon_workspace_bytes(sh), dtype=torch.uint8, device=dev)
            mfsdp.muon_owner_step(sh, g, mom, upd, ws, **kw)
            assert mfsdp.muon_device_status(ws)[0] == mfsdp.OK
        tp = torch.from_numpy(_flat_tail(tl, nt, 0)).to(dev)
        tm, tv = torch.zeros_like(tp), torch.zeros_like(tp)
        if nt:
            tg = torch.from_numpy(_flat_tail(tl, nt, 1)).to(dev)
            mfsdp.adamw_tail_step(tp, tg, tm, tv, lr=LR, beta1=BETAS[0], beta2=BETAS[1], eps=EPS, wd=WD, step=1)
        torch.cuda.synchronize()
        mfsdp.checkpoint_save(str(tmp_path / f"r{r}.ck"), 8, r, 5, 128, sh, tl, mom, tp, tm, tv, adam_step=1)

    # ---- reload under 3 ranks: gather each new rank's state from the old buffers
    cks = [mfsdp.checkpoint_load(str(tmp_path / f"r{r}.ck")) for r in range(8)]
    assert all(ck.header.world == 8 and ck.header.adam_step == 1 for ck in cks)

    def dev_buf(a):
        return torch.from_numpy(a).to(dev) if a.size else torch.zeros(1, device=dev)
    old_mom = [dev_buf(ck.momentum) for ck in cks]
    old_tail = {f: [dev_buf(getattr(ck, f)) for ck in cks] for f in ("tail_p", "tail_m", "tail_v")}
    src_m = _placements(mfsdp, [s for ck in cks for s in ck.matrix_shards], True)
    src_t = _placements(mfsdp, [s for ck in cks for s in ck.tail_shards], False)
    new = mfsdp.plan_owners(params, 3, 5, 128)
    dst_m = _placements(mfsdp, new.matrix_shards, True)
    dst_t = _placements(mfsdp, new.tail_shards, False)
    g1_of = {s.param_id: _grad_bits(s.param_id, s.rows, s.cols, 1) for s in old.matrix_shards}
    checked = 0
    for r in range(3):
        sh, tl = new.rank_matrices(r), new.rank_tails(r)
        n, nt = new.rank_matrix_elems[r], new.rank_tail_elems[r]
        mom = torch.full((n,), float("nan"), dtype=torch.float32, device=dev)
        mfsdp.segment_copy(old_mom, mfsdp.placement_segments(src_m, dst_m, r), mfsdp.SEGMENT_GATHER, mom)
        tails = {}
        for f in ("tail_p", "tail_m", "tail_v"):
            tails[f] = torch.full((max(nt, 1),), float("nan"), dtype=torch.float32, device=dev)[:nt]
            if nt:
                mfsdp.segment_copy(old_tail[f], mfsdp.placement_segments(src_t, dst_t, r), mfsdp.SEGMENT_GATHER,
                                   tails[f])
        torch.cuda.synchronize()
        for t in tl:                                 # the gathered tail state is the saved one, bit for bit
            o = next(x for x in old.tail_shards if x.param_id == t.param_id)
            for f in ("tail_p", "tail_m", "tail_v"):
                assert np.array_equal(tails[f][t.offset:t.offset + t.numel].cpu().numpy(),
                                      getattr(cks[o.owner], f)[o.offset:o.offset + t.numel]), (t.param_id, f)
        mom_np = mom.cpu().numpy()
        for s in sh:                                 # the gathered momentum is the saved G1, bit for bit
            assert np.array_equal(mom_np[s.offset:s.offset + s.rows * s.cols],
                                  bf16_bits_to_f64(g1_of[s.param_id]).astype(np.float32)), s.param_id

        # ---- step 2 on the new rank
        g2 = _flat_grads(sh, n, 2)
        upd = torch.zeros(n, dtype=torch.float32, device=dev)
        ws = torch.empty(mfsdp.muon_workspace_bytes(sh), dtype=torch.uint8, device=dev)
        mfsdp.muon_owner_step(sh, to_dev_bits(g2), mom, upd, ws, **kw)
        assert mfsdp.muon_device_status(ws)[0] == mfsdp.OK
        if nt:
            mfsdp.adamw_tail_step(tails["tail_p"], torch.from_numpy(_flat_tail(tl, nt, 2)).to(dev), tails["tail_m"],
                                  tails["tail_v"], lr=LR, beta1=BETAS[0], beta2=BETAS[1], eps=EPS, wd=WD, step=2)
        torch.cuda.synchronize()
        upd_np, mom_np = upd.cpu().numpy(), mom.cpu().numpy()
        for s in sh:
            seg = slice(s.offset, s.offset + s.rows * s.cols)
            G1 = bf16_bits_to_f64(g1_of[s.param_id]).reshape(s.rows, s.cols)
            G2 = bf16_bits_to_f64(g2[seg]).reshape(s.rows, s.cols)
            M_ref, O_ref = muon_matrix_ref(G2, G1, 0.95, False, 5, A, B, C, W.NS_EPS)
            M = mom_np[seg].astype(np.float64).reshape(s.rows, s.cols)
            assert np.all(np.abs(M - M_ref) <= H.MOM_REL * (0.95 * np.abs(G1) + np.abs(G2)) + 1e-30), s.param_id
            O = upd_np[seg].astype(np.float64).reshape(s.rows, s.cols)
            assert H.rel_fro(O, O_ref) <= H.ns_tol(s.rows, s.cols), (s.param_id, H.rel_fro(O, O_ref))
            H.check_blocks(O, O_ref, f"param {s.param_id}")
            checked += 1
        for t in tl:
            # the state saved after step 1: the oracle's first step, and what the gather brought over
            p0, g1, g2t = (_tail_vals(t.param_id, t.numel, k) for k in (0, 1, 2))
            o = next(x for x in old.tail_shards if x.param_id == t.param_id)
            saved = [getattr(cks[o.owner], f)[o.offset:o.offset + t.numel] for f in ("tail_p", "tail_m", "tail_v")]
            ref1 = adamw_ref(p0, g1, np.zeros(t.numel), np.zeros(t.numel), LR, BETAS[0], BETAS[1], EPS, WD, 1)
            for got, ref in zip(saved, ref1):
                assert H.adam_err(got, ref) <= H.ADAM_REL, t.param_id
            # step 2 continues from the saved fp32 state, as the next step would
            ref2 = adamw_ref(*[x.astype(np.float64) for x in (saved[0], g2t, saved[1], saved[2])], LR, BETAS[0],
                             BETAS[1], EPS, WD, 2)
            seg = slice(t.offset, t.offset + t.numel)
            for got, ref in zip((tails["tail_p"], tails["tail_m"], tails["tail_v"]), ref2):
                assert H.adam_err(got[seg].cpu().numpy(), ref) <= H.ADAM_REL, t.param_id
    assert checked == sum(1 for p in params if p[2] == W.KIND_MATRIX)
