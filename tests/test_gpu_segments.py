"""GPU parity of the owner-segment reduce and owner-shard resharding.

MatrixFSDP -- Abstract: the ordinary backward reduction lands each matrix's full
gradient on its owner (an uneven, deterministic reduce over owner segments);
owner-shard checkpoint resharding moves shards between layouts.  Simulated
ranks' local gradients are separate flat buffers in the model layout.
  * REDUCE: bit-exact against the same sum taken in rank order in fp32 and
    rounded once (NumPy emulation), and within that rounding of the fp64
    oracle; elements outside the segments keep their NaN canaries.
  * GATHER: a plan-to-plan reshard is an exact copy (bitwise).
"""
import numpy as np
import pytest

from oracle import segment_gather_ref, segment_reduce_ref
from matrix_optimizers_under_gb300 import workloads as W
from tests import helpers as H

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _bf16_dev(bits: np.ndarray, dev):
    return torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)


def _emulate_reduce(srcs_f32, segs, n, out_bf16):
    """Rank-order fp32 sum, rounded once: what the kernel computes."""
    out = np.full(n, np.nan, np.float32)
    for g in segs:
        acc = np.zeros(g.numel, np.float32)
        for s in srcs_f32:
            acc = (acc + s[g.src_offset:g.src_offset + g.numel]).astype(np.float32)
        out[g.dst_offset:g.dst_offset + g.numel] = acc
    if out_bf16:
        return H.bf16_bits_to_f32(W.f32_to_bf16_bits(out))
    return out


@pytest.mark.parametrize("world", [1, 3, 8])
def test_owner_segment_reduce(mfsdp, world):
    dev = _dev()
    params = W.ragged_params(world + 20, 40, max_dim=300)
    model = mfsdp.model_placements(params, 128)
    _, total = mfsdp.model_layout(params, 128)
    plan = mfsdp.plan_owners(params, world, 5, 128)
    mp, tp = mfsdp.placements(plan)
    rng = np.random.default_rng(world)
    bits = [W.f32_to_bf16_bits((rng.standard_normal(total) * 1e-3).astype(np.float32)) for _ in range(world)]
    srcs_f32 = [H.bf16_bits_to_f32(b) for b in bits]
    srcs = [_bf16_dev(b, dev) for b in bits]
    for r in range(world):
        for pl, n, out_bf16 in ((mp, plan.rank_matrix_elems[r], True), (tp, plan.rank_tail_elems[r], False)):
            if n == 0:
                continue
            segs = mfsdp.placement_segments(model, pl, r)
            dt = torch.bfloat16 if out_bf16 else torch.float32
            out = torch.full((n,), float("nan"), dtype=dt, device=dev)
            mfsdp.segment_copy(srcs, segs, mfsdp.SEGMENT_REDUCE, out)
            got = out.float().cpu().numpy()
            want = _emulate_reduce(srcs_f32, segs, n, out_bf16)
            assert np.array_equal(np.isnan(got), np.isnan(want)), "canaries"
            assert np.array_equal(np.nan_to_num(got).view(np.uint32), np.nan_to_num(want).view(np.uint32))
            ref = segment_reduce_ref(srcs_f32, [g.as_dict() for g in segs], n)
            mask = ~np.isnan(ref)
            mag = sum(np.abs(np.nan_to_num(segment_reduce_ref([s], [g.as_dict() for g in segs], n))) for s in srcs_f32)
            bound = world * 2.0 ** -24 * mag + (2.0 ** -8 * np.abs(ref) if out_bf16 else 0.0)
            assert np.all(np.abs(got[mask] - ref[mask]) <= bound[mask] + 1e-30)
            out2 = torch.full((n,), float("nan"), dtype=dt, device=dev)
            mfsdp.segment_copy(srcs, segs, mfsdp.SEGMENT_REDUCE, out2)
            assert torch.equal(out.view(torch.int16 if out_bf16 else torch.int32),
                               out2.view(torch.int16 if out_bf16 else torch.int32)), "deterministic"


@pytest.mark.parametrize("worlds", [(4, 3), (2, 5), (8, 1)])
def test_reshard_gather_is_exact(mfsdp, worlds):
    dev = _dev()
    wa, wb = worlds
    params = W.ragged_params(31, 60, max_dim=260)
    pa, pb = mfsdp.plan_owners(params, wa, 5, 128), mfsdp.plan_owners(params, wb, 5, 128)
    (am, at), (bm, bt) = mfsdp.placements(pa), mfsdp.placements(pb)
    rng = np.random.default_rng(wa * 10 + wb)
    for a_pl, b_pl, a_ext, b_ext in ((am, bm, pa.rank_matrix_elems, pb.rank_matrix_elems),
                                     (at, bt, pa.rank_tail_elems, pb.rank_tail_elems)):
        olds = [rng.standard_normal(max(n, 1)).astype(np.float32) for n in a_ext]   # e.g. fp32 momentum
        srcs = [torch.from_numpy(o).to(dev) for o in olds]
        for r in range(wb):
            if b_ext[r] == 0:
                continue
            segs = mfsdp.placement_segments(a_pl, b_pl, r)
            out = torch.full((b_ext[r],), float("nan"), dtype=torch.float32, device=dev)
            mfsdp.segment_copy(srcs, segs, mfsdp.SEGMENT_GATHER, out)
            ref = segment_gather_ref(olds, [g.as_dict() for g in segs], b_ext[r])
            got = out.cpu().numpy().astype(np.float64)
            assert np.array_equal(np.isnan(got), np.isnan(ref))
            assert np.array_equal(got[~np.isnan(ref)], ref[~np.isnan(ref)])


@pytest.mark.slow
def test_reduce_full_model_sampled(mfsdp):
    """The 1.3B model, 8 simulated ranks, reduced onto the benched owner: sampled
    segments against the fp64 oracle computed from the same source bytes."""
    dev = _dev()
    w = W.get("llama_1p3b_rank")
    params = w.param_table()
    model = mfsdp.model_placements(params, 128)
    _, total = mfsdp.model_layout(params, 128)
    plan = mfsdp.plan_owners(params, w.world, w.ns_steps, w.align_elems)
    r = H.heaviest_rank(plan)
    mp, _ = mfsdp.placements(plan)
    gen = torch.Generator(device=dev).manual_seed(2)
    srcs = [(torch.randn(total, generator=gen, device=dev) * 1e-3).to(torch.bfloat16) for _ in range(w.world)]
    segs = mfsdp.placement_segments(model, mp, r)
    n = plan.rank_matrix_elems[r]
    out = torch.full((n,), float("nan"), dtype=torch.bfloat16, device=dev)
    mfsdp.segment_copy(srcs, segs, mfsdp.SEGMENT_REDUCE, out)
    torch.cuda.synchronize()
    for g in segs[:: max(1, len(segs) // 4)]:
        part = [s[g.src_offset:g.src_offset + g.numel].float().cpu().numpy() for s in srcs]
        ref = np.sum([p.astype(np.float64) for p in part], axis=0)
        got = out[g.dst_offset:g.dst_offset + g.numel].float().cpu().numpy()
        bound = 8 * 2.0 ** -24 * np.sum(np.abs(part), axis=0) + 2.0 ** -8 * np.abs(ref)
        assert np.all(np.abs(got - ref) <= bound + 1e-30)
    del srcs
