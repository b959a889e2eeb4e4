"""Host-side checks of the bench's single-kernel cases (no GPU).

The owner-segment reduce case that the full ncu capture of `segment_kernel`
runs on is a three-layer Llama-1.3B-shaped stack planned over 8 simulated
ranks.  Its layout is fixed here so that the sizes the profile quotes (model
elements per rank buffer, segments and elements of the heaviest owner) stay
true, and so that the case covers exactly that owner's matrices (MatrixFSDP --
Abstract: each owner holds whole matrices, described by offset, rows, cols).
"""
import pytest

import bench
from matrix_optimizers_under_gb300 import workloads as W


def test_segment_case_layout(mfsdp):
    table = W.llama_param_table(3, 2048, 5504, 2048)
    assert len(table) == 3 * 9 + 1
    plan = mfsdp.plan_owners(table, 8, 5, 128)
    owner = bench.heaviest_rank(plan)
    model = mfsdp.model_placements(table, 128)
    _, model_total = mfsdp.model_layout(table, 128)
    mp, _ = mfsdp.placements(plan)
    segs = mfsdp.placement_segments(model, mp, owner)
    owned = sum(s.numel for s in segs)
    # Every matrix of the owner, and nothing else, lands in its flat buffer.
    mine = [s for s in plan.matrix_shards if s.owner == owner]
    assert owned == sum(s.rows * s.cols for s in mine) == plan.rank_matrix_elems[owner]
    assert (model_total, len(segs), owned) == (151_795_712, 2, 22_544_384)
    # 8 bf16 sources read and one bf16 destination written per element.
    assert owned * 2 * 9 == 405_798_912


def test_kernel_case_flag_choices():
    with pytest.raises(SystemExit):
        bench.main(["--kernel", "momentum"])


def test_kernel_digest_ignores_comments():
    """The traffic figure is keyed by the Newton-Schulz kernel's code, not its
    comments or layout: a comment edit keeps the digest, a code edit changes it."""
    import os
    csrc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "matrix_optimizers_under_gb300",
                        "csrc")
    srcs = {n: open(os.path.join(csrc, n)).read() for n in bench.NS_SOURCES}
    base = bench.ns_source_digest(srcs)
    assert base == bench.ns_source_digest()
    commented = dict(srcs)
    commented["ns_gemm.cu"] = "// a new comment\n/* and a block\n comment */\n" + srcs["ns_gemm.cu"].replace("\n", "\n  ")
    assert bench.ns_source_digest(commented) == base
    changed = dict(srcs)
    changed["ptx.cuh"] = srcs["ptx.cuh"].replace("kSuspendHintNs = 32", "kSuspendHintNs = 64")
    assert changed["ptx.cuh"] != srcs["ptx.cuh"] and bench.ns_source_digest(changed) != base


def test_figures_leave_zero_matrices_out(mfsdp):
    """The MoE set's all-zero experts skip every Newton-Schulz product, so the
    bench's FLOP counts are those of its nonzero matrices only: 29.22 TFLOP
    dense over the 246 nonzero matrices of 272."""
    import types
    w = W.get("moe_skewed")
    plan = mfsdp.plan_owners(w.param_table(), w.world, w.ns_steps, w.align_elems)
    shards = plan.rank_matrices(bench.heaviest_rank(plan))
    active = [s for s in shards if s.param_id not in w.zero_params]
    assert (len(shards), len(active)) == (272, 246)
    step = types.SimpleNamespace(w=w, shards=shards, tail_numel=0)
    ms = {"ns": 1.0, "momentum": 1.0, "adamw": 0.0}
    fig = bench.figures(mfsdp, step, ms, {"bf16_tflops_sustained": 1.0, "hbm_gbs": 1.0})
    assert (fig["flops_dense"], fig["flops_executed"]) == mfsdp.muon_step_flops(active, w.ns_steps)
    assert round(fig["flops_dense"] / 1e12, 2) == 29.22


def test_ncu_figures_keyed_to_the_current_kernel():
    """The DRAM traffic and tensor-pipe share the bench reports for the headline
    owner set come from ncu captures of the kernel as committed: their key is
    the digest of the current Newton-Schulz sources."""
    digest = bench.ns_source_digest()
    for name in ("llama3_8b_rank", "llama_1p3b_rank"):
        assert (digest, name) in bench.NS_GEMM_TRAFFIC, name
        assert (digest, name) in bench.NS_TENSOR_ACTIVE, name
    assert all(0.0 < v <= 1.0 for v in bench.NS_TENSOR_ACTIVE.values())
