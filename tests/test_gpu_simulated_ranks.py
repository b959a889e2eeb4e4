"""Every simulated rank of an owner plan, run one after another on one GPU.

MatrixFSDP: Communication-Free Matrix Optimizers Under ZeRO-3 Parameter
Sharding -- Abstract: each 2D weight is owned whole by exactly one rank (the
others hold empty shards), and the owner-local update matches full-matrix
Muon.  Over the GPT-2 block's parameters and world sizes 1, 2, 3 and 8 (so
some ranks own no matrix): every matrix is updated by exactly one rank; its
update is bit-identical whichever world size and rank own it; it matches the
fp64 oracle; and nothing outside a rank's segments is written.
"""
import numpy as np
import pytest

from matrix_optimizers_under_gb300 import workloads as W
from tests import helpers as H
from tests.test_gpu_parity import check_matrix, check_padding, run_step

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def test_every_simulated_rank(mfsdp):
    w = W.get("gpt2_block")
    table = w.param_table()
    first = {}                                   # param id -> update bits of its first owner
    for world in (1, 2, 3, 8):
        plan = mfsdp.plan_owners(table, world, w.ns_steps, w.align_elems)
        seen = []
        for r in range(world):
            shards = plan.rank_matrices(r)
            numel = plan.rank_matrix_elems[r]
            if not shards:
                assert numel == 0
                continue
            grad = H.build_grad_buffer(w, shards, numel)
            mom0 = np.zeros(numel, np.float32)
            upd, mom, _ = run_step(mfsdp, shards, grad, mom0, update_dtype=torch.bfloat16)
            check_padding(upd, mom, shards, numel)
            for s in shards:
                seen.append(s.param_id)
                bits = upd[s.offset:s.offset + s.rows * s.cols].view(np.uint32).copy()
                if s.param_id in first:
                    assert np.array_equal(first[s.param_id], bits), \
                        f"param {s.param_id}: update differs at world size {world}, rank {r}"
                else:
                    first[s.param_id] = bits
                    check_matrix(s, upd, mom, grad, mom0, ns_steps=w.ns_steps)
        matrices = sorted(s.param_id for s in plan.matrix_shards)
        assert sorted(seen) == matrices and len(set(seen)) == len(seen), f"world {world}: ownership"
        if world == 8:
            assert sum(1 for r in range(world) if not plan.rank_matrices(r)) == 8 - len(matrices)
