"""The owner step for callers that cannot allocate device memory.

Some callers cannot hand the library a workspace: a plug-in running inside a
framework that owns every device allocation, a callback that must not
allocate, a C program that links only this library.  For them
mfsdp_muon_owner_step_static_scratch uses a fixed device array inside the
library as scratch.  This file checks, through the C ABI, that two calls in a
row give bit for bit the same updates and momentum as the regular entry point
(the same kernels on the same inputs; only the scratch's address differs), and
that an owner set too large for the array is rejected before anything runs.

It is named to be collected last, so that a run stopping at the first failure
has run every other test first; it passes alone in a fresh process too (the
first call on the device sets the array's address up).
"""
import numpy as np
import pytest

from matrix_optimizers_under_gb300 import workloads as W
from tests import helpers as H

torch = pytest.importorskip("torch")


def _grads(w, shards, numel, step):
    """Seeded gradient buffer for one call (a different draw per step)."""
    buf = H.build_grad_buffer(w, shards, numel)
    if step:
        rng = np.random.default_rng(100 + step)
        vals = (rng.standard_normal(numel) * w.grad_scale).astype(np.float32)
        fresh = W.f32_to_bf16_bits(vals)
        for s in shards:
            buf[s.offset:s.offset + s.rows * s.cols] = fresh[s.offset:s.offset + s.rows * s.cols]
    return torch.from_numpy(buf.view(np.int16)).cuda().view(torch.bfloat16)


@pytest.mark.gpu
def test_static_scratch_matches_workspace_entry_point(mfsdp):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    w = W.get("gpt2_block")
    plan = mfsdp.plan_owners(w.param_table(), w.world, w.ns_steps, w.align_elems)
    shards = plan.rank_matrices(0)
    numel = plan.rank_matrix_elems[0]
    assert mfsdp.muon_workspace_bytes(shards) <= mfsdp.STATIC_SCRATCH_BYTES
    kw = dict(beta=w.beta, ns_steps=w.ns_steps, coeffs=w.ns_coeffs, eps=w.ns_eps)
    dev = torch.device("cuda:0")
    mom_ref = torch.zeros(numel, dtype=torch.float32, device=dev)
    mom_new = torch.zeros(numel, dtype=torch.float32, device=dev)
    ws = torch.empty(mfsdp.muon_workspace_bytes(shards), dtype=torch.uint8, device=dev)
    for step in range(2):                      # two calls in a row
        g = _grads(w, shards, numel, step)
        upd_ref = torch.zeros(numel, dtype=torch.bfloat16, device=dev)
        upd_new = torch.zeros(numel, dtype=torch.bfloat16, device=dev)
        mfsdp.muon_owner_step(shards, g, mom_ref, upd_ref, ws, **kw)
        mfsdp.muon_owner_step_static_scratch(shards, g, mom_new, upd_new, **kw)
        torch.cuda.synchronize()
        for s in shards:
            seg = slice(s.offset, s.offset + s.rows * s.cols)
            assert torch.equal(upd_new[seg].view(torch.int16), upd_ref[seg].view(torch.int16)), (step, s.param_id)
            assert torch.equal(mom_new[seg].view(torch.int32), mom_ref[seg].view(torch.int32)), (step, s.param_id)
        st, detail = mfsdp.muon_static_scratch_status()
        assert st == mfsdp.OK, (step, st, detail)

    # A further call allocates nothing: torch's allocator and the device's free
    # memory are the same before and after it.
    g = _grads(w, shards, numel, 2)
    upd_new = torch.zeros(numel, dtype=torch.bfloat16, device=dev)
    torch.cuda.synchronize()
    alloc0, free0 = torch.cuda.memory_allocated(dev), torch.cuda.mem_get_info(dev)[0]
    mfsdp.muon_owner_step_static_scratch(shards, g, mom_new, upd_new, **kw)
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated(dev) == alloc0
    assert torch.cuda.mem_get_info(dev)[0] == free0

    # an owner set whose scratch exceeds the fixed array is refused up front
    big = [mfsdp.make_shard(0, 4096, 4096)]
    assert mfsdp.muon_workspace_bytes(big) > mfsdp.STATIC_SCRATCH_BYTES
    with pytest.raises(mfsdp.MfsdpError) as e:
        mfsdp.muon_owner_step_static_scratch(big, torch.zeros(4096 * 4096, dtype=torch.bfloat16, device=dev),
                                             torch.zeros(4096 * 4096, device=dev),
                                             torch.zeros(4096 * 4096, dtype=torch.bfloat16, device=dev), **kw)
    assert e.value.status == mfsdp.ERR_WORKSPACE_TOO_SMALL
