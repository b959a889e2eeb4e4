"""The owner step captured in a CUDA graph.

Every launch of a step carries its tables as kernel parameters (the Newton-
Schulz kernel also its tensor maps) and the workspace counters are reset by
memset nodes, so a captured step replays without host work.  Two replays
must equal two eager steps bit for bit, momentum carried from one step to the
next included.
"""
import numpy as np
import pytest

from matrix_optimizers_under_gb300 import workloads as W
from tests import helpers as H

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def test_owner_step_in_cuda_graph(mfsdp):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda:0")
    w = W.get("gpt2_block")
    plan = mfsdp.plan_owners(w.param_table(), w.world, w.ns_steps, w.align_elems)
    r = H.heaviest_rank(plan)
    shards, numel = plan.rank_matrices(r), plan.rank_matrix_elems[r]
    grad_np = H.build_grad_buffer(w, shards, numel, only={s.param_id for s in shards})
    grad = torch.from_numpy(grad_np.view(np.int16)).to(dev).view(torch.bfloat16)
    kw = dict(beta=0.95, ns_steps=w.ns_steps, coeffs=W.NS_COEFFS, eps=W.NS_EPS)

    def buffers():
        return (torch.zeros(numel, dtype=torch.float32, device=dev),
                torch.zeros(numel, dtype=torch.bfloat16, device=dev),
                torch.empty(mfsdp.muon_workspace_bytes(shards), dtype=torch.uint8, device=dev))

    mom_e, upd_e, ws_e = buffers()
    eager = []
    for _ in range(2):
        mfsdp.muon_owner_step(shards, grad, mom_e, upd_e, ws_e, **kw)
        eager.append((upd_e.clone(), mom_e.clone()))
    torch.cuda.synchronize()

    mom_g, upd_g, ws_g = buffers()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        mfsdp.muon_owner_step(shards, grad, mom_g, upd_g, ws_g, **kw)
    for k in range(2):
        graph.replay()
        torch.cuda.synchronize()
        st, detail = mfsdp.muon_device_status(ws_g)
        assert st == mfsdp.OK, (st, detail)
        assert torch.equal(upd_g.view(torch.int16), eager[k][0].view(torch.int16)), f"update of replay {k}"
        assert torch.equal(mom_g, eager[k][1]), f"momentum of replay {k}"
