"""Failure detection on the GPU without a fault: a bounded wait runs out.

The test hook makes one tile of the next Newton-Schulz launch wait for a
dependency that nothing satisfies.  The first wait on it to pass its 2 s limit
(its pair's producers', the roles waiting behind them, or roles waiting to be
handed a tile) records the status word.  Every other wait of every CTA sees
the word and stops, so the kernel ends in bounded time.  The host reads
MFSDP_ERR_DEVICE_TIMEOUT with the waiting role and product in the detail
word.  The context stays usable: the next step succeeds and matches the
oracle.
"""
import time

import numpy as np
import pytest

from matrix_optimizers_under_gb300 import workloads as W
from tests import helpers as H
from tests.test_gpu_parity import check_matrix, run_step

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ROLE_DEPENDENCY = 5   # a wait for the stalled tile's dependency (producer, or a role behind it)
ROLE_TILE_FULL = 8    # a role of the stalled pair waiting for that tile to be handed out


def test_bounded_wait_gives_up_and_reports(mfsdp):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda:0")
    w = W.get("tiny")
    plan = mfsdp.plan_owners(w.param_table(), w.world, w.ns_steps, w.align_elems)
    r = H.heaviest_rank(plan)
    shards, numel = plan.rank_matrices(r), plan.rank_matrix_elems[r]
    grad_np = H.build_grad_buffer(w, shards, numel)
    grad = torch.from_numpy(grad_np.view(np.int16) if grad_np.dtype == np.uint16 else grad_np).to(dev)
    if grad_np.dtype == np.uint16:
        grad = grad.view(torch.bfloat16)
    mom = torch.zeros(numel, dtype=torch.float32, device=dev)
    upd = torch.zeros(numel, dtype=torch.float32, device=dev)
    ws = torch.empty(mfsdp.muon_workspace_bytes(shards), dtype=torch.uint8, device=dev)

    mfsdp.test_inject_stall(0)                     # the first tile of the next launch
    t0 = time.monotonic()
    mfsdp.muon_owner_step(shards, grad, mom, upd, ws, ns_steps=w.ns_steps, coeffs=W.NS_COEFFS, eps=W.NS_EPS)
    st, detail = mfsdp.muon_device_status(ws)      # synchronises
    waited = time.monotonic() - t0
    assert st == mfsdp.ERR_DEVICE_TIMEOUT, (st, detail)
    # Both waits hang on the stalled tile; the readers of its pair start
    # waiting first, so either may be the first to run out.
    assert detail & 0xFF in (ROLE_DEPENDENCY, ROLE_TILE_FULL), detail
    # the first wait to run out records its product: the stalled tile's (0),
    # or a later product of the same matrix whose wait started a little earlier
    assert 0 <= detail >> 8 < 3 * w.ns_steps, detail
    assert 1.5 < waited < 30.0, waited

    # The context is still usable and the hook has cleared itself.
    upd_np, mom_np, _ = run_step(mfsdp, shards, grad_np, np.zeros(numel, np.float32), update_dtype=torch.float32)
    for s in shards:
        check_matrix(s, upd_np, mom_np, grad_np, np.zeros(numel, np.float32), ns_steps=w.ns_steps)


def test_bounded_wait_in_a_gram_space_final_product(mfsdp):
    """The same for a tile of the Gram-space form's final product Q X0 (list
    position 3T): one 200 x 640 matrix runs 8 narrow tiles per iteration (A,
    P, and C with Q, two 128-wide tiles each) and then its 5 final tiles, so
    tile 40 is the first of those.  The wait that gives up records role 5 with
    product 3T, or role 8 (no product); the next step is correct."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda:0")
    shards = [mfsdp.make_shard(0, 200, 640)]
    assert mfsdp.muon_gram_space_layout(shards, 5)[0][0] == 1
    numel = 200 * 640
    rng = np.random.default_rng(8)
    grad_np = (rng.standard_normal(numel) * 1e-3).astype(np.float32)
    grad = torch.from_numpy(grad_np).to(dev)
    mom = torch.zeros(numel, dtype=torch.float32, device=dev)
    upd = torch.zeros(numel, dtype=torch.float32, device=dev)
    ws = torch.empty(mfsdp.muon_workspace_bytes(shards), dtype=torch.uint8, device=dev)

    mfsdp.test_inject_stall(40)
    t0 = time.monotonic()
    mfsdp.muon_owner_step(shards, grad, mom, upd, ws, ns_steps=5, coeffs=W.NS_COEFFS, eps=W.NS_EPS)
    st, detail = mfsdp.muon_device_status(ws)
    waited = time.monotonic() - t0
    assert st == mfsdp.ERR_DEVICE_TIMEOUT, (st, detail)
    assert (detail & 0xFF, detail >> 8) in ((ROLE_DEPENDENCY, 15), (ROLE_TILE_FULL, 0)), detail
    assert 1.5 < waited < 30.0, waited

    upd_np, mom_np, _ = run_step(mfsdp, shards, grad_np, np.zeros(numel, np.float32), update_dtype=torch.float32)
    check_matrix(shards[0], upd_np, mom_np, grad_np, np.zeros(numel, np.float32), ns_steps=5)


def test_static_scratch_timeout_is_reported(mfsdp):
    """The static-scratch entry point keeps its status word in the library's
    scratch array, out of the caller's reach: a bounded wait that gives up
    there is read back with mfsdp_muon_static_scratch_status, and the next
    call on the same array succeeds and clears it."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda:0")
    w = W.get("tiny")
    plan = mfsdp.plan_owners(w.param_table(), w.world, w.ns_steps, w.align_elems)
    r = H.heaviest_rank(plan)
    shards, numel = plan.rank_matrices(r), plan.rank_matrix_elems[r]
    grad_np = H.build_grad_buffer(w, shards, numel)
    grad = torch.from_numpy(grad_np).to(dev)
    kw = dict(beta=w.beta, ns_steps=w.ns_steps, coeffs=W.NS_COEFFS, eps=W.NS_EPS)

    mom = torch.zeros(numel, dtype=torch.float32, device=dev)
    upd = torch.zeros(numel, dtype=torch.float32, device=dev)
    mfsdp.test_inject_stall(0)
    mfsdp.muon_owner_step_static_scratch(shards, grad, mom, upd, **kw)
    st, detail = mfsdp.muon_static_scratch_status()     # synchronises
    assert st == mfsdp.ERR_DEVICE_TIMEOUT, (st, detail)
    assert detail & 0xFF in (ROLE_DEPENDENCY, ROLE_TILE_FULL), detail

    mom = torch.zeros(numel, dtype=torch.float32, device=dev)
    upd = torch.zeros(numel, dtype=torch.float32, device=dev)
    mfsdp.muon_owner_step_static_scratch(shards, grad, mom, upd, **kw)
    st, detail = mfsdp.muon_static_scratch_status()
    assert st == mfsdp.OK, (st, detail)
    zeros = np.zeros(numel, np.float32)
    for s in shards:
        check_matrix(s, upd.cpu().numpy(), mom.cpu().numpy(), grad_np, zeros, ns_steps=w.ns_steps)
