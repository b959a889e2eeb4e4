"""Full-size parity: the large owner sets run on the GPU exactly as bench.py runs
them (one call of the owner step over the whole owner set, bf16 update).

  * Against the fp64 oracle: from every launch of the set (128 matrices per
    launch, in shard order) the first matrix of every shape and up to two
    all-zero matrices.  Each sampled update is checked as a whole (relative
    Frobenius error) and block by block: every 128 x 128 block within the
    block bounds, so that one wrong tile cannot hide in a whole-matrix norm.
  * Against itself run alone: every matrix of the set is run again as a
    one-matrix owner set at the same offsets, and the whole update and
    momentum buffers must match the owner-set run bit for bit (MatrixFSDP --
    Abstract: the update matches full-matrix Muon).  A batch-offset or
    scheduling mistake in the second or third launch of the MoE set changes
    bits even where it stays within the oracle's tolerance.

The AdamW tail is checked element by element at its full size.  These need
minutes of oracle time on the host cores; they are marked slow as well as gpu.
"""
import numpy as np
import pytest

from oracle import adamw_ref, bf16_bits_to_f64, muon_matrix_ref
from matrix_optimizers_under_gb300 import workloads as W
from tests import helpers as H

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.slow]

A, B, C = W.NS_COEFFS
LAUNCH = 128   # matrices per Newton-Schulz launch (the library's batch)


def _sample(shards, w):
    """Per launch (runs of LAUNCH shards in the order given): the first matrix
    of every (rows, cols) and up to two all-zero matrices."""
    out = []
    for base in range(0, len(shards), LAUNCH):
        seen = set()
        batch = shards[base:base + LAUNCH]
        for s in batch:
            if s.param_id not in w.zero_params and (s.rows, s.cols) not in seen:
                seen.add((s.rows, s.cols))
                out.append(s)
        out += [s for s in batch if s.param_id in w.zero_params][:2]
    return out


def _standalone_matches(mfsdp, shards, grad, mom, upd, kw):
    """Every shard run alone, at its own offset of the same buffers: the whole
    update and momentum buffers equal the owner-set run's bit for bit."""
    dev = grad.device
    mom1 = torch.zeros_like(mom)
    upd1 = torch.zeros_like(upd)
    ws1 = torch.empty(max(mfsdp.muon_workspace_bytes([s]) for s in shards), dtype=torch.uint8, device=dev)
    for s in shards:
        mfsdp.muon_owner_step([s], grad, mom1, upd1, ws1, **kw)
    st, detail = mfsdp.muon_device_status(ws1)
    assert st == mfsdp.OK, (st, detail)
    torch.cuda.synchronize()
    assert torch.equal(upd1.view(torch.int16), upd.view(torch.int16)), "update differs from the standalone runs"
    assert torch.equal(mom1.view(torch.int32), mom.view(torch.int32)), "momentum differs from the standalone runs"


@pytest.mark.parametrize("name", ["llama_1p3b_rank", "llama3_8b_rank", "moe_skewed"])
def test_full_owner_set(mfsdp, name):
    w = W.get(name)
    plan = mfsdp.plan_owners(w.param_table(), w.world, w.ns_steps, w.align_elems)
    r = H.heaviest_rank(plan)
    shards = plan.rank_matrices(r)
    numel = plan.rank_matrix_elems[r]
    grad_np = W.owner_grad_buffer(w, shards, numel)
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda:0")
    grad = torch.from_numpy(grad_np.view(np.int16)).to(dev).view(torch.bfloat16)
    mom = torch.zeros(numel, dtype=torch.float32, device=dev)
    upd = torch.zeros(numel, dtype=torch.bfloat16, device=dev)
    ws = torch.empty(mfsdp.muon_workspace_bytes(shards), dtype=torch.uint8, device=dev)
    kw = dict(beta=w.beta, ns_steps=w.ns_steps, coeffs=w.ns_coeffs, eps=w.ns_eps)
    mfsdp.muon_owner_step(shards, grad, mom, upd, ws, **kw)
    st, detail = mfsdp.muon_device_status(ws)
    assert st == mfsdp.OK, (st, detail)
    torch.cuda.synchronize()
    del ws
    _standalone_matches(mfsdp, shards, grad, mom, upd, kw)

    errs = {}
    sample = _sample(shards, w)
    if len(shards) > LAUNCH:   # the sample reaches every launch
        index = {s.param_id: i for i, s in enumerate(shards)}
        launches = {index[s.param_id] // LAUNCH for s in sample if s.param_id not in w.zero_params}
        assert launches == set(range(-(-len(shards) // LAUNCH))), launches
    for s in sample:
        n = s.rows * s.cols
        seg = slice(s.offset, s.offset + n)
        O = upd[seg].float().cpu().numpy().astype(np.float64).reshape(s.rows, s.cols)
        M = mom[seg].cpu().numpy().reshape(s.rows, s.cols)
        G = bf16_bits_to_f64(grad_np[seg]).reshape(s.rows, s.cols)
        M_ref, O_ref = muon_matrix_ref(G, np.zeros_like(G), w.beta, False, w.ns_steps, A, B, C, w.ns_eps)
        assert np.array_equal(M, M_ref.astype(np.float32)), "step-1 momentum must equal G exactly"
        if s.param_id in w.zero_params:
            assert np.all(O == 0.0)
            continue
        errs[s.param_id] = H.rel_fro(O, O_ref)
        assert errs[s.param_id] <= H.ns_tol(s.rows, s.cols), (s.param_id, errs)
        H.check_blocks(O, O_ref, f"param {s.param_id} {s.rows}x{s.cols}")
    print(name, {k: round(v, 5) for k, v in errs.items()})


def test_full_size_adamw_tail(mfsdp):
    """The 50M-element packed tail of the MoE owner set, element by element."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    w = W.get("moe_skewed")
    tid = [i for i, p in enumerate(w.params) if p.kind == W.KIND_TAIL][0]
    p0 = W.tail_param_f32(w, tid)
    g = W.grad_f32(w, tid)
    dev = torch.device("cuda:0")
    tp, tg = torch.from_numpy(p0.copy()).to(dev), torch.from_numpy(g).to(dev)
    tm, tv = torch.zeros_like(tp), torch.zeros_like(tp)
    mfsdp.adamw_tail_step(tp, tg, tm, tv, lr=w.lr, beta1=w.betas[0], beta2=w.betas[1], eps=w.adam_eps,
                          wd=w.weight_decay, step=1)
    rp, rm, rv = adamw_ref(p0, g, np.zeros_like(p0), np.zeros_like(p0), w.lr, w.betas[0], w.betas[1], w.adam_eps,
                           w.weight_decay, 1)
    assert H.adam_err(tp.cpu().numpy(), rp) <= H.ADAM_REL
    assert H.adam_err(tm.cpu().numpy(), rm) <= H.ADAM_REL
    assert H.adam_err(tv.cpu().numpy(), rv) <= H.ADAM_REL


def test_full_owner_set_second_step_fp32_update(mfsdp):
    """The 1.3B rank at full size for two steps with different gradients and an
    fp32 update: the second step starts from momentum G1, so M = beta G1 + G2
    and the Newton-Schulz input is that sum (MatrixFSDP -- Abstract:
    momentum-smoothed updates), and the last epilogue writes fp32 in the stored
    orientation.  One matrix of every shape is checked against the fp64 oracle."""
    w = W.get("llama_1p3b_rank")
    plan = mfsdp.plan_owners(w.param_table(), w.world, w.ns_steps, w.align_elems)
    r = H.heaviest_rank(plan)
    shards = plan.rank_matrices(r)
    numel = plan.rank_matrix_elems[r]
    g1_np = W.owner_grad_buffer(w, shards, numel)
    rng = np.random.default_rng([w.seed, 2])
    g2_np = W.f32_to_bf16_bits((rng.standard_normal(numel) * w.grad_scale).astype(np.float32))
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda:0")
    kw = dict(beta=w.beta, ns_steps=w.ns_steps, coeffs=w.ns_coeffs, eps=w.ns_eps)
    mom = torch.zeros(numel, dtype=torch.float32, device=dev)
    upd = torch.full((numel,), float("nan"), dtype=torch.float32, device=dev)
    ws = torch.empty(mfsdp.muon_workspace_bytes(shards), dtype=torch.uint8, device=dev)
    for g_np in (g1_np, g2_np):
        grad = torch.from_numpy(g_np.view(np.int16)).to(dev).view(torch.bfloat16)
        mfsdp.muon_owner_step(shards, grad, mom, upd, ws, **kw)
        st, detail = mfsdp.muon_device_status(ws)
        assert st == mfsdp.OK, (st, detail)
    torch.cuda.synchronize()
    del ws
    errs = {}
    for s in _sample(shards, w):
        seg = slice(s.offset, s.offset + s.rows * s.cols)
        G1 = bf16_bits_to_f64(g1_np[seg]).reshape(s.rows, s.cols)
        G2 = bf16_bits_to_f64(g2_np[seg]).reshape(s.rows, s.cols)
        M_ref, O_ref = muon_matrix_ref(G2, G1, w.beta, False, w.ns_steps, A, B, C, w.ns_eps)
        M = mom[seg].cpu().numpy().astype(np.float64).reshape(s.rows, s.cols)
        bound = H.MOM_REL * (np.abs(w.beta * G1) + np.abs(G2)) + 1e-30
        assert np.all(np.abs(M - M_ref) <= bound), s.param_id
        O = upd[seg].cpu().numpy().astype(np.float64).reshape(s.rows, s.cols)
        assert np.all(np.isfinite(O)), s.param_id
        errs[(s.rows, s.cols)] = H.rel_fro(O, O_ref)
        assert errs[(s.rows, s.cols)] <= H.ns_tol(s.rows, s.cols), (s.param_id, errs)
        H.check_blocks(O, O_ref, f"param {s.param_id} {s.rows}x{s.cols}")
    print({k: round(v, 5) for k, v in errs.items()})


def test_full_owner_set_apply(mfsdp):
    """The fused weight update at full size (1.3B rank, fp32 weights, the Muon
    shape scale): every element of the sampled matrices is W (1 - lr wd) -
    lr scale O for the update O the same call wrote (one fp32 rounding), and
    the weight change matches the fp64 oracle's within the Newton-Schulz
    tolerance."""
    from oracle import muon_apply_ref, muon_scale_ref
    w = W.get("llama_1p3b_rank")
    plan = mfsdp.plan_owners(w.param_table(), w.world, w.ns_steps, w.align_elems)
    r = H.heaviest_rank(plan)
    shards = plan.rank_matrices(r)
    numel = plan.rank_matrix_elems[r]
    grad_np = W.owner_grad_buffer(w, shards, numel)
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda:0")
    lr, wd, mode = 0.02, 0.1, mfsdp.SCALE_MUON
    W0 = (np.random.default_rng([w.seed, 3]).standard_normal(numel) * 0.02).astype(np.float32)
    Wt = torch.from_numpy(W0).to(dev)
    grad = torch.from_numpy(grad_np.view(np.int16)).to(dev).view(torch.bfloat16)
    mom = torch.zeros(numel, dtype=torch.float32, device=dev)
    upd = torch.full((numel,), float("nan"), dtype=torch.float32, device=dev)
    ws = torch.empty(mfsdp.muon_workspace_bytes(shards), dtype=torch.uint8, device=dev)
    mfsdp.muon_owner_step_apply(shards, grad, mom, upd, Wt, ws, lr=lr, weight_decay=wd, scale_mode=mode,
                                beta=w.beta, ns_steps=w.ns_steps, coeffs=w.ns_coeffs, eps=w.ns_eps)
    st, detail = mfsdp.muon_device_status(ws)
    assert st == mfsdp.OK, (st, detail)
    torch.cuda.synchronize()
    del ws
    decay = np.float64(np.float32(1.0 - lr * wd))
    errs = {}
    for s in _sample(shards, w):
        seg = slice(s.offset, s.offset + s.rows * s.cols)
        O = upd[seg].cpu().numpy().astype(np.float64)
        Wn = Wt[seg].cpu().numpy().astype(np.float64)
        W0s = W0[seg].astype(np.float64)
        scale = muon_scale_ref(s.rows, s.cols, mode)
        expect = W0s * decay - lr * scale * O
        tol = 2.0 ** -23 * 4 * (np.abs(W0s) + lr * scale * np.abs(O))
        assert np.all(np.abs(Wn - expect) <= tol + 1e-30), s.param_id
        G = bf16_bits_to_f64(grad_np[seg]).reshape(s.rows, s.cols)
        _, O_ref = muon_matrix_ref(G, np.zeros_like(G), w.beta, False, w.ns_steps, A, B, C, w.ns_eps)
        W_ref = muon_apply_ref(W0s.reshape(s.rows, s.cols), O_ref, lr, wd, scale)
        base = W0s.reshape(s.rows, s.cols) * decay
        errs[(s.rows, s.cols)] = H.rel_fro(Wn.reshape(s.rows, s.cols) - base, W_ref - base)
        assert errs[(s.rows, s.cols)] <= H.ns_tol(s.rows, s.cols), (s.param_id, errs)
    print({k: round(v, 5) for k, v in errs.items()})
