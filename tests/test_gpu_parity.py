"""GPU parity of the owner-local optimizer step against the fp64 oracle.

Every case calls the CUDA library through its C ABI (via the thin binding) on
seeded inputs and compares element by element with the oracle:
  * momentum buffer: fp32 within one rounding of beta*M + G;
  * Newton-Schulz update: relative Frobenius error <= 2e-2 per matrix, exact
    zero for all-zero matrices;
  * AdamW: max relative error <= 1e-5 (floor 1e-2 * max |reference|);
  * padding between segments (filled with NaN canaries) is never read or written.
Equivalence (MatrixFSDP -- Abstract: the update matches full-matrix Muon):
an owner set's update equals, bit for bit, the update of each matrix run alone
from its own buffer.
"""
import numpy as np
import pytest

from oracle import adamw_ref, muon_matrix_ref, bf16_bits_to_f64, newton_schulz_ref
from matrix_optimizers_under_gb300 import workloads as W
from tests import helpers as H

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

A, B, C = W.NS_COEFFS


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def to_dev_grad(buf: np.ndarray):
    if buf.dtype == np.uint16:
        return torch.from_numpy(buf.view(np.int16)).to(_dev()).view(torch.bfloat16)
    return torch.from_numpy(buf).to(_dev())


def from_dev(t) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return H.bf16_bits_to_f32(t.view(torch.int16).cpu().numpy().view(np.uint16))
    return t.cpu().numpy()


def run_step(mfsdp, shards, grad_np, mom_np, *, update_dtype, ns_steps=5, beta=0.95, nesterov=False,
             coeffs=W.NS_COEFFS, eps=W.NS_EPS, ws_extra=0):
    dev = _dev()
    grad = to_dev_grad(grad_np)
    mom = torch.from_numpy(mom_np.copy()).to(dev)
    numel = grad_np.size
    upd = torch.full((numel,), float("nan"), dtype=update_dtype, device=dev)
    ws = torch.empty(mfsdp.muon_workspace_bytes(shards) + ws_extra, dtype=torch.uint8, device=dev)
    mfsdp.muon_owner_step(shards, grad, mom, upd, ws, beta=beta, nesterov=nesterov, ns_steps=ns_steps,
                          coeffs=coeffs, eps=eps)
    st, detail = mfsdp.muon_device_status(ws)
    assert st == mfsdp.OK, (st, detail)
    torch.cuda.synchronize()
    return from_dev(upd), mom.cpu().numpy(), ws


def grad_f64(buf, s):
    seg = buf[s.offset:s.offset + s.rows * s.cols]
    return (bf16_bits_to_f64(seg) if seg.dtype == np.uint16 else seg.astype(np.float64)).reshape(s.rows, s.cols)


def check_matrix(s, upd, mom, grad_np, mom0, *, ns_steps, beta=0.95, nesterov=False, zero=False):
    G = grad_f64(grad_np, s)
    M0 = mom0[s.offset:s.offset + s.rows * s.cols].astype(np.float64).reshape(s.rows, s.cols)
    M_ref, O_ref = muon_matrix_ref(G, M0, beta, nesterov, ns_steps, A, B, C, W.NS_EPS)
    O = upd[s.offset:s.offset + s.rows * s.cols].reshape(s.rows, s.cols)
    M = mom[s.offset:s.offset + s.rows * s.cols].reshape(s.rows, s.cols)
    bound = H.MOM_REL * (np.abs(beta * M0) + np.abs(G)) + 1e-30
    assert np.all(np.abs(M - M_ref) <= bound), f"momentum mismatch param {s.param_id}"
    if zero:
        assert np.all(O == 0.0), f"zero matrix {s.param_id} not exactly zero"
        return 0.0
    err = H.rel_fro(O, O_ref)
    assert np.all(np.isfinite(O)), f"non-finite update param {s.param_id}"
    assert err <= H.ns_tol(s.rows, s.cols), f"param {s.param_id} {s.rows}x{s.cols}: rel Frobenius error {err:.3e}"
    return err


def check_padding(upd, mom, shards, numel):
    used = np.zeros(numel, bool)
    for s in shards:
        used[s.offset:s.offset + s.rows * s.cols] = True
    assert np.all(np.isnan(upd[~used])), "update written outside the segments"
    assert np.all(mom[~used] == 0.0), "momentum written outside the segments"


def owner_set(mfsdp, w, rank=None):
    plan = mfsdp.plan_owners(w.param_table(), w.world, w.ns_steps, w.align_elems)
    r = H.heaviest_rank(plan) if rank is None else rank
    return plan, r, plan.rank_matrices(r), plan.rank_matrix_elems[r]


# ------------------------------------------------------------------ AdamW
@pytest.mark.parametrize("n", [1, 3, 13, 4096, 4097, 9984, 1 << 20])
def test_adamw_parity(mfsdp, n):
    dev = _dev()
    w = W.get("tiny")
    rng = np.random.default_rng(n)
    p = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    tp, tm, tv = (torch.from_numpy(x.copy()).to(dev) for x in (p, m, v))
    rp, rm, rv = p.astype(np.float64), m.astype(np.float64), v.astype(np.float64)
    for t in (1, 2, 3):
        g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
        tg = torch.from_numpy(g).to(dev)
        mfsdp.adamw_tail_step(tp, tg, tm, tv, lr=w.lr, beta1=w.betas[0], beta2=w.betas[1], eps=w.adam_eps,
                              wd=w.weight_decay, step=t)
        # the oracle continues from the GPU's fp32 state, as the next step would
        rp, rm, rv = adamw_ref(rp, g, rm, rv, w.lr, w.betas[0], w.betas[1], w.adam_eps, w.weight_decay, t)
        gp, gm, gv = (x.cpu().numpy() for x in (tp, tm, tv))
        assert H.adam_err(gp, rp) <= H.ADAM_REL
        assert H.adam_err(gm, rm) <= H.ADAM_REL
        assert H.adam_err(gv, rv) <= H.ADAM_REL
        rp, rm, rv = gp.astype(np.float64), gm.astype(np.float64), gv.astype(np.float64)


def test_adamw_tiny_workload_first_step_closed_form(mfsdp):
    dev = _dev()
    w = W.get("tiny")
    tid = [i for i, p in enumerate(w.params) if p.kind == W.KIND_TAIL][0]
    p0 = W.tail_param_f32(w, tid)
    g = W.grad_f32(w, tid)
    tp, tg = torch.from_numpy(p0.copy()).to(dev), torch.from_numpy(g).to(dev)
    tm, tv = torch.zeros_like(tp), torch.zeros_like(tp)
    mfsdp.adamw_tail_step(tp, tg, tm, tv, lr=w.lr, beta1=0.9, beta2=0.95, eps=1e-8, wd=0.1, step=1)
    g64 = g.astype(np.float64)
    closed = p0.astype(np.float64) * (1 - 1e-3 * 0.1) - 1e-3 * g64 / (np.abs(g64) + 1e-8)
    assert H.adam_err(tp.cpu().numpy(), closed) <= H.ADAM_REL
    assert H.adam_err(tm.cpu().numpy(), 0.1 * g64) <= H.ADAM_REL
    assert H.adam_err(tv.cpu().numpy(), 0.05 * g64 * g64) <= H.ADAM_REL


# ------------------------------------------------------- momentum + NS
@pytest.mark.parametrize("ns_steps", [0, 1, 2, 5])
@pytest.mark.parametrize("upd_dtype", ["f32", "bf16"])
def test_tiny_workload(mfsdp, ns_steps, upd_dtype):
    w = W.get("tiny")
    plan, r, shards, numel = owner_set(mfsdp, w)
    grad = H.build_grad_buffer(w, shards, numel)
    mom0 = np.zeros(numel, np.float32)
    dt = torch.float32 if upd_dtype == "f32" else torch.bfloat16
    upd, mom, _ = run_step(mfsdp, shards, grad, mom0, update_dtype=dt, ns_steps=ns_steps)
    for s in shards:
        check_matrix(s, upd, mom, grad, mom0, ns_steps=ns_steps)


@pytest.mark.parametrize("ns_steps", [1, 2])
def test_each_product_from_workspace(mfsdp, ns_steps):
    """Isolates every kernel: the workspace keeps X0 = bf16(U) and the last
    products, so each is checked against fp64 arithmetic on the bf16 inputs it
    actually read.  ns_steps=1 covers the first-iteration prescale paths,
    ns_steps=2 the plain ones.  The GPT-2 block has both forms of the
    iteration: 768 x 768 runs the direct one (A, B and, for two steps, X1
    kept), the three long matrices the Gram-space one (A, P, C and Q kept).
    Symmetric products are read back as stored: their blocks on or above the
    diagonal of 256 x 256 blocks, the others their mirror images' transposes,
    and each product of two of them is the true product of those matrices."""
    w = W.get("gpt2_block")
    plan, r, shards, numel = owner_set(mfsdp, w)
    grad = H.build_grad_buffer(w, shards, numel)
    mom0 = np.zeros(numel, np.float32)
    upd, mom, ws = run_step(mfsdp, shards, grad, mom0, update_dtype=torch.float32, ns_steps=ns_steps)
    wsb = ws.cpu().numpy()
    programs = mfsdp.muon_gram_space_layout(shards, ns_steps)
    assert sorted(g[0] for g in programs) == [0, 1, 1, 1]
    for s, (x0, x1, a_off, b_off, sp, lp, sd, ld), (gram, c_off, q0_off, q1_off) in zip(
            shards, mfsdp.muon_workspace_layout(shards), programs):
        G = grad_f64(grad, s)
        X = G.T if s.rows > s.cols else G
        Yw = H.unblock(wsb, x0, sp, lp).astype(np.float64)
        assert np.array_equal(Yw[:sd, :ld], X), "X0 is not bf16(U) (G is bf16 and M = G)"
        assert np.all(Yw[sd:, :] == 0) and np.all(Yw[:, ld:] == 0), "X0 padding not zero"

        def sym(off):
            return H.symmetric_from_upper(H.unblock(wsb, off, sp, sp)).astype(np.float64)[:sd, :sd]
        O = upd[s.offset:s.offset + s.rows * s.cols].reshape(s.rows, s.cols).astype(np.float64)
        O = O.T if s.rows > s.cols else O
        inv = 1.0 / (np.sqrt(np.sum(X * X)) + W.NS_EPS)
        I = np.eye(sd)
        if not gram:
            Aw, Bw = sym(a_off), sym(b_off)
            if ns_steps == 1:
                Xin, scale_a, scale_x = X, inv * inv, inv
            else:
                Xin = H.unblock(wsb, x1, sp, lp).astype(np.float64)[:sd, :ld]
                scale_a = scale_x = 1.0
            assert H.rel_fro(Aw, scale_a * (Xin @ Xin.T)) < 1e-2, "Gram product"
            assert H.rel_fro(Bw, B * Aw + C * (Aw @ Aw)) < 1e-2, "polynomial product"
            assert H.rel_fro(O, scale_x * (A * Xin + Bw @ Xin)) < 1e-2, "update product"
            continue
        # Gram space: P_0 = Q_0 in Q_even, P_k (k >= 1) in B; A holds A_{T-1}
        A0 = inv * inv * (X @ X.T)
        Aw = sym(a_off)
        if ns_steps == 1:
            assert H.rel_fro(Aw, A0) < 1e-2, "Gram product A_0"
            P0 = sym(q0_off)
            assert H.rel_fro(P0, A * I + B * Aw + C * (Aw @ Aw)) < 1e-2, "polynomial P_0"
            assert H.rel_fro(O, inv * (P0 @ X)) < 1e-2, "final product Q_0 X0"
        else:
            P0, C0, P1, Q1 = sym(q0_off), sym(c_off), sym(b_off), sym(q1_off)
            assert H.rel_fro(C0, P0 @ A0) < 1e-2, "product C_0 = P_0 A_0"
            assert H.rel_fro(Aw, C0 @ P0) < 1e-2, "product A_1 = C_0 P_0"
            assert H.rel_fro(P1, A * I + B * Aw + C * (Aw @ Aw)) < 1e-2, "polynomial P_1"
            assert H.rel_fro(Q1, P1 @ P0) < 1e-2, "product Q_1 = P_1 Q_0"
            assert H.rel_fro(O, inv * (Q1 @ X)) < 1e-2, "final product Q_1 X0"


@pytest.mark.parametrize("upd_dtype", ["f32", "bf16"])
def test_gpt2_block_workload(mfsdp, upd_dtype):
    w = W.get("gpt2_block")
    plan, r, shards, numel = owner_set(mfsdp, w)
    grad = H.build_grad_buffer(w, shards, numel)
    mom0 = np.zeros(numel, np.float32)
    dt = torch.float32 if upd_dtype == "f32" else torch.bfloat16
    upd, mom, _ = run_step(mfsdp, shards, grad, mom0, update_dtype=dt)
    for s in shards:
        check_matrix(s, upd, mom, grad, mom0, ns_steps=5)
    check_padding(upd, mom, shards, numel)


RAGGED = [(1, 1), (1, 9), (9, 1), (7, 300), (300, 7), (130, 257), (257, 130), (129, 129), (200, 640), (513, 96)]


@pytest.mark.parametrize("gdt", ["f32", "bf16"])
def test_ragged_shapes_odd_offsets(mfsdp, gdt):
    """Shapes that are not multiples of any tile, at offsets that are not
    multiples of 8 (scalar paths), plus a zero matrix."""
    rng = np.random.default_rng(123)
    shards, off = [], 0
    for i, (r, c) in enumerate(RAGGED):
        off += int(rng.integers(1, 40))
        shards.append(mfsdp.make_shard(off, r, c, param_id=i))
        off += r * c
    numel = off + 5
    vals = (rng.standard_normal(numel) * 1e-3).astype(np.float32)
    zero = shards[3]
    vals[zero.offset:zero.offset + zero.rows * zero.cols] = 0
    grad = vals if gdt == "f32" else W.f32_to_bf16_bits(vals)
    mom0 = (rng.standard_normal(numel) * 1e-3).astype(np.float32)   # a second step: M != 0
    mom0[zero.offset:zero.offset + zero.rows * zero.cols] = 0
    upd, mom, _ = run_step(mfsdp, shards, grad, mom0, update_dtype=torch.float32)
    for s in shards:
        check_matrix(s, upd, mom, grad, mom0, ns_steps=5, zero=(s is zero))


# tall shapes with ragged sides: four in the Gram-space form (long side at
# least twice the short one), two in the standard form
TALL = [(1000, 200), (700, 136), (1544, 392), (1000, 130), (1500, 1000), (1000, 520)]


@pytest.mark.parametrize("udt", [torch.float32, torch.bfloat16])
def test_tall_final_store_paths(mfsdp, udt):
    """Tall matrices write their update through the epilogue's stage,
    transposed, when the stored rows start 16-byte aligned (offset and s
    multiples of 8), and element by element otherwise (s = 130, or an offset
    that is not a multiple of 8), in both forms of the iteration.  Both paths
    store the same values: the aligned set matches the oracle, and each matrix
    run again at an odd offset gives the same bits."""
    rng = np.random.default_rng(77)
    shards, off = [], 0
    for i, (r, c) in enumerate(TALL):
        shards.append(mfsdp.make_shard(off, r, c, param_id=i))
        off += -(-(r * c) // 128) * 128
    assert [g[0] for g in mfsdp.muon_gram_space_layout(shards, 5)] == [1, 1, 1, 1, 0, 0]
    numel = off
    vals = (rng.standard_normal(numel) * 1e-3).astype(np.float32)
    grad = W.f32_to_bf16_bits(vals)
    mom0 = np.zeros(numel, np.float32)
    upd, mom, _ = run_step(mfsdp, shards, grad, mom0, update_dtype=udt)
    for s in shards:
        check_matrix(s, upd, mom, grad, mom0, ns_steps=5)
    for s in shards:
        n = s.rows * s.cols
        shifted = [mfsdp.make_shard(3, s.rows, s.cols, param_id=s.param_id)]
        g1 = np.zeros(n + 3, grad.dtype)
        g1[3:] = grad[s.offset:s.offset + n]
        u1, _, _ = run_step(mfsdp, shifted, g1, np.zeros(n + 3, np.float32), update_dtype=udt)
        a, b = upd[s.offset:s.offset + n], u1[3:]
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), f"{s.rows}x{s.cols}: store paths differ"


@pytest.mark.parametrize("ns_steps", [3, 4, 6])
def test_gram_space_step_counts(mfsdp, ns_steps):
    """Wide and tall shapes of the Gram-space form (ragged sides, aligned and
    odd offsets) at the step counts the other tests do not run: 3 and 4 (the
    form's null tiles -- no Q in the first iteration, no C in the last -- and
    the Q ping-pong's parity) and 6 (past its bound: every matrix takes the
    standard form).  A second step from non-zero momentum, fp32 gradients,
    Nesterov, fp32 update, against the oracle."""
    shapes = [(200, 640), (640, 200), (384, 1032), (1032, 384), (256, 896)]
    rng = np.random.default_rng(ns_steps)
    shards, off = [], 0
    for i, (r, c) in enumerate(shapes):
        off += 128 if i % 2 == 0 else 131
        shards.append(mfsdp.make_shard(off, r, c, param_id=i))
        off += r * c
    want = [1 if ns_steps <= 5 else 0] * len(shapes)
    assert [g[0] for g in mfsdp.muon_gram_space_layout(shards, ns_steps)] == want
    numel = off + 7
    grad = (rng.standard_normal(numel) * 1e-3).astype(np.float32)
    mom0 = (rng.standard_normal(numel) * 1e-3).astype(np.float32)
    upd, mom, _ = run_step(mfsdp, shards, grad, mom0, update_dtype=torch.float32, ns_steps=ns_steps, nesterov=True)
    for s in shards:
        check_matrix(s, upd, mom, grad, mom0, ns_steps=ns_steps, nesterov=True)


def test_nesterov_and_second_step(mfsdp):
    w = W.get("gpt2_block")
    plan, r, shards, numel = owner_set(mfsdp, w)
    grad = H.build_grad_buffer(w, shards, numel)
    rng = np.random.default_rng(5)
    mom0 = np.zeros(numel, np.float32)
    for s in shards:
        mom0[s.offset:s.offset + s.rows * s.cols] = rng.standard_normal(s.rows * s.cols) * 1e-3
    upd, mom, _ = run_step(mfsdp, shards, grad, mom0, update_dtype=torch.float32, nesterov=True)
    for s in shards:
        check_matrix(s, upd, mom, grad, mom0, ns_steps=5, nesterov=True)


def test_equivalence_owner_set_vs_standalone(mfsdp):
    """The owner-set update equals each matrix's standalone update, bitwise."""
    w = W.get("gpt2_block")
    plan, r, shards, numel = owner_set(mfsdp, w)
    grad = H.build_grad_buffer(w, shards, numel)
    mom0 = np.zeros(numel, np.float32)
    upd, mom, _ = run_step(mfsdp, shards, grad, mom0, update_dtype=torch.bfloat16)
    for s in shards:
        n = s.rows * s.cols
        alone = [mfsdp.make_shard(0, s.rows, s.cols, param_id=s.param_id)]
        u1, m1, _ = run_step(mfsdp, alone, grad[s.offset:s.offset + n].copy(), np.zeros(n, np.float32),
                             update_dtype=torch.bfloat16)
        assert np.array_equal(u1.view(np.uint32), upd[s.offset:s.offset + n].view(np.uint32))
        assert np.array_equal(m1, mom[s.offset:s.offset + n])


def test_phase_split_matches_full_step(mfsdp):
    """Momentum phase then Newton-Schulz phase == one full step, bitwise."""
    dev = _dev()
    w = W.get("gpt2_block")
    plan, r, shards, numel = owner_set(mfsdp, w)
    grad = H.build_grad_buffer(w, shards, numel)
    mom0 = np.zeros(numel, np.float32)
    u1, m1, _ = run_step(mfsdp, shards, grad, mom0, update_dtype=torch.bfloat16)
    g = to_dev_grad(grad)
    mom = torch.zeros(numel, dtype=torch.float32, device=dev)
    upd = torch.full((numel,), float("nan"), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(mfsdp.muon_workspace_bytes(shards), dtype=torch.uint8, device=dev)
    mfsdp.muon_owner_step(shards, g, mom, upd, ws, phases=mfsdp.PHASE_MOMENTUM)
    mfsdp.muon_owner_step(shards, g, mom, upd, ws, phases=mfsdp.PHASE_NEWTON_SCHULZ)
    torch.cuda.synchronize()
    assert np.array_equal(from_dev(upd).view(np.uint32), u1.view(np.uint32))
    assert np.array_equal(mom.cpu().numpy(), m1)


@pytest.mark.parametrize("name,n_groups", [("llama_1p3b_rank", 5), ("llama3_8b_rank", 10)])
def test_host_buffer_library_groups_match_resident_step(mfsdp, name, n_groups):
    """The library's own group choice on sets large enough to leave offset
    order -- the 1.3B rank's small -> large -> small ramp (5 groups) and the 8B
    rank's balanced groups between a head and a tail (10 groups): update and
    momentum bit-identical to the resident step, and the staging buffer holds
    exactly the copied gradient."""
    dev = _dev()
    w = W.get(name)
    plan, r, shards, numel = owner_set(mfsdp, w)
    ng, gof = mfsdp.host_step_groups(shards)
    assert ng == n_groups and sorted(set(gof)) == list(range(ng))
    order = sorted(range(len(shards)), key=lambda i: shards[i].offset)
    assert any(gof[order[k]] > gof[order[k + 1]] for k in range(len(order) - 1))   # not offset order
    gen = torch.Generator(device=dev)
    gen.manual_seed(13)
    g_dev = (torch.randn(numel, device=dev, generator=gen) * 1e-3).to(torch.bfloat16)
    m0 = torch.randn(numel, device=dev, generator=gen) * 1e-3
    ws = torch.empty(mfsdp.muon_workspace_bytes(shards), dtype=torch.uint8, device=dev)
    mom_ref, upd_ref = m0.clone(), torch.empty(numel, dtype=torch.bfloat16, device=dev)
    mfsdp.muon_owner_step(shards, g_dev, mom_ref, upd_ref, ws)
    gh = g_dev.cpu().pin_memory()
    uh = torch.full((numel,), float("nan"), dtype=torch.bfloat16).pin_memory()
    gd = torch.zeros(numel, dtype=torch.bfloat16, device=dev)
    ud = torch.empty(numel, dtype=torch.bfloat16, device=dev)
    mom = m0.clone()
    mfsdp.muon_owner_step_host(shards, gh, gd, mom, ud, uh, ws, groups=0)
    torch.cuda.synchronize()
    assert mfsdp.muon_device_status(ws)[0] == mfsdp.OK
    assert torch.equal(mom, mom_ref)
    ref = upd_ref.cpu()
    for s in shards:
        seg = slice(s.offset, s.offset + s.rows * s.cols)
        assert torch.equal(uh[seg].view(torch.int16), ref[seg].view(torch.int16)), s.param_id
        assert torch.equal(gd[seg], g_dev[seg]), s.param_id


@pytest.mark.parametrize("groups", [1, 3])
@pytest.mark.parametrize("gdt,udt", [("f32", "f32"), ("f32", "bf16"), ("bf16", "f32"), ("bf16", "bf16")])
def test_host_buffer_dtypes_ragged(mfsdp, gdt, udt, groups):
    """Every gradient / update dtype pair through the host-buffer step, on a
    ragged owner set (dimensions that fill no tile; 128-element aligned
    offsets with gaps): the copies move grad- and update-sized ranges, so the
    result must be bit-identical to the resident step with the same inputs."""
    dev = _dev()
    params = [p for p in W.ragged_params(41, 24) if p[2] == W.KIND_MATRIX][:9]
    plan = mfsdp.plan_owners(params, 1, 5, 128)
    shards = plan.rank_matrices(0)
    numel = plan.rank_matrix_elems[0]
    tg = torch.float32 if gdt == "f32" else torch.bfloat16
    tu = torch.float32 if udt == "f32" else torch.bfloat16
    rng = np.random.default_rng(4242)
    g_cpu = torch.from_numpy((rng.standard_normal(numel) * 1e-2).astype(np.float32)).to(tg)
    m_cpu = torch.from_numpy((rng.standard_normal(numel) * 1e-3).astype(np.float32))
    ws = torch.empty(mfsdp.muon_workspace_bytes(shards), dtype=torch.uint8, device=dev)
    g_dev, mom_ref = g_cpu.to(dev), m_cpu.to(dev)
    upd_ref = torch.full((numel,), float("nan"), dtype=tu, device=dev)
    mfsdp.muon_owner_step(shards, g_dev, mom_ref, upd_ref, ws)
    gh = g_cpu.pin_memory()
    uh = torch.full((numel,), float("nan"), dtype=tu).pin_memory()
    gd = torch.zeros(numel, dtype=tg, device=dev)
    ud = torch.full((numel,), float("nan"), dtype=tu, device=dev)
    mom = m_cpu.to(dev)
    mfsdp.muon_owner_step_host(shards, gh, gd, mom, ud, uh, ws, groups=groups)
    torch.cuda.synchronize()
    assert mfsdp.muon_device_status(ws)[0] == mfsdp.OK
    assert mfsdp.host_step_groups(shards, tg, tu, groups)[0] == min(groups, len(shards))
    assert torch.equal(mom, mom_ref)
    ref = upd_ref.cpu()
    view = torch.int32 if tu == torch.float32 else torch.int16
    for s in shards:
        seg = slice(s.offset, s.offset + s.rows * s.cols)
        assert torch.equal(uh[seg].view(view), ref[seg].view(view)), (s.param_id, s.rows, s.cols)


@pytest.mark.parametrize("groups", [0, 1, 2, 3, 8])
def test_host_buffer_pipeline_matches_resident_step(mfsdp, groups):
    """Gradient from pinned host memory, update back to it, copies overlapped with
    compute group by group: bit-identical to the resident step."""
    dev = _dev()
    w = W.get("gpt2_block")
    plan, r, shards, numel = owner_set(mfsdp, w)
    grad = H.build_grad_buffer(w, shards, numel)
    mom0 = np.zeros(numel, np.float32)
    u_ref, m_ref, _ = run_step(mfsdp, shards, grad, mom0, update_dtype=torch.bfloat16)
    gh = torch.from_numpy(grad.view(np.int16)).view(torch.bfloat16).pin_memory()
    uh = torch.full((numel,), float("nan"), dtype=torch.bfloat16).pin_memory()
    gd = torch.empty(numel, dtype=torch.bfloat16, device=dev)
    ud = torch.full((numel,), float("nan"), dtype=torch.bfloat16, device=dev)
    mom = torch.zeros(numel, dtype=torch.float32, device=dev)
    ws = torch.empty(mfsdp.muon_workspace_bytes(shards), dtype=torch.uint8, device=dev)
    mfsdp.muon_owner_step_host(shards, gh, gd, mom, ud, uh, ws, groups=groups)
    torch.cuda.synchronize()
    out = H.bf16_bits_to_f32(uh.view(torch.int16).numpy().view(np.uint16))
    for s in shards:
        seg = slice(s.offset, s.offset + s.rows * s.cols)
        assert np.array_equal(out[seg].view(np.uint32), u_ref[seg].view(np.uint32)), (groups, s.param_id)
    assert np.array_equal(mom.cpu().numpy(), m_ref)


@pytest.mark.parametrize("wdt", ["f32", "bf16"])
@pytest.mark.parametrize("mode", [0, 1, 2])
def test_apply_update_to_weights(mfsdp, wdt, mode):
    """W <- W*(1 - lr*wd) - lr*scale*O fused into the last epilogue.  Each
    element against the call's own O (one rounding), and the weight change
    against the fp64 oracle's: within the Newton-Schulz tolerance for fp32
    weights, and within it plus one bf16 rounding of the new weights (relative
    to the change) for bf16 weights, which start small enough (N(0, 1e-3))
    that a 10 % error in the applied scale cannot hide in that rounding."""
    from oracle import muon_apply_ref, muon_scale_ref
    dev = _dev()
    w = W.get("gpt2_block")
    plan, r, shards, numel = owner_set(mfsdp, w)
    grad = H.build_grad_buffer(w, shards, numel)
    zero = shards[1]                                   # one matrix with zero gradient: weights only decay
    grad[zero.offset:zero.offset + zero.rows * zero.cols] = 0
    mom0 = np.zeros(numel, np.float32)
    u_ref, _, _ = run_step(mfsdp, shards, grad, mom0, update_dtype=torch.float32)
    lr, wd = 0.02, 0.1
    rng = np.random.default_rng(17)
    W0 = (rng.standard_normal(numel) * (0.02 if wdt == "f32" else 1e-3)).astype(np.float32)
    tdt = torch.float32 if wdt == "f32" else torch.bfloat16
    Wt = torch.from_numpy(W0).to(dev).to(tdt)
    W0v = from_dev(Wt).astype(np.float64)              # the exact starting weights (bf16-rounded if bf16)
    g = to_dev_grad(grad)
    mom = torch.zeros(numel, dtype=torch.float32, device=dev)
    upd = torch.full((numel,), float("nan"), dtype=torch.float32, device=dev)
    ws = torch.empty(mfsdp.muon_workspace_bytes(shards), dtype=torch.uint8, device=dev)
    mfsdp.muon_owner_step_apply(shards, g, mom, upd, Wt, ws, lr=lr, weight_decay=wd, scale_mode=mode)
    torch.cuda.synchronize()
    O = from_dev(upd)
    Wn = from_dev(Wt).astype(np.float64)
    decay = np.float64(np.float32(1.0 - lr * wd))
    for s in shards:
        seg = slice(s.offset, s.offset + s.rows * s.cols)
        assert np.array_equal(O[seg].view(np.uint32), u_ref[seg].view(np.uint32)), "O must not change"
        scale = muon_scale_ref(s.rows, s.cols, mode)
        expect = W0v[seg] * decay - lr * scale * O[seg].astype(np.float64)   # from the GPU's own O
        tol = (2.0 ** -23 * 4 if wdt == "f32" else 2.0 ** -8) * (np.abs(W0v[seg]) + lr * scale * np.abs(O[seg]))
        assert np.all(np.abs(Wn[seg] - expect) <= tol + 1e-30), (s.param_id, mode)
        if s is zero:
            assert np.all(O[seg] == 0)
        else:
            G = grad_f64(grad, s)
            _, O_ref = muon_matrix_ref(G, np.zeros_like(G), w.beta, False, w.ns_steps, A, B, C, W.NS_EPS)
            W_ref = muon_apply_ref(W0v[seg].reshape(s.rows, s.cols), O_ref, lr, wd, scale)
            base = W0v[seg].reshape(s.rows, s.cols) * decay
            dW, dW_ref = Wn[seg].reshape(s.rows, s.cols) - base, W_ref - base
            bound = H.ns_tol(s.rows, s.cols)
            if wdt == "bf16":   # the new weights are rounded once to bf16 (half an ulp <= 2^-8 |W|)
                bound += 2.0 ** -8 * np.linalg.norm(W_ref) / np.linalg.norm(dW_ref)
            assert H.rel_fro(dW, dW_ref) <= bound, (s.param_id, mode, H.rel_fro(dW, dW_ref), bound)
    # without an update buffer the weights come out the same
    Wt2 = torch.from_numpy(W0).to(dev).to(tdt)
    mom2 = torch.zeros(numel, dtype=torch.float32, device=dev)
    mfsdp.muon_owner_step_apply(shards, g, mom2, None, Wt2, ws, lr=lr, weight_decay=wd, scale_mode=mode)
    torch.cuda.synchronize()
    assert torch.equal(Wt2.view(torch.int16 if wdt == "bf16" else torch.int32),
                       Wt.view(torch.int16 if wdt == "bf16" else torch.int32))


def test_determinism(mfsdp):
    w = W.get("gpt2_block")
    plan, r, shards, numel = owner_set(mfsdp, w)
    grad = H.build_grad_buffer(w, shards, numel)
    mom0 = np.zeros(numel, np.float32)
    u1, m1, _ = run_step(mfsdp, shards, grad, mom0, update_dtype=torch.float32)
    u2, m2, _ = run_step(mfsdp, shards, grad, mom0, update_dtype=torch.float32)
    assert np.array_equal(u1.view(np.uint32), u2.view(np.uint32))
    assert np.array_equal(m1, m2)


def test_in_place_update_over_grad(mfsdp):
    dev = _dev()
    w = W.get("gpt2_block")
    plan, r, shards, numel = owner_set(mfsdp, w)
    grad = H.build_grad_buffer(w, shards, numel)
    mom0 = np.zeros(numel, np.float32)
    ref_upd, _, _ = run_step(mfsdp, shards, grad, mom0, update_dtype=torch.bfloat16)
    g = to_dev_grad(grad)
    mom = torch.zeros(numel, dtype=torch.float32, device=dev)
    ws = torch.empty(mfsdp.muon_workspace_bytes(shards), dtype=torch.uint8, device=dev)
    mfsdp.muon_owner_step(shards, g, mom, g, ws)
    out = from_dev(g)
    for s in shards:
        seg = slice(s.offset, s.offset + s.rows * s.cols)
        assert np.array_equal(out[seg].view(np.uint32), ref_upd[seg].view(np.uint32))


def test_empty_owner_set(mfsdp):
    dev = _dev()
    g = torch.zeros(16, dtype=torch.bfloat16, device=dev)
    mfsdp.muon_owner_step([], g, torch.zeros(16, device=dev), g, None)


def test_narrow_and_full_width_tiles_agree(mfsdp):
    """A launch with few tiles per iteration (fewer than twice the SMs) runs
    256 x 128 tiles for each product with fewer full-width tiles than CTA
    pairs, a larger one 256 x 256 tiles throughout; each output element sums
    the same products in the same order either way.  The 768 x 2304 matrix run
    alone (narrow tiles), beside the GPT-2 block's other three matrices (narrow
    Gram and polynomial tiles, full-width update tiles) and inside a launch
    with twenty 2048 x 2048 matrices (full width) gives the same update and
    momentum, bit for bit."""
    dev = _dev()
    rng = np.random.default_rng(31)
    shapes = [(768, 2304)] + [(2048, 2048)] * 20
    shards, off = [], 0
    for i, (r, c) in enumerate(shapes):
        shards.append(mfsdp.make_shard(off, r, c, param_id=i))
        off += r * c
    numel = off
    grad = W.f32_to_bf16_bits((rng.standard_normal(numel) * 1e-3).astype(np.float32))
    mom0 = np.zeros(numel, np.float32)
    upd, mom, _ = run_step(mfsdp, shards, grad, mom0, update_dtype=torch.bfloat16)
    s = shards[0]
    n = s.rows * s.cols
    u1, m1, _ = run_step(mfsdp, [s], grad[:n].copy(), np.zeros(n, np.float32), update_dtype=torch.bfloat16)
    assert np.array_equal(u1.view(np.uint32), upd[:n].view(np.uint32))
    assert np.array_equal(m1, mom[:n])
    mixed = [(768, 2304), (768, 768), (768, 3072), (3072, 768)]
    shards_m, off = [], 0
    for i, (r, c) in enumerate(mixed):
        shards_m.append(mfsdp.make_shard(off, r, c, param_id=i))
        off += r * c
    grad_m = np.concatenate([grad[:n], W.f32_to_bf16_bits((rng.standard_normal(off - n) * 1e-3).astype(np.float32))])
    u2, m2, _ = run_step(mfsdp, shards_m, grad_m, np.zeros(off, np.float32), update_dtype=torch.bfloat16)
    assert np.array_equal(u2[:n].view(np.uint32), upd[:n].view(np.uint32))
    assert np.array_equal(m2[:n], mom[:n])
    check_matrix(s, upd, mom, grad, mom0, ns_steps=5)
