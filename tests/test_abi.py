"""Host-side tests of the C ABI (no GPU needed): the library loads and exports
every entry point include/mfsdp.h declares, the C++ planner reproduces the
oracle planner bit for bit, and every argument error is reported with its
status code before any device work is queued.

All pointers below are fake; every case is rejected by the host checks, so no
CUDA call is made (these tests are safe on a machine with a GPU too)."""
import ctypes
import os
import re

import pytest

from oracle.planner import plan_owners_ref
from matrix_optimizers_under_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "mfsdp.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mfsdp_\w+)\s*\(", src)))


def test_exports_every_declared_symbol(mfsdp):
    decl = declared_functions()
    assert len(decl) >= 8
    lib = mfsdp.raw_lib()
    for name in decl:
        assert hasattr(lib, name), name
    assert sorted(mfsdp.EXPORTED) == decl
    assert mfsdp.version().count(".") == 2


def test_status_strings(mfsdp):
    seen = set()
    for code in range(0, -10, -1):
        s = mfsdp.status_string(code)
        assert s and s != "unknown status"
        seen.add(s)
    assert len(seen) == 10
    assert mfsdp.status_string(-1234) == "unknown status"


def _compare(plan, ref):
    assert [s.as_dict() for s in plan.matrix_shards] == ref["matrix_shards"]
    assert [s.as_dict() for s in plan.tail_shards] == ref["tail_shards"]
    assert plan.rank_matrix_elems == ref["rank_matrix_elems"]
    assert plan.rank_tail_elems == ref["rank_tail_elems"]


@pytest.mark.parametrize("name", W.ORDER)
def test_planner_bit_exact_on_workloads(mfsdp, name):
    w = W.get(name)
    params = w.param_table()
    for world in sorted({1, 2, w.world, 64}):
        _compare(mfsdp.plan_owners(params, world, w.ns_steps, w.align_elems),
                 plan_owners_ref(params, world, w.ns_steps, w.align_elems))


@pytest.mark.parametrize("seed", range(25))
def test_planner_bit_exact_fuzz(mfsdp, seed):
    params = W.ragged_params(seed, 1 + seed * 7)
    for world in (1, 3, 8):
        for align in (1, 64, 128):
            for steps in (0, 1, 5):
                _compare(mfsdp.plan_owners(params, world, steps, align), plan_owners_ref(params, world, steps, align))


def test_planner_errors(mfsdp):
    with pytest.raises(mfsdp.MfsdpError) as e:
        mfsdp.plan_owners([(4, 4, 0)], 0)
    assert e.value.status == mfsdp.ERR_INVALID_ARG
    with pytest.raises(mfsdp.MfsdpError) as e:
        mfsdp.plan_owners([(0, 4, 0)], 2)
    assert e.value.status == mfsdp.ERR_UNSUPPORTED_SHAPE
    with pytest.raises(mfsdp.MfsdpError) as e:
        mfsdp.plan_owners([(4, 4, 7)], 2)
    assert e.value.status == mfsdp.ERR_INVALID_ARG
    with pytest.raises(mfsdp.MfsdpError) as e:   # cost above 2^64
        mfsdp.plan_owners([(1 << 24, 1 << 24, 0)], 2, ns_steps=64)
    assert e.value.status == mfsdp.ERR_UNSUPPORTED_SHAPE
    plan = mfsdp.plan_owners([], 3)
    assert plan.matrix_shards == [] and plan.rank_matrix_elems == [0, 0, 0]


def gram_shape(s, l):
    """Shapes that may run the Gram-space form (include/mfsdp.h)."""
    return s >= 128 and l >= 2 * s and l >= s + 384


def test_workspace_layout(mfsdp):
    shards = [mfsdp.make_shard(0, 256, 512), mfsdp.make_shard(131072, 300, 130), mfsdp.make_shard(200000, 1, 9),
              mfsdp.make_shard(200064, 200, 640)]
    lay = mfsdp.muon_workspace_layout(shards)
    total = mfsdp.muon_workspace_bytes(shards)
    assert [l[4:] for l in lay] == [(256, 512, 256, 512), (256, 384, 130, 300), (256, 128, 1, 9),
                                    (256, 640, 200, 640)]
    end = 0
    for x0, x1, a, b, sp, lp, s_, l_ in lay:
        assert x0 % 1024 == 0 and x0 >= end
        # the second X region also holds C and both Q of the Gram-space form
        # for shapes that may run it
        x1_bytes = max(sp * lp, 3 * sp * sp) * 2 if gram_shape(s_, l_) else sp * lp * 2
        assert x1 == x0 + sp * lp * 2 and a == x1 + x1_bytes and b == a + sp * sp * 2
        end = b + sp * sp * 2
    assert total == end
    assert mfsdp.muon_workspace_bytes([mfsdp.make_shard(0, 0, 5)]) == 0
    assert mfsdp.muon_workspace_bytes([mfsdp.make_shard(0, 40000, 40000)]) == 0
    # the Gram-space form: 200 x 640 only (256 x 512 and 130 x 300: l < s +
    # 384 with s < 384; 1 x 9: s < 128), for 1 .. 5 steps; C and the Q
    # ping-pong follow each other in X1's region
    for steps, want in [(0, [0, 0, 0, 0]), (1, [0, 0, 0, 1]), (5, [0, 0, 0, 1]), (6, [0, 0, 0, 0])]:
        gl = mfsdp.muon_gram_space_layout(shards, steps)
        assert [g[0] for g in gl] == want
        for (flag, c, q0, q1), (x0, x1, a, b, sp, lp, _, _) in zip(gl, lay):
            assert c == x1 and q0 == c + sp * sp * 2 and q1 == q0 + sp * sp * 2
    dense, executed = mfsdp.muon_step_flops(shards[3:], 5)
    # 200 x 640 in Gram space (padded to 256 x 640): A_0 (K = 640), 5 P, 4
    # each of C, A, Q (K = 256) and the final Q X0, each a single 256 x 256
    # tile but the last
    tile = 2 * 256 * 256
    assert executed == tile * 640 + (5 + 3 * 4) * tile * 256 + 2 * 256 * 256 * 640
    assert dense == 5 * (4 * 200 * 200 * 640 + 2 * 200 ** 3)


# ------------------------------------------------------------ error paths
BF, F32 = 1, 0
G, M, U, WS = 0x10000000, 0x20000000, 0x30000000, 0x40000000   # fake, aligned, disjoint


def step(mfsdp, shards, grad=G, gdt=BF, mom=M, upd=U, udt=BF, numel=1 << 20, ns=5, ws=WS, wsb=None,
         beta=0.95, nesterov=0, eps=1e-7, phases=None):
    arr = (mfsdp.MatrixShard * max(len(shards), 1))(*shards)
    if wsb is None:
        wsb = mfsdp.muon_workspace_bytes(shards) if shards else 0
    args = (arr, len(shards), grad, gdt, mom, upd, udt, numel, beta, nesterov, ns, 3.4445, -4.775, 2.0315, eps, ws,
            wsb, None)
    if phases is None:
        return mfsdp.raw_lib().mfsdp_muon_owner_step(*args)
    return mfsdp.raw_lib().mfsdp_muon_owner_step_phases(*args, phases)


def test_step_error_paths(mfsdp):
    ok = [mfsdp.make_shard(0, 256, 512), mfsdp.make_shard(131072, 512, 256)]
    assert step(mfsdp, [], grad=None, mom=None, upd=None, ws=None) == mfsdp.OK   # empty owner set: no-op
    assert step(mfsdp, ok, gdt=7) == mfsdp.ERR_UNSUPPORTED_DTYPE
    assert step(mfsdp, ok, udt=2) == mfsdp.ERR_UNSUPPORTED_DTYPE
    assert step(mfsdp, ok, ns=-1) == mfsdp.ERR_INVALID_ARG
    assert step(mfsdp, ok, ns=65) == mfsdp.ERR_INVALID_ARG
    assert step(mfsdp, ok, nesterov=2) == mfsdp.ERR_INVALID_ARG
    assert step(mfsdp, ok, eps=-1.0) == mfsdp.ERR_INVALID_ARG
    assert step(mfsdp, ok, beta=float("nan")) == mfsdp.ERR_INVALID_ARG
    assert step(mfsdp, ok, grad=None) == mfsdp.ERR_INVALID_ARG
    assert step(mfsdp, ok, numel=-5) == mfsdp.ERR_INVALID_ARG
    assert step(mfsdp, ok, grad=G + 2) == mfsdp.ERR_MISALIGNED
    assert step(mfsdp, ok, mom=M + 4) == mfsdp.ERR_MISALIGNED
    assert step(mfsdp, ok, ws=WS + 16) == mfsdp.ERR_MISALIGNED
    assert step(mfsdp, [mfsdp.make_shard(0, 0, 4)]) == mfsdp.ERR_UNSUPPORTED_SHAPE
    assert step(mfsdp, [mfsdp.make_shard(0, 40000, 40000)], numel=1 << 31) == mfsdp.ERR_UNSUPPORTED_SHAPE
    assert step(mfsdp, [mfsdp.make_shard(-128, 16, 16)]) == mfsdp.ERR_OUT_OF_BOUNDS
    assert step(mfsdp, [mfsdp.make_shard(1 << 20, 16, 16)]) == mfsdp.ERR_OUT_OF_BOUNDS
    assert step(mfsdp, ok, numel=131072 + 512 * 255) == mfsdp.ERR_OUT_OF_BOUNDS
    assert step(mfsdp, [mfsdp.make_shard(0, 256, 512), mfsdp.make_shard(131071, 4, 4)]) == mfsdp.ERR_OVERLAP
    # distinct buffers that overlap
    assert step(mfsdp, ok, mom=G + 1024) == mfsdp.ERR_OVERLAP
    assert step(mfsdp, ok, upd=G + 1024) == mfsdp.ERR_OVERLAP
    assert step(mfsdp, ok, upd=G, udt=F32) == mfsdp.ERR_OVERLAP        # same address, different dtype
    assert step(mfsdp, ok, ws=G) == mfsdp.ERR_OVERLAP
    assert step(mfsdp, ok, wsb=mfsdp.muon_workspace_bytes(ok) - 1) == mfsdp.ERR_WORKSPACE_TOO_SMALL
    # the phase-split entry point checks the same arguments, plus the phase set
    assert step(mfsdp, ok, phases=0) == mfsdp.ERR_INVALID_ARG
    assert step(mfsdp, ok, phases=4) == mfsdp.ERR_INVALID_ARG
    assert step(mfsdp, ok, phases=mfsdp.PHASE_MOMENTUM, grad=G + 2) == mfsdp.ERR_MISALIGNED
    assert step(mfsdp, ok, phases=mfsdp.PHASE_NEWTON_SCHULZ, ns=-1) == mfsdp.ERR_INVALID_ARG
    assert step(mfsdp, [], phases=mfsdp.PHASE_NEWTON_SCHULZ, grad=None, mom=None, upd=None, ws=None) == mfsdp.OK


def test_host_entry_error_paths(mfsdp):
    lib = mfsdp.raw_lib()
    ok = [mfsdp.make_shard(0, 256, 512)]
    arr = (mfsdp.MatrixShard * 1)(*ok)
    wsb = mfsdp.muon_workspace_bytes(ok)
    H1, H2 = 0x50000000, 0x60000000

    def call(gh=H1, uh=H2, groups=4, grad=G, ws=WS):
        return lib.mfsdp_muon_owner_step_host(arr, 1, gh, grad, BF, M, U, uh, BF, 1 << 20, 0.95, 0, 5, 3.4445,
                                              -4.775, 2.0315, 1e-7, ws, wsb, groups, None)
    assert call(groups=-1) == mfsdp.ERR_INVALID_ARG
    assert call(gh=None) == mfsdp.ERR_INVALID_ARG
    assert call(uh=None) == mfsdp.ERR_INVALID_ARG
    assert call(grad=G + 2) == mfsdp.ERR_MISALIGNED
    assert call(ws=G) == mfsdp.ERR_OVERLAP


def test_apply_entry_error_paths(mfsdp):
    lib = mfsdp.raw_lib()
    ok = [mfsdp.make_shard(0, 256, 512)]
    arr = (mfsdp.MatrixShard * 1)(*ok)
    wsb = mfsdp.muon_workspace_bytes(ok)
    Wt = 0x70000000

    def call(w=Wt, wdt=F32, upd=U, mode=1, ns=5, lr=0.02):
        return lib.mfsdp_muon_owner_step_apply(arr, 1, G, BF, M, upd, BF, w, wdt, 1 << 20, 0.95, 0, ns, 3.4445,
                                               -4.775, 2.0315, 1e-7, lr, 0.1, mode, WS, wsb, None)
    assert call(wdt=5) == mfsdp.ERR_UNSUPPORTED_DTYPE
    assert call(mode=3) == mfsdp.ERR_INVALID_ARG
    assert call(ns=0) == mfsdp.ERR_INVALID_ARG
    assert call(lr=float("nan")) == mfsdp.ERR_INVALID_ARG
    assert call(w=None) == mfsdp.ERR_INVALID_ARG
    assert call(w=Wt + 4) == mfsdp.ERR_MISALIGNED
    assert call(w=G) == mfsdp.ERR_OVERLAP
    assert call(w=U) == mfsdp.ERR_OVERLAP
    assert call(w=None, upd=None) == mfsdp.ERR_INVALID_ARG


def test_adamw_error_paths(mfsdp):
    lib = mfsdp.raw_lib()
    P, Gp, Mm, V = 0x10000000, 0x20000000, 0x30000000, 0x40000000

    def call(p=P, g=Gp, m=Mm, v=V, n=4096, b1=0.9, b2=0.95, step=1, lr=1e-3):
        return lib.mfsdp_adamw_tail_step(p, g, m, v, n, lr, b1, b2, 1e-8, 0.1, step, None)
    assert call(n=0, p=None, g=None, m=None, v=None) == mfsdp.OK
    assert call(n=-1) == mfsdp.ERR_INVALID_ARG
    assert call(step=0) == mfsdp.ERR_INVALID_ARG
    assert call(b1=1.0) == mfsdp.ERR_INVALID_ARG
    assert call(b2=-0.1) == mfsdp.ERR_INVALID_ARG
    assert call(lr=float("inf")) == mfsdp.ERR_INVALID_ARG
    assert call(g=None) == mfsdp.ERR_INVALID_ARG
    assert call(v=V + 8) == mfsdp.ERR_MISALIGNED
    assert call(m=P + 1024) == mfsdp.ERR_OVERLAP


def test_step_flops(mfsdp):
    shards = [mfsdp.make_shard(0, 4096, 14336), mfsdp.make_shard(0, 1024, 4096), mfsdp.make_shard(0, 300, 130),
              mfsdp.make_shard(0, 1408, 2048)]
    dense, executed = mfsdp.muon_step_flops(shards, 5)
    want_dense = sum(5 * (4 * min(r, c) ** 2 * max(r, c) + 2 * min(r, c) ** 3) for r, c in
                     [(4096, 14336), (1024, 4096), (300, 130), (1408, 2048)])
    assert dense == want_dense

    def ex(s, l, steps=5):   # outputs: short side padded to 256, long to 128; upper-triangle 256x256 tiles when
        # symmetric; a contraction over the short side runs to s rounded up to 128
        sp, lp, ks = -(-s // 256) * 256, -(-l // 128) * 128, -(-s // 128) * 128
        nb2 = sp // 256
        tiles = nb2 * (nb2 + 1) // 2
        gram, sym, upd = tiles * 256 * 256 * 2 * lp, tiles * 256 * 256 * 2 * ks, 2 * sp * lp * ks
        if gram_shape(s, l) and 1 <= steps <= 5:
            # Gram space: A_0, one P per step, C, A and Q for all but one, the final Q X0
            return gram + steps * sym + 3 * (steps - 1) * sym + upd
        return steps * (gram + sym + upd)
    # the first two run the Gram-space form, 130 x 300 and 1408 x 2048 the direct one
    # (1408 x 2048: outputs 1536 rows, contractions over the short side K = 1408)
    assert executed == ex(4096, 14336) + ex(1024, 4096) + ex(130, 300) + ex(1408, 2048)
    sym_1408 = 21 * 256 * 256 * 2 * 1408
    assert ex(1408, 2048) == 5 * (21 * 256 * 256 * 2 * 2048 + sym_1408 + 2 * 1536 * 2048 * 1408)
    assert executed < dense     # the symmetric skipping outweighs the padding here
    assert mfsdp.muon_step_flops([], 5) == (0, 0)
    # at 6 steps every shape takes the direct form
    dense6, executed6 = mfsdp.muon_step_flops(shards, 6)
    assert executed6 == sum(ex(s, l, 6) for s, l in [(4096, 14336), (1024, 4096), (130, 300), (1408, 2048)])


def test_newton_schulz_index_limits(mfsdp):
    """The one-launch Newton-Schulz kernel indexes tiles and counts completions in
    int32, and its tensor copies address the workspace in 128-byte rows with int32
    coordinates.  Owner sets past either limit are refused on the host, before
    anything is queued (the pointers here are fake)."""
    big = [mfsdp.make_shard(0, 32768, 1 << 24)]          # 2 * 8256 + 128 * 65536 tiles per iteration
    assert step(mfsdp, big, numel=32768 << 24, ns=64, wsb=1 << 62) == mfsdp.ERR_UNSUPPORTED_SHAPE
    wide = [mfsdp.make_shard(0, 16384, 1 << 24)]         # counts fit over 5 steps, workspace > 2^31 rows
    assert step(mfsdp, wide, numel=16384 << 24, ns=5, wsb=1 << 62) == mfsdp.ERR_UNSUPPORTED_SHAPE
    # the same shape with a workspace that is too small still reports the shape first
    assert step(mfsdp, wide, numel=16384 << 24, ns=5, wsb=1 << 20) == mfsdp.ERR_UNSUPPORTED_SHAPE


def test_inject_stall_rejects_negative_tile(mfsdp):
    assert mfsdp.raw_lib().mfsdp_test_inject_stall(-1) == mfsdp.ERR_INVALID_ARG


def test_host_step_groups(mfsdp):
    """groups = 0: g = round(sqrt(copy bytes / 50 MB)); one group for g <= 1;
    cost-balanced offset ranges for g == 2 or fewer than 5 shards; for g >= 6
    min(g, 16) balanced ranges between a head and a tail of up to two of the
    smallest shards with the largest short side (at most 1/(2 min(g, 16)) of
    the elements per end); for 3 <= g <= 5 the ramp (small -> large -> small by
    size, cut at 4/28/72/96 % of the bytes, a shard placed by the midpoint of
    its bytes).  groups >= 1: offset ranges of balanced cost 4 s^2 l + 2 s^3 +
    s l.  Expected values worked by hand."""
    import torch
    bf, f32 = torch.bfloat16, torch.float32

    def layout(dims):
        out, off = [], 0
        for i, (r, c) in enumerate(dims):
            out.append(mfsdp.make_shard(off, r, c, param_id=i))
            off += r * c
        return out

    assert mfsdp.host_step_groups(layout([(5000, 5000)]), bf, bf) == (1, [0])          # 100 MB: g = 1
    four = layout([(8192, 8192)] * 4)                                  # 1.07 GB: g = 5, but 4 shards
    assert mfsdp.host_step_groups(four, bf, bf) == (4, [0, 1, 2, 3])
    three = layout([(4096, 4096)] * 3)                                 # 201 MB: g = 2
    assert mfsdp.host_step_groups(three, bf, bf) == (2, [0, 0, 1])
    # 499 MB, g = 3: the ramp.  By size s0 < s5 < s1 < s2 < s3 < s4, so the
    # sequence is s0 s1 s3 | s4 s2 s5; byte midpoints at 0.4, 2.5, 17.6, 58.0,
    # 91.6 and 99.2 % of the total.
    six = layout([(1024, 1024), (2048, 2048), (4096, 4096), (4096, 8192), (8192, 8192), (1024, 2048)])
    assert mfsdp.host_step_groups(six, bf, bf) == (5, [0, 0, 3, 1, 2, 4])
    eight = layout([(8192, 8192)] * 8)                                 # 2.15 GB: g = 7, balanced
    assert mfsdp.host_step_groups(eight, bf, bf) == (7, [0, 0, 1, 2, 3, 4, 5, 6])
    # 40 equal shards, 10.7 GB: g = 15; one shard (67M elements) fits the
    # 1/30 limit (89M) at each end: head, 15 balanced groups, tail
    many = layout([(8192, 8192)] * 40)
    ng, gof = mfsdp.host_step_groups(many, bf, bf)
    assert ng == 17 and gof[0] == 0 and gof[1] == 16 and gof[2:] == sorted(gof[2:]) and set(gof[2:]) == set(range(1, 16))
    assert mfsdp.host_step_groups(many, f32, f32)[0] == 18            # 21.5 GB: g = 21, capped at 16 + 2
    # layers of 5 wide 4096x14336, one 4096^2 and one 1024x4096: 5.03 GB, g = 10,
    # limit 62.9M elements per end; the largest short side is 4096 and the
    # smallest such shards are the 4096^2 ones: two at each end, in offset order
    layers = layout(([(4096, 14336)] * 5 + [(4096, 4096), (1024, 4096)]) * 4)
    ng, gof = mfsdp.host_step_groups(layers, bf, bf)
    sq = [i for i in range(28) if i % 7 == 5]
    assert ng == 12 and [gof[i] for i in sq] == [0, 0, 11, 11]
    rest = [gof[i] for i in range(28) if i % 7 != 5]
    assert rest == sorted(rest) and set(rest) == set(range(1, 11))
    # explicit groups: s4 holds 74 % of the cost, so the cut falls after it
    assert mfsdp.host_step_groups(six, bf, bf, groups=2) == (2, [0, 0, 0, 0, 0, 1])
    assert mfsdp.host_step_groups(six, bf, bf, groups=1) == (1, [0] * 6)
    assert mfsdp.host_step_groups(three, f32, f32, groups=16) == (3, [0, 1, 2])
    # fp32 gradients: 6 bytes per element -> 749 MB, g = 4: still the ramp
    assert mfsdp.host_step_groups(six, f32, bf)[0] == 5
    for bad in (dict(groups=-1), dict(grad_dtype=torch.float16), dict(update_dtype=torch.int32)):
        kw = dict(grad_dtype=bf, update_dtype=bf, groups=0)
        kw.update(bad)
        assert mfsdp.host_step_groups(six, **kw) == (0, [])
    assert mfsdp.host_step_groups([], bf, bf) == (0, [])


def test_static_scratch_error_paths(mfsdp):
    """The no-workspace entry point checks its arguments on the host, with the
    regular entry point's statuses, before it looks up its scratch array."""
    lib = mfsdp.raw_lib()
    ok = [mfsdp.make_shard(0, 256, 512)]
    arr = (mfsdp.MatrixShard * 1)(*ok)
    big = (mfsdp.MatrixShard * 1)(mfsdp.make_shard(0, 4096, 4096))

    def call(shards=arr, n=1, grad=G, gdt=BF, upd=U, udt=BF, numel=1 << 20, ns=5, beta=0.95):
        return lib.mfsdp_muon_owner_step_static_scratch(shards, n, grad, gdt, M, upd, udt, numel, beta, 0, ns,
                                                        3.4445, -4.775, 2.0315, 1e-7, None)
    assert call(grad=None) == mfsdp.ERR_INVALID_ARG
    assert call(gdt=7) == mfsdp.ERR_UNSUPPORTED_DTYPE
    assert call(udt=7) == mfsdp.ERR_UNSUPPORTED_DTYPE
    assert call(grad=G + 2) == mfsdp.ERR_MISALIGNED
    assert call(ns=-1) == mfsdp.ERR_INVALID_ARG
    assert call(beta=float("nan")) == mfsdp.ERR_INVALID_ARG
    assert call(numel=100) == mfsdp.ERR_OUT_OF_BOUNDS
    assert call(upd=G, udt=F32) == mfsdp.ERR_OVERLAP         # the same buffer in another dtype (in place needs both equal)
    assert call(shards=big, numel=4096 * 4096) == mfsdp.ERR_WORKSPACE_TOO_SMALL
    assert call(shards=None, n=0, grad=None, upd=None) == mfsdp.OK
    assert call(shards=None, n=-1) == mfsdp.ERR_INVALID_ARG


def test_device_status_error_paths(mfsdp):
    import ctypes
    lib = mfsdp.raw_lib()
    detail = ctypes.c_int32(7)
    assert lib.mfsdp_muon_device_status(None, None, ctypes.byref(detail)) == mfsdp.ERR_INVALID_ARG


def test_static_scratch_status_without_device(mfsdp):
    """With no usable GPU the static-scratch status query cannot look up its
    array and reports a CUDA error (it never reads a host-side stand-in)."""
    import ctypes
    import torch
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present")
    detail = ctypes.c_int32(7)
    assert mfsdp.raw_lib().mfsdp_muon_static_scratch_status(None, ctypes.byref(detail)) == mfsdp.ERR_CUDA
