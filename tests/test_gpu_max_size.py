"""The owner step at the largest short side the ABI accepts, checked exactly
where the oracle's dense form is out of reach.

G = c * P with P a signed (partial) permutation: every one of its s singular
values is c, so the Newton-Schulz output is phi(1/sqrt(s)) * P (MatrixFSDP --
Abstract: the owner-local update is full-matrix Muon; the singular-value
closed form is pinned in the oracle's own tests), and every entry off the
permutation's pattern is exactly zero (all products of zeros are exact zeros).
phi(1/sqrt(s)) is taken from the oracle on the 2 x 2 matrix
diag(1/sqrt(s), sqrt(1 - 1/s)), which has unit norm like the big input and the
same first normalised singular value.  The big case still runs every tile of a
32768-wide Gram, polynomial and update, the transposed reads of the symmetric
products' blocks below the diagonal and (for the tall cases) the transposed
final stores.  65537 x 32768 (over 2^31 elements, long side at least twice the
short one) runs the Gram-space form at the largest short side: every tile of
its 32768-wide A, P, C and Q products and of the final Q X0.
"""
import math

import numpy as np
import pytest

from oracle import newton_schulz_ref
from matrix_optimizers_under_gb300 import workloads as W
from tests import helpers as H

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

A, B, C = W.NS_COEFFS


def phi_at(s: int) -> float:
    x = 1.0 / math.sqrt(s)
    D = np.diag([x, math.sqrt(1.0 - x * x)])
    return float(newton_schulz_ref(D, 5, A, B, C, W.NS_EPS)[0, 0])


@pytest.mark.parametrize("rows,cols", [(32768, 32768), (40001, 20483), (65537, 32768)])
def test_signed_permutation_at_max_short_side(mfsdp, rows, cols):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda:0")
    s = min(rows, cols)
    gen = torch.Generator().manual_seed(rows * 7 + cols)
    # one nonzero in each of s distinct rows and columns
    if rows <= cols:
        r_idx = torch.arange(rows)
        c_idx = torch.randperm(cols, generator=gen)[:rows]
    else:
        c_idx = torch.arange(cols)
        r_idx = torch.randperm(rows, generator=gen)[:cols]
    sign = torch.where(torch.rand(s, generator=gen) < 0.5, -1.0, 1.0)
    c = 2.0 ** -8                                     # exact in bf16
    flat = (r_idx * cols + c_idx).to(dev)
    numel = rows * cols
    grad = torch.zeros(numel, dtype=torch.bfloat16, device=dev)
    grad[flat] = (c * sign).to(torch.bfloat16).to(dev)
    mom = torch.zeros(numel, dtype=torch.float32, device=dev)
    upd = torch.full((numel,), float("nan"), dtype=torch.bfloat16, device=dev)
    shards = [mfsdp.make_shard(0, rows, cols)]
    gram = mfsdp.muon_gram_space_layout(shards, 5)[0][0]
    assert gram == (1 if max(rows, cols) >= 2 * s else 0), "program chosen for the shape"
    ws = torch.empty(mfsdp.muon_workspace_bytes(shards), dtype=torch.uint8, device=dev)
    mfsdp.muon_owner_step(shards, grad, mom, upd, ws, beta=0.95, ns_steps=5, coeffs=W.NS_COEFFS, eps=W.NS_EPS)
    st, detail = mfsdp.muon_device_status(ws)
    assert st == mfsdp.OK, (st, detail)
    torch.cuda.synchronize()
    # momentum from zero is the gradient, bit for bit
    assert torch.equal(mom[flat], (c * sign).to(dev).float())
    expect = phi_at(s) * sign.double()
    got = upd[flat].double().cpu()
    err = float(torch.linalg.vector_norm(got - expect) / torch.linalg.vector_norm(expect))
    assert err <= H.NS_REL_FRO, f"{rows}x{cols}: relative error {err:.3e} on the permutation's entries"
    upd[flat] = 0
    assert int(torch.count_nonzero(upd)) == 0, "nonzero update off the permutation's pattern"
    del grad, mom, upd, ws
    torch.cuda.empty_cache()
