"""Seeded synthetic workloads for the owner-local optimizer step.

This module is the one piece that both the CUDA path's callers and the fp64
oracle's callers share: it holds parameter lists (shapes and kinds), seeds,
value distributions and hyper-parameters, and nothing of the method's own
arithmetic (no momentum, no Newton-Schulz, no AdamW, no planning).

Shapes follow the transformer workloads the MatrixFSDP paper trains on
(MatrixFSDP: Communication-Free Matrix Optimizers Under ZeRO-3 Parameter
Sharding -- Abstract: "for each 2D weight" / "non-matrix tensors are packed into
tail owners").  The pages fix no sizes; the five owner sets below are the
synthetic stand-ins named in the design notes, sized like GPT-2-small, a
1.3B Llama-style model, Llama-3-8B and a skewed mixture-of-experts layer.

Random numbers: every tensor draws from its own NumPy PCG64 stream seeded with
``[config_seed, param_id]`` (plus a salt for the AdamW tail's second tensor), so a
test can regenerate any single tensor without generating the whole set.
Gradients are drawn in fp32 and, for bf16 workloads, rounded to bf16 with
round-to-nearest-even; the same bytes feed the GPU and the oracle.
"""
from __future__ import annotations

import dataclasses
import multiprocessing as mp
import os
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

KIND_MATRIX = 0  # a 2D weight that Muon updates
KIND_TAIL = 1    # a tensor packed into a tail owner and updated by AdamW

# Muon's published quintic Newton-Schulz coefficients and step count
# (Muon, Jordan et al. 2024, the matrix optimizer the MatrixFSDP paper's
# Section 1 builds on).  The MatrixFSDP pages do not restate them.
NS_COEFFS = (3.4445, -4.7750, 2.0315)
NS_STEPS = 5
NS_EPS = 1e-7


@dataclasses.dataclass(frozen=True)
class Param:
    name: str
    rows: int
    cols: int
    kind: int

    @property
    def numel(self) -> int:
        return self.rows * self.cols


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    params: Tuple[Param, ...]
    world: int               # simulated data-parallel ranks for the planner
    seed: int
    grad_dtype: str          # "f32" or "bf16" storage of the flat gradient buffer
    grad_dist: str           # "normal" or "student_t3"
    grad_scale: float        # std (normal) or scale (Student-t)
    tail_scale: float        # std of AdamW tail params and grads
    zero_params: Tuple[int, ...] = ()   # param ids whose gradient is all zero
    beta: float = 0.95
    nesterov: bool = False
    ns_steps: int = NS_STEPS
    ns_coeffs: Tuple[float, float, float] = NS_COEFFS
    ns_eps: float = NS_EPS
    lr: float = 1e-3
    betas: Tuple[float, float] = (0.9, 0.95)
    adam_eps: float = 1e-8
    weight_decay: float = 0.1
    step: int = 1
    align_elems: int = 128

    def param_table(self) -> List[Tuple[int, int, int]]:
        return [(p.rows, p.cols, p.kind) for p in self.params]


def _tiny() -> Workload:
    params = (Param("w", 256, 512, KIND_MATRIX), Param("tail", 4096, 1, KIND_TAIL))
    return Workload("tiny", params, world=1, seed=0, grad_dtype="f32",
                    grad_dist="normal", grad_scale=1e-2, tail_scale=1e-3)


def _gpt2_block() -> Workload:
    d = 768
    p = [
        Param("ln1.weight", d, 1, KIND_TAIL), Param("ln1.bias", d, 1, KIND_TAIL),
        Param("attn.c_attn.weight", d, 3 * d, KIND_MATRIX), Param("attn.c_attn.bias", 3 * d, 1, KIND_TAIL),
        Param("attn.c_proj.weight", d, d, KIND_MATRIX), Param("attn.c_proj.bias", d, 1, KIND_TAIL),
        Param("ln2.weight", d, 1, KIND_TAIL), Param("ln2.bias", d, 1, KIND_TAIL),
        Param("mlp.c_fc.weight", d, 4 * d, KIND_MATRIX), Param("mlp.c_fc.bias", 4 * d, 1, KIND_TAIL),
        Param("mlp.c_proj.weight", 4 * d, d, KIND_MATRIX), Param("mlp.c_proj.bias", d, 1, KIND_TAIL),
    ]
    return Workload("gpt2_block", tuple(p), world=1, seed=1, grad_dtype="bf16",
                    grad_dist="normal", grad_scale=1e-3, tail_scale=1e-3)


def _llama(layers: int, d: int, ffn: int, kv: int, vocab: Optional[int]) -> List[Param]:
    """Llama-style parameter list in declaration order (weights are [out, in])."""
    p: List[Param] = []
    if vocab is not None:
        p.append(Param("embed_tokens.weight", vocab, d, KIND_TAIL))
    for i in range(layers):
        pre = f"layers.{i}."
        p += [
            Param(pre + "input_layernorm.weight", d, 1, KIND_TAIL),
            Param(pre + "self_attn.q_proj.weight", d, d, KIND_MATRIX),
            Param(pre + "self_attn.k_proj.weight", kv, d, KIND_MATRIX),
            Param(pre + "self_attn.v_proj.weight", kv, d, KIND_MATRIX),
            Param(pre + "self_attn.o_proj.weight", d, d, KIND_MATRIX),
            Param(pre + "post_attention_layernorm.weight", d, 1, KIND_TAIL),
            Param(pre + "mlp.gate_proj.weight", ffn, d, KIND_MATRIX),
            Param(pre + "mlp.up_proj.weight", ffn, d, KIND_MATRIX),
            Param(pre + "mlp.down_proj.weight", d, ffn, KIND_MATRIX),
        ]
    p.append(Param("norm.weight", d, 1, KIND_TAIL))
    if vocab is not None:
        p.append(Param("lm_head.weight", vocab, d, KIND_TAIL))
    return p


def llama_param_table(layers: int, d: int, ffn: int, kv: int) -> List[Tuple[int, int, int]]:
    """(rows, cols, kind) of a Llama-style layer stack without embedding or head."""
    return [(p.rows, p.cols, p.kind) for p in _llama(layers, d, ffn, kv, None)]


def _llama_1p3b() -> Workload:
    # 24 layers, d=2048, ffn=5504, no grouped-query attention stated, vocab 32000
    # untied embedding and head, both kept on AdamW.
    params = _llama(24, 2048, 5504, 2048, 32000)
    return Workload("llama_1p3b_rank", tuple(params), world=8, seed=2, grad_dtype="bf16",
                    grad_dist="normal", grad_scale=1e-3, tail_scale=1e-3)


def _llama3_8b() -> Workload:
    params = _llama(32, 4096, 14336, 1024, None)
    return Workload("llama3_8b_rank", tuple(params), world=8, seed=3, grad_dtype="bf16",
                    grad_dist="student_t3", grad_scale=1e-3, tail_scale=1e-3)


def _moe() -> Workload:
    p: List[Param] = []
    for i in range(4):
        for n in ("q", "k", "v", "o"):
            p.append(Param(f"attn.{i}.{n}_proj.weight", 2048, 2048, KIND_MATRIX))
    n_exp = 128
    for e in range(n_exp):
        p.append(Param(f"experts.{e}.up_proj.weight", 1408, 2048, KIND_MATRIX))
        p.append(Param(f"experts.{e}.down_proj.weight", 2048, 1408, KIND_MATRIX))
    p.append(Param("packed_tail", 50_000_000, 1, KIND_TAIL))
    seed = 4
    # 10% of experts (13 of 128) are unrouted: their gradients are exactly zero.
    perm = np.random.default_rng([seed, 1_000_003]).permutation(n_exp)
    zero_experts = sorted(int(e) for e in perm[:13])
    zero_ids = []
    for e in zero_experts:
        zero_ids += [16 + 2 * e, 16 + 2 * e + 1]
    return Workload("moe_skewed", tuple(p), world=1, seed=seed, grad_dtype="bf16",
                    grad_dist="normal", grad_scale=1e-3, tail_scale=1e-3,
                    zero_params=tuple(zero_ids))


WORKLOADS: Dict[str, Workload] = {w.name: w for w in
                                  (_tiny(), _gpt2_block(), _llama_1p3b(), _llama3_8b(), _moe())}
ORDER = ("tiny", "gpt2_block", "llama_1p3b_rank", "llama3_8b_rank", "moe_skewed")


def get(name: str) -> Workload:
    return WORKLOADS[name]


# ----------------------------------------------------------------------------
# value generators
# ----------------------------------------------------------------------------

def _rng(w: Workload, param_id: int, salt: int = 0) -> np.random.Generator:
    return np.random.default_rng([w.seed, param_id, salt])


def _student_t_polar(rng: np.random.Generator, n: int, nu: float) -> np.ndarray:
    """n Student-t(nu) variates in fp32 by Bailey's polar method (Bailey 1994,
    Math. Comp. 62): (U, V) uniform on the square (-1, 1)^2 kept when
    W = U^2 + V^2 < 1, then T = U * sqrt(nu * (W^(-2/nu) - 1) / W)."""
    out = np.empty(n, np.float32)
    got = 0
    while got < n:
        m = int((n - got) * 1.3) + 1024
        u = rng.random(m, dtype=np.float32) * np.float32(2.0) - np.float32(1.0)
        v = rng.random(m, dtype=np.float32) * np.float32(2.0) - np.float32(1.0)
        wsq = u * u + v * v
        keep = (wsq < 1.0) & (wsq > 0.0)
        u, wsq = u[keep], wsq[keep]
        t = u * np.sqrt(np.float32(nu) * (np.power(wsq, np.float32(-2.0 / nu)) - np.float32(1.0)) / wsq)
        k = min(t.size, n - got)
        out[got:got + k] = t[:k]
        got += k
    return out


def grad_f32(w: Workload, param_id: int) -> np.ndarray:
    """fp32 gradient of one parameter, shape (rows, cols) (tail tensors: (numel,))."""
    p = w.params[param_id]
    shape = (p.rows, p.cols) if p.kind == KIND_MATRIX else (p.numel,)
    if param_id in w.zero_params:
        return np.zeros(shape, np.float32)
    rng = _rng(w, param_id)
    if p.kind == KIND_TAIL:
        return (rng.standard_normal(shape, dtype=np.float32) * np.float32(w.tail_scale))
    if w.grad_dist == "normal":
        x = rng.standard_normal(shape, dtype=np.float32)
    elif w.grad_dist == "student_t3":
        x = _student_t_polar(rng, p.numel, 3.0).reshape(shape)
    else:
        raise ValueError(w.grad_dist)
    return x * np.float32(w.grad_scale)


def tail_param_f32(w: Workload, param_id: int) -> np.ndarray:
    p = w.params[param_id]
    return _rng(w, param_id, 1).standard_normal((p.numel,), dtype=np.float32) * np.float32(w.tail_scale)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (round to nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def grad_storage(w: Workload, param_id: int) -> np.ndarray:
    """The gradient exactly as stored in the flat buffer: fp32 values or bf16 bits."""
    g = grad_f32(w, param_id)
    return g if w.grad_dtype == "f32" else f32_to_bf16_bits(g)


def ragged_params(seed: int, n: int, max_dim: int = 640) -> List[Tuple[int, int, int]]:
    """A seeded random layout of matrices and tail tensors with ragged sizes
    (dimensions that are not multiples of any tile), for planner fuzzing and
    ragged-tail parity cases."""
    rng = np.random.default_rng([seed, 77])
    out = []
    for _ in range(n):
        if rng.random() < 0.7:
            out.append((int(rng.integers(1, max_dim)), int(rng.integers(1, max_dim)), KIND_MATRIX))
        else:
            out.append((int(rng.integers(1, 5000)), 1, KIND_TAIL))
    return out


def _gen_one(args):
    name, pid = args
    return pid, grad_storage(get(name), pid)


def owner_grad_buffer(w: Workload, shards, numel: int, workers: Optional[int] = None) -> np.ndarray:
    """Flat gradient buffer of one rank as stored (bf16 bits or fp32), each shard
    (objects with param_id, offset, rows, cols) filled with its seeded gradient;
    padding is zero.  Large owner sets are generated per matrix in a
    spawn-started process pool (spawned workers inherit no CUDA state, so the
    call is safe before or after CUDA work in this process)."""
    dtype = np.uint16 if w.grad_dtype == "bf16" else np.float32
    buf = np.zeros(numel, dtype)
    jobs = [(w.name, s.param_id) for s in shards]
    by_id = {s.param_id: s for s in shards}
    n = workers if workers is not None else max(1, min(len(jobs), os.cpu_count() or 2, 16))
    if n > 1 and sum(s.rows * s.cols for s in shards) > 8_000_000:
        with mp.get_context("spawn").Pool(n) as pool:
            results = pool.imap_unordered(_gen_one, jobs)
            for pid, g in results:
                s = by_id[pid]
                buf[s.offset:s.offset + s.rows * s.cols] = g.reshape(-1)
    else:
        for j in jobs:
            pid, g = _gen_one(j)
            s = by_id[pid]
            buf[s.offset:s.offset + s.rows * s.cols] = g.reshape(-1)
    return buf
