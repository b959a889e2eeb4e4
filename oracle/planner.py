"""Balance-aware owner planner and MatrixShard layout (oracle).

MatrixFSDP: Communication-Free Matrix Optimizers Under ZeRO-3 Parameter
Sharding -- Abstract: for each 2D weight one data-parallel rank owns the whole
matrix and the other ranks hold empty shards; non-matrix tensors are packed
into tail owners; the runtime carries the plan in MatrixShard metadata and
assigns owners with a balance-aware planner.  FAQ (docshare page): the metadata
carries the owner plan through optimizer routing; the collectives are
deterministic owner segments, not equal-size slices.

The pages give neither the planner's algorithm nor its cost model.  Readings
taken here (all integer, so the result is exact):
  * cost of a matrix = dense Newton-Schulz FLOPs T*(4 s^2 l + 2 s^3),
    s = min(rows, cols), l = max(rows, cols);
  * matrix pass = longest-processing-time-first: matrices sorted by
    (cost descending, param id ascending), each given to the rank with the
    smallest (load, rank id);
  * tail pass: tail tensors sorted by (numel descending, param id ascending),
    each given to the rank with the smallest (tail load, matrix load, rank id),
    i.e. toward the ranks with the least Newton-Schulz work;
  * per rank, segments laid out in ascending param id, each offset rounded up
    to align_elems; matrix and tail buffers are separate; a buffer's extent is
    its end rounded up to align_elems;
  * transposed = rows > cols.
"""
from __future__ import annotations

from typing import Dict, List, Sequence, Tuple


def _roundup(x: int, a: int) -> int:
    return (x + a - 1) // a * a


def ns_cost(rows: int, cols: int, ns_steps: int) -> int:
    s, l = min(rows, cols), max(rows, cols)
    return ns_steps * (4 * s * s * l + 2 * s ** 3)


def plan_owners_ref(params: Sequence[Tuple[int, int, int]], world: int, ns_steps: int,
                    align_elems: int = 128) -> Dict[str, object]:
    """params: (rows, cols, kind) per parameter, kind 0 = matrix, 1 = tail.

    Returns a dict with
      matrix_shards: list of dicts (param_id, owner, offset, rows, cols,
                     transposed, cost), ordered by (owner, param_id);
      tail_shards:   list of dicts (param_id, owner, offset, numel), same order;
      rank_matrix_elems, rank_tail_elems: per-rank buffer extents;
      rank_cost: per-rank total matrix cost;
      rank_tail_numel: per-rank total tail elements (without padding).
    """
    if world < 1 or align_elems < 1 or ns_steps < 0:
        raise ValueError("bad planner arguments")
    mats = [i for i, p in enumerate(params) if p[2] == 0]
    tails = [i for i, p in enumerate(params) if p[2] == 1]
    cost = {i: ns_cost(params[i][0], params[i][1], ns_steps) for i in mats}

    load = [0] * world
    owner: Dict[int, int] = {}
    for i in sorted(mats, key=lambda i: (-cost[i], i)):
        r = min(range(world), key=lambda r: (load[r], r))
        owner[i] = r
        load[r] += cost[i]

    tload = [0] * world
    towner: Dict[int, int] = {}
    for i in sorted(tails, key=lambda i: (-(params[i][0] * params[i][1]), i)):
        r = min(range(world), key=lambda r: (tload[r], load[r], r))
        towner[i] = r
        tload[r] += params[i][0] * params[i][1]

    mshards: List[dict] = []
    tshards: List[dict] = []
    mext = [0] * world
    text = [0] * world
    for r in range(world):
        off = 0
        for i in sorted(k for k in mats if owner[k] == r):
            off = _roundup(off, align_elems)
            rows, cols = params[i][0], params[i][1]
            mshards.append(dict(param_id=i, owner=r, offset=off, rows=rows, cols=cols,
                                transposed=int(rows > cols), cost=cost[i]))
            off += rows * cols
        mext[r] = _roundup(off, align_elems)
        off = 0
        for i in sorted(k for k in tails if towner[k] == r):
            off = _roundup(off, align_elems)
            n = params[i][0] * params[i][1]
            tshards.append(dict(param_id=i, owner=r, offset=off, numel=n))
            off += n
        text[r] = _roundup(off, align_elems)
    return dict(matrix_shards=mshards, tail_shards=tshards, rank_matrix_elems=mext,
                rank_tail_elems=text, rank_cost=load, rank_tail_numel=tload)


def heaviest_rank_ref(plan: Dict[str, object]) -> int:
    """The rank a benchmark of one owner set uses: largest matrix cost, then the
    smallest tail, then the lowest rank id (reading; the pages name no rank)."""
    cost = plan["rank_cost"]
    tail = plan["rank_tail_numel"]
    return min(range(len(cost)), key=lambda r: (-cost[r], tail[r], r))
