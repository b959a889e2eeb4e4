"""Owner-segment reduce and owner-shard resharding (oracle).

MatrixFSDP: Communication-Free Matrix Optimizers Under ZeRO-3 Parameter
Sharding -- Abstract: the ordinary backward reduction lands each matrix's full
gradient on its owner (an uneven reduce-scatter over owner segments), made
deterministic by owner-segment collectives; owner-shard checkpoint resharding
moves owner-shaped shards between layouts.  FAQ (docshare page): owner
segments replace equal-size shard assumptions.

Readings (the pages give no formulas):
  * model layout: the unsharded flat buffer a rank's local gradient lives in
    is the parameters in declaration order, each offset rounded up to
    align_elems;
  * reduce: an owner's segment is the sum over the data-parallel ranks'
    local gradients of that parameter's elements, taken in rank order;
  * resharding: every parameter's segment moves from its owner and offset under
    the old plan to its owner and offset under the new plan, unchanged.
Values are float64 sums of the exact stored values.
"""
from __future__ import annotations

from typing import Dict, List, Sequence, Tuple

import numpy as np


def model_layout_ref(params: Sequence[Tuple[int, int, int]], align_elems: int) -> Tuple[List[int], int]:
    """Offsets of every parameter (declaration order) in the unsharded flat
    buffer, and its extent (end rounded up to align_elems)."""
    off, offsets = 0, []
    for r, c, _ in params:
        off = (off + align_elems - 1) // align_elems * align_elems
        offsets.append(off)
        off += r * c
    total = (off + align_elems - 1) // align_elems * align_elems
    return offsets, total


def placement_segments_ref(src: Sequence[dict], dst: Sequence[dict], dst_owner: int) -> List[dict]:
    """For every parameter that `dst` places on dst_owner: where it sits in `src`
    (owner = source buffer index, offset) and where it goes (offset).  Entries
    carry param_id, owner, offset, numel."""
    by_id: Dict[int, dict] = {e["param_id"]: e for e in src}
    out = []
    for e in sorted((e for e in dst if e["owner"] == dst_owner), key=lambda e: e["offset"]):
        s = by_id[e["param_id"]]
        assert s["numel"] == e["numel"]
        out.append(dict(src_index=s["owner"], src_offset=s["offset"], dst_offset=e["offset"], numel=e["numel"]))
    return out


def segment_reduce_ref(srcs: Sequence[np.ndarray], segs: Sequence[dict], dst_numel: int) -> np.ndarray:
    """dst[dst_offset + i] = sum over k of srcs[k][src_offset + i] (float64;
    elements outside every segment are NaN)."""
    out = np.full(dst_numel, np.nan)
    for g in segs:
        acc = np.zeros(g["numel"])
        for s in srcs:
            acc = acc + np.asarray(s[g["src_offset"]:g["src_offset"] + g["numel"]], np.float64)
        out[g["dst_offset"]:g["dst_offset"] + g["numel"]] = acc
    return out


def segment_gather_ref(srcs: Sequence[np.ndarray], segs: Sequence[dict], dst_numel: int) -> np.ndarray:
    """dst[dst_offset + i] = srcs[src_index][src_offset + i] (float64)."""
    out = np.full(dst_numel, np.nan)
    for g in segs:
        s = np.asarray(srcs[g["src_index"]], np.float64)
        out[g["dst_offset"]:g["dst_offset"] + g["numel"]] = s[g["src_offset"]:g["src_offset"] + g["numel"]]
    return out
