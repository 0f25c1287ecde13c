"""Top-k softmax router and stable route map (oracle; test use only).

Router: the workloads draw router logits and take "softmax then top-k
renormalised"; routing ids and route weights are the custom-op outputs that
flashinfer PR #69 "b12x fused MoE: TrellisMX (procedural NPK) source format
with an in-tree P8 runtime" lists among its routing changes (commit list:
selected logits, IDs and route weights).

Route map: per-expert counts, an exclusive scan of the counts with every
expert's segment padded to the block size, and a permutation that lists each
expert's routes (sparkinfer PR #90 "moe: integrate EXL3 Trellis into the fused
W4A16 API", review of route_pack.py: route count kernel, prefix-from-counts
kernel with BLOCK_SIZE, expert_offsets and packed_route_count; b12x PR #433
"Share trellis preparation across native and EXL3 containers", review of
route_pack.py: a stable, token-major route order).

Readings where the pages leave the step open:
  * Router ties between equal logits go to the lower expert id; the k selected
    experts are listed by descending logit. The weights are
    exp(l_j - max) / sum over the k selected of exp(l - max), which equals a
    full softmax renormalised over the selected k.
  * Route r = t*k + j is token t's j-th selection. Within an expert, routes are
    listed in ascending r (stable, token-major). Padding slots hold -1.
"""
from __future__ import annotations

import numpy as np


def route_topk_softmax(logits: np.ndarray, k: int):
    """logits float32 [T, E] -> (ids int32 [T, k], weights float64 [T, k])."""
    lg = np.asarray(logits, dtype=np.float32)
    T, E = lg.shape
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    for t in range(T):
        # lexicographic order: larger logit first, then lower expert id
        order = sorted(range(E), key=lambda e: (-float(lg[t, e]), e))
        sel = order[:k]
        ids[t] = sel
        v = lg[t, sel].astype(np.float64)
        ex = np.exp(v - v.max())
        w[t] = ex / ex.sum()
    return ids, w


def route_map(ids: np.ndarray, E: int, block: int):
    """Stable route map of ids [T, k] with expert segments padded to ``block``.

    Returns dict with counts int32 [E], offsets int32 [E+1] (padded exclusive
    scan; offsets[E] = padded total), route_of_slot int32 [offsets[E]] (-1 for
    padding) and slot_of_route int32 [T*k].
    """
    flat = np.asarray(ids, dtype=np.int64).reshape(-1)
    R = flat.size
    counts = np.zeros(E, dtype=np.int64)
    for e in flat:
        counts[e] += 1
    padded = ((counts + block - 1) // block) * block
    offsets = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + padded[e]
    route_of_slot = np.full(int(offsets[E]), -1, dtype=np.int64)
    slot_of_route = np.empty(R, dtype=np.int64)
    fill = offsets[:E].copy()
    for r in range(R):                  # ascending route id: stable, token-major
        e = flat[r]
        route_of_slot[fill[e]] = r
        slot_of_route[r] = fill[e]
        fill[e] += 1
    return {
        "counts": counts.astype(np.int32),
        "offsets": offsets.astype(np.int32),
        "route_of_slot": route_of_slot.astype(np.int32),
        "slot_of_route": slot_of_route.astype(np.int32),
    }
