"""Pins for the oracle's router and route map (CPU only)."""
import itertools

import numpy as np
import pytest

from oracle import route
from trellis_quantized_moe_route_gb300 import synth


def test_router_picks_largest_and_breaks_ties_by_id():
    lg = np.array([[0.5, 2.0, 2.0, -1.0, 2.0],
                   [1.0, 1.0, 1.0, 1.0, 1.0]], dtype=np.float32)
    ids, w = route.route_topk_softmax(lg, 3)
    assert ids.tolist() == [[1, 2, 4], [0, 1, 2]]
    assert np.allclose(w, 1.0 / 3.0)


def test_router_matches_full_softmax_renormalised():
    cfg = synth.CONFIGS["tiny"]
    _, lg = synth.make_tokens(cfg)
    ids, w = route.route_topk_softmax(lg, cfg.topk)
    for t in range(lg.shape[0]):
        p = np.exp(lg[t].astype(np.float64) - lg[t].max())
        p /= p.sum()
        top = np.argsort(-p, kind="stable")[:cfg.topk]
        assert sorted(top.tolist()) == sorted(ids[t].tolist())
        assert np.allclose(w[t], p[ids[t]] / p[ids[t]].sum(), rtol=1e-12)
        assert abs(w[t].sum() - 1.0) < 1e-12
        assert np.all(np.diff(lg[t, ids[t]]) <= 0)


@pytest.mark.parametrize("T,E,k,block", [(4, 8, 2, 1), (3, 5, 2, 4), (1, 8, 8, 8), (4, 4, 4, 3), (0, 4, 2, 4)])
def test_route_map_brute_force(T, E, k, block):
    ids = synth.random_ids(7 + T, T, E, k)
    m = route.route_map(ids, E, block)
    flat = ids.reshape(-1)
    # counts from a histogram, offsets from padding, order from a stable sort
    assert m["counts"].tolist() == np.bincount(flat, minlength=E).tolist()
    pad = -(-m["counts"] // block) * block
    assert m["offsets"].tolist() == [0] + np.cumsum(pad).tolist()
    order = np.argsort(flat, kind="stable")
    listed = [r for r in m["route_of_slot"].tolist() if r >= 0]
    assert listed == order.tolist()
    for r in range(flat.size):
        s = int(m["slot_of_route"][r])
        assert m["route_of_slot"][s] == r
        e = flat[r]
        assert m["offsets"][e] <= s < m["offsets"][e] + m["counts"][e]
    assert int((m["route_of_slot"] < 0).sum()) == int(pad.sum() - m["counts"].sum())


def test_route_map_exhaustive_tiny():
    """All id patterns of T=2, k=2 over E=3 (distinct per token)."""
    pairs = [p for p in itertools.permutations(range(3), 2)]
    for a, b in itertools.product(pairs, pairs):
        ids = np.array([a, b], dtype=np.int32)
        m = route.route_map(ids, 3, 2)
        seen = {}
        for s, r in enumerate(m["route_of_slot"].tolist()):
            if r < 0:
                continue
            e = int(ids.reshape(-1)[r])
            seen.setdefault(e, []).append(r)
        for e, rs in seen.items():
            assert rs == sorted(rs)
