"""Pins for the EAGLE-2 tree post-processing in the oracle (rerank by path
value, keep m, flatten by depth, ancestor-only attention mask).

- The page's worked example (golden fixture): the values it prints, its
  order of all eleven nodes, the eight kept nodes, the flattened order and
  the relative positions, and masks that match the three branches it lists.
- The kept set equals a best-first expansion from the root (a different
  algorithm: a frontier priority queue), on random trees.
- Values equal the fp64 product of the confidences along the path within
  fp32 rounding; masks equal the ancestor relation found by walking parents.
- Ties of value go to the shallower node, then the lower id; m >= N keeps
  everything, m = 1 keeps the root; malformed inputs are reported.
"""
import heapq

import numpy as np
import pytest

import oracle
from tests.conftest import read_table


def _golden():
    meta, rows = read_table("eagle2_candidates.txt")
    names = [r[1] for r in rows]
    parents = np.array([int(r[2]) for r in rows], np.int32)
    conf = np.array([float(r[3]) for r in rows], np.float32)
    printed_v = np.array([float(r[4]) for r in rows])
    return meta, names, parents, conf, printed_v


def test_worked_example():
    meta, names, parents, conf, printed_v = _golden()
    N = len(names)
    # all eleven in the page's order: m = N keeps everything, flattened;
    # the rank order is read off the values
    full = oracle.tree_rerank(parents[None], conf[None], N)
    v = np.empty(N)
    v[full["sel_nodes"][0]] = full["sel_value"][0]
    np.testing.assert_allclose(v, printed_v, atol=5e-7)
    order = sorted(range(N), key=lambda i: (-v[i], i))
    assert [names[i] for i in order] == meta["rerank"].split()
    keep = int(meta["keep"])
    o = oracle.tree_rerank(parents[None], conf[None], keep, node_tok=np.arange(N, dtype=np.int32)[None])
    assert o["status"][0] == 0 and o["n_sel"][0] == keep
    assert [names[i] for i in o["sel_nodes"][0]] == meta["flatten"].split()
    assert o["sel_depth"][0].tolist() == [int(x) for x in meta["positions"].split()]
    assert o["sel_tok"][0].tolist() == o["sel_nodes"][0].tolist()
    flat = meta["flatten"].split()
    # the three branches the page lists, each leaf attending to its branch
    for branch in (["I", "do", "it", "now"], ["I", "do", "this"], ["I", "make", "a", "plan"]):
        row = o["mask"][0, flat.index(branch[-1])]
        assert sorted(np.flatnonzero(row).tolist()) == sorted(flat.index(w) for w in branch)
    # flattened parents point at the parent's flattened slot
    for j, u in enumerate(o["sel_nodes"][0]):
        pj = o["sel_parents"][0, j]
        assert (pj == -1) if u == 0 else (o["sel_nodes"][0, pj] == parents[u])


def _random_tree(rng, N, max_children=4, tie=False):
    parents = np.full(N, -1, np.int32)
    kids = np.zeros(N, np.int32)
    for i in range(1, N):
        cand = [j for j in range(i) if kids[j] < max_children]
        parents[i] = rng.choice(cand)
        kids[parents[i]] += 1
    conf = rng.random(N).astype(np.float32)
    if tie:  # many equal values: confidences from a tiny set, some exactly 1
        conf = rng.choice(np.array([1.0, 0.5, 0.25], np.float32), N)
    conf[0] = 1.0
    return parents, conf


def _best_first(parents, conf, m):
    """Best-first expansion from the root: repeatedly take the frontier node
    of largest value (ties: shallower, then lower id)."""
    N = len(parents)
    kids = [[] for _ in range(N)]
    for i in range(1, N):
        kids[parents[i]].append(i)
    val = {0: np.float32(1.0)}
    depth = {0: 0}
    heap, kept = [(-1.0, 0, 0)], []
    while heap and len(kept) < m:
        _, d, u = heapq.heappop(heap)
        kept.append(u)
        for c in kids[u]:
            val[c] = np.float32(val[u] * conf[c])
            depth[c] = d + 1
            heapq.heappush(heap, (-float(val[c]), d + 1, c))
    return kept, val, depth


@pytest.mark.parametrize("seed", range(40))
def test_kept_set_is_best_first_expansion(seed):
    rng = np.random.default_rng(seed)
    N = int(rng.integers(2, 40))
    parents, conf = _random_tree(rng, N, tie=seed % 3 == 0)
    m = int(rng.integers(1, N + 2))
    o = oracle.tree_rerank(parents[None], conf[None], m, node_tok=(np.arange(N) * 7 + 3).astype(np.int32)[None])
    kept, val, depth = _best_first(parents, conf, m)
    n = min(m, N)
    assert o["n_sel"][0] == n and o["status"][0] == 0
    sel = o["sel_nodes"][0, :n].tolist()
    assert sorted(sel) == sorted(kept)
    assert sel == sorted(kept, key=lambda u: (depth[u], u))          # flattened: depth, then id
    assert o["sel_depth"][0, :n].tolist() == [depth[u] for u in sel]
    assert (o["sel_nodes"][0, n:] == -1).all() and (o["sel_depth"][0, n:] == -1).all()
    assert o["sel_tok"][0, :n].tolist() == [u * 7 + 3 for u in sel]
    for j, u in enumerate(sel):
        # value: the fp64 product along the path, within fp32 rounding
        prod, a = 1.0, u
        anc = set()
        while a != 0:
            prod *= float(conf[a])
            anc.add(a)
            a = parents[a]
        anc.add(0)
        assert abs(o["sel_value"][0, j] - prod) <= 1e-6 * max(prod, 1e-30) + 1e-37
        # mask row: exactly the ancestors (and itself)
        assert set(np.flatnonzero(o["mask"][0, j]).tolist()) == {sel.index(x) for x in anc}
    assert not o["mask"][0, n:].any() and not o["mask"][0, :, n:].any()


def test_ties_prefer_shallow_then_low_id():
    # a chain 0-1-2-3 of confidence 1 beside a sibling 4 of the root with confidence 1
    parents = np.array([[-1, 0, 1, 2, 0]], np.int32)
    conf = np.ones((1, 5), np.float32)
    o = oracle.tree_rerank(parents, conf, 3)
    assert o["sel_nodes"][0].tolist() == [0, 1, 4]      # depths 0, 1, 1 before depth 2
    o = oracle.tree_rerank(parents, conf, 1)
    assert o["sel_nodes"][0].tolist() == [0]


def test_bad_inputs_reported():
    good = np.array([-1, 0, 0, 1], np.int32)
    conf = np.array([1.0, 0.5, 0.5, 0.5], np.float32)
    cases = [(np.array([0, 0, 0, 1], np.int32), conf),            # root has a parent
             (np.array([-1, 0, 3, 1], np.int32), conf),           # parent not earlier
             (good, np.array([1.0, 1.5, 0.5, 0.5], np.float32)),  # confidence above 1
             (good, np.array([1.0, 0.5, np.nan, 0.5], np.float32)),
             (good, np.array([1.0, -0.1, 0.5, 0.5], np.float32))]
    P = np.stack([c[0] for c in cases])
    C = np.stack([c[1] for c in cases])
    o = oracle.tree_rerank(P, C, 3)
    assert (o["status"] == 2).all() and (o["n_sel"] == 0).all() and (o["sel_nodes"] == -1).all()
    # depth beyond max_depth
    o = oracle.tree_rerank(good[None], conf[None], 3, max_depth=1)
    assert o["status"][0] == 2
