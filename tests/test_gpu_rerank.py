"""GPU parity of spec_tree_rerank (EAGLE-2 tree post-processing) against the
oracle, bit for bit: kept nodes and their flattened order, flattened
parents, depths, fp32 values, tokens, the attention mask, n_sel and status.
The values decide the ranking, so both sides compute them in fp32 from the
root down; they must agree exactly.

Also: the page's worked example, ties and zero confidences, malformed
inputs, every size up to SPEC_MAX_NODES, and the pipeline the post-processing
feeds -- rerank, then spec_verify_tree on the flattened tree, equal to the
oracle doing the same.
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_02_gb300 import api, workloads
from tests.conftest import read_table
from tests.parity import check_tree, host, poison_like, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _gpu(parents, conf, m, max_depth=64, node_tok=None):
    args = dict(max_depth=max_depth, node_tok=None if node_tok is None else to_dev(node_tok))
    o = api.spec_tree_rerank(to_dev(parents), to_dev(conf), m, **args)
    for k, v in o.items():            # a second call into poisoned outputs
        if v is not None:
            v.fill_(0x5A if v.dtype == torch.uint8 else -7)
    o = api.spec_tree_rerank(to_dev(parents), to_dev(conf), m, out=o, **args)
    torch.cuda.synchronize()
    return {k: (None if v is None else v.cpu().numpy()) for k, v in o.items()}


def _same(g, r):
    for k in ("sel_nodes", "sel_parents", "sel_depth", "sel_tok", "n_sel", "status"):
        if r.get(k) is not None:
            np.testing.assert_array_equal(g[k], r[k], err_msg=k)
    np.testing.assert_array_equal(g["sel_value"].view(np.uint32), r["sel_value"].view(np.uint32))
    np.testing.assert_array_equal(g["mask"], r["mask"])


def test_worked_example():
    meta, rows = read_table("eagle2_candidates.txt")
    names = [r[1] for r in rows]
    parents = np.array([[int(r[2]) for r in rows]], np.int32)
    conf = np.array([[float(r[3]) for r in rows]], np.float32)
    tok = np.arange(len(rows), dtype=np.int32)[None]
    g = _gpu(parents, conf, int(meta["keep"]), node_tok=tok)
    _same(g, oracle.tree_rerank(parents, conf, int(meta["keep"]), node_tok=tok))
    assert [names[i] for i in g["sel_nodes"][0]] == meta["flatten"].split()
    assert g["sel_depth"][0].tolist() == [int(x) for x in meta["positions"].split()]


def _random_trees(rng, B, N, ties=False):
    parents = np.full((B, N), -1, np.int32)
    for b in range(B):
        for i in range(1, N):
            # mostly recent parents (deep trees) or any earlier node (bushy)
            parents[b, i] = rng.integers(max(0, i - 4), i) if b % 2 else rng.integers(0, i)
    conf = rng.random((B, N)).astype(np.float32)
    if ties:
        conf = rng.choice(np.array([1.0, 0.5, 0.0, -0.0], np.float32), (B, N))
    conf[:, 0] = 1.0
    return parents, conf


@pytest.mark.parametrize("seed,B,N,m,ties", [(1, 8, 11, 8, False), (2, 16, 60, 60, False), (3, 16, 511, 60, False),
                                             (4, 8, 1000, 90, True), (5, 3, 4096, 64, False), (6, 4, 4096, 4096, True),
                                             (7, 5, 1, 3, False), (8, 6, 37, 1, True), (9, 4, 129, 200, False)])
def test_parity_random(seed, B, N, m, ties):
    rng = np.random.default_rng(seed)
    parents, conf = _random_trees(rng, B, N, ties)
    depth_cap = 64
    # keep the trees within the depth cap: re-parent nodes whose depth would pass it
    depth = np.zeros((B, N), np.int32)
    for b in range(B):
        for i in range(1, N):
            if depth[b, parents[b, i]] + 1 > depth_cap:
                parents[b, i] = 0
            depth[b, i] = depth[b, parents[b, i]] + 1
    tok = rng.integers(0, 50000, (B, N)).astype(np.int32)
    g = _gpu(parents, conf, m, depth_cap, node_tok=tok)
    r = oracle.tree_rerank(parents, conf, m, depth_cap, node_tok=tok)
    _same(g, r)
    assert (r["status"] == 0).all()


def test_workload_shape():
    p = workloads.eagle2_candidates()
    g = _gpu(p["parents"], p["conf"], 60, node_tok=p["node_tok"])
    r = oracle.tree_rerank(p["parents"], p["conf"], 60, node_tok=p["node_tok"])
    _same(g, r)
    assert (g["n_sel"] == 60).all() and g["sel_depth"].max() >= 3


def test_bad_inputs():
    good = np.array([-1, 0, 0, 1, 3], np.int32)
    c = np.array([1.0, 0.5, 0.5, 0.5, 0.5], np.float32)
    P = np.stack([np.array([0, 0, 0, 1, 3], np.int32), np.array([-1, 0, 4, 1, 3], np.int32), good, good, good, good])
    C = np.stack([c, c, np.array([1, 1.5, .5, .5, .5], np.float32), np.array([1, .5, np.nan, .5, .5], np.float32), c, c])
    g = _gpu(P, C, 4, max_depth=2)   # the last two: depth 3 beyond max_depth 2
    r = oracle.tree_rerank(P, C, 4, max_depth=2)
    _same(g, r)
    assert (g["status"] == 2).all() and (g["n_sel"] == 0).all()
    g = _gpu(P[2:3] * 0 + good, C[4:5], 4, max_depth=3)
    assert g["status"][0] == 0 and g["n_sel"][0] == 4


def test_rerank_then_verify_tree():
    """The flattened output is a tree spec_verify_tree accepts; verifying it on
    the GPU equals the oracle verifying the oracle's flattened tree."""
    B, m, V = 6, 24, 4096
    cand = workloads.eagle2_candidates(workloads.SEED_BASE + 16, B=B, depth=4, expand=3, branch=4, V=V)
    g = _gpu(cand["parents"], cand["conf"], m, node_tok=cand["node_tok"])
    r = oracle.tree_rerank(cand["parents"], cand["conf"], m, node_tok=cand["node_tok"])
    _same(g, r)
    # logits for the kept nodes in their flattened order
    rng = np.random.default_rng(7)
    t = rng.normal(0, 2, (B, m, V)).astype(np.float32)
    d = (t + rng.normal(0, 0.7, (B, m, V))).astype(np.float32)
    tok = np.where(g["sel_tok"] >= 0, g["sel_tok"] % V, 0).astype(np.int32)
    u = rng.random((B, m + 1), dtype=np.float32)
    prob = dict(target=t, draft_logits=d, parents=g["sel_parents"], node_tok=tok, uniforms=u, T=1.0, depth=4)
    out = api.spec_verify_tree(to_dev(t), to_dev(d), to_dev(g["sel_parents"]), to_dev(tok), to_dev(u), 1.0, 4)
    torch.cuda.synchronize()
    orc = oracle.verify_tree(t, d, r["sel_parents"], tok, u, 1.0, 4)
    check_tree(prob, host(out), orc)
    assert (host(out)["status"] == 0).all()
