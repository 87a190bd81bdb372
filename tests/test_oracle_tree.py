"""Pins for tree verification.

- A tree that is a single chain must verify exactly like the chain verifier
  (both modes), uniform for uniform.
- Greedy walks over the EAGLE-2 worked tree (golden fixture) follow the
  target's choices along the three branches the page lists.
- Losslessness: with two siblings drawn i.i.d. from q, the first emitted
  token is distributed exactly as p.  Each acceptance threshold and the final
  residual draw are measured by scanning one uniform over a 2^16 grid; the
  composition over both sibling tokens must equal p to ~1e-4, and the
  planted mistake (no residual update between siblings) must not.  With
  three siblings drawn WITHOUT replacement, the rule that also removes each
  rejected token from q emits exactly p, and the i.i.d. rule does not.
- Malformed trees and out-of-range tokens are reported per request.
"""
import numpy as np
import pytest

import oracle
from speculative_decoding_verification_02_gb300 import workloads
from tests.conftest import read_table

M = 1 << 16
U_REJECT = np.float32(1.0 - 2.0 ** -24)


def _softmax64(x):
    z = np.asarray(x, np.float64)
    e = np.exp(z - z.max())
    return e / e.sum()


@pytest.mark.parametrize("T", [1.0, 0.7, 0.0])
def test_chain_shaped_tree_equals_chain(T):
    prob = workloads.chain_problem(11, B=24, k=5, V=96, dtype="bf16", T=T if T > 0 else 1.0,
                                   target_std=1.5, noise_std=0.6)
    B, k = prob["B"], prob["k"]
    N = k + 1
    parents = np.tile(np.arange(-1, N - 1, dtype=np.int32), (B, 1))
    node_tok = np.concatenate([np.zeros((B, 1), np.int32), prob["draft"]], 1)
    dl = np.concatenate([prob["draft_logits"], prob["draft_logits"][:, :1]], 1)  # leaf row unused
    u_tree = np.concatenate([np.zeros((B, 1), np.float32), prob["uniforms"]], 1)  # u[c] <-> chain u[c-1]
    tree = oracle.verify_tree(prob["target"], dl, parents, node_tok, u_tree, T, max_depth=k)
    if T > 0:
        chain = oracle.verify_sample(prob["target"], prob["draft_logits"], prob["draft"],
                                     prob["uniforms"], T)
    else:
        chain = oracle.verify_greedy(prob["target"], prob["draft"])
    np.testing.assert_array_equal(tree["accepted_len"], chain["accepted"])
    np.testing.assert_array_equal(tree["n_emit"], chain["n_emit"])
    np.testing.assert_array_equal(tree["out_tokens"], chain["out_tokens"])
    for b in range(B):
        m = tree["accepted_len"][b]
        assert list(tree["path_nodes"][b, :m + 1]) == list(range(m + 1))
    if T > 0:
        assert 0 < tree["accepted_len"].mean() < k      # both outcomes occur


WORDS = ["I", "do", "make", "it", "this", "a", "now", "plan", "later", "list", "some", ".", "!", "?"]


def _eagle_tree():
    _, rows = read_table("eagle2_tree.txt")
    ids = {w: i for i, w in enumerate(WORDS)}
    parents = np.array([int(r[2]) for r in rows], np.int32)
    tok = np.array([ids[r[1]] for r in rows], np.int32)
    assert [r[1] for r in rows] == ["I", "do", "make", "it", "this", "a", "now", "plan"]
    assert [int(r[3]) for r in rows] == [0, 1, 1, 2, 2, 2, 3, 3]
    return parents, tok, ids


@pytest.mark.parametrize("branch,expect_tokens,expect_path", [
    (["do", "it", "now", "."], ["do", "it", "now", "."], [0, 1, 3, 6]),
    (["make", "a", "plan", "!"], ["make", "a", "plan", "!"], [0, 2, 5, 7]),
    (["do", "this", "?"], ["do", "this", "?"], [0, 1, 4]),
    (["later"], ["later"], [0]),
    (["do", "some"], ["do", "some"], [0, 1]),
])
def test_greedy_walk_on_worked_tree(branch, expect_tokens, expect_path):
    parents, tok, ids = _eagle_tree()
    N, V = len(parents), len(WORDS)
    # the target's choice after each node on the branch; other rows prefer "."
    target = np.zeros((1, N, V), np.float32)
    target[0, :, ids["."]] = 1.0
    node = 0
    for w in branch:
        target[0, node, :] = 0.0
        target[0, node, ids[w]] = 3.0
        nxt = [c for c in range(N) if parents[c] == node and tok[c] == ids[w]]
        if not nxt:
            break
        node = nxt[0]
    out = oracle.verify_tree(target, None, parents[None], tok[None],
                             np.zeros((1, N + 1), np.float32), 0.0, max_depth=3)
    n = out["n_emit"][0]
    assert [WORDS[t] for t in out["out_tokens"][0, :n]] == expect_tokens
    assert list(out["path_nodes"][0, :out["accepted_len"][0] + 1]) == expect_path
    assert out["accepted_len"][0] == len(expect_path) - 1


def _tree_first_token_law(lp, lq, variant, n=2, replace=True):
    """Root with n sibling leaves drawn from q (i.i.d., or without replacement);
    the first emitted token's law, threshold by threshold: sibling j's
    acceptance rate is measured by scanning u_j over a 2^16 grid with the
    earlier siblings' uniforms set to reject, and the final draw by scanning
    u_final with every sibling rejected."""
    import itertools
    V = lp.size
    N = n + 1
    q = _softmax64(lq)
    grid = (np.arange(M, dtype=np.float64) / M).astype(np.float32)
    target = np.broadcast_to(np.stack([lp] * N), (M, N, V))
    dl = np.broadcast_to(np.stack([lq] * N), (M, N, V))
    parents = np.broadcast_to(np.array([-1] + [0] * n, np.int32), (M, N))
    law = np.zeros(V)
    half = np.full(M, 0.5, np.float32)
    rej = np.full(M, U_REJECT, np.float32)

    def run(xs, us):
        tok = np.broadcast_to(np.array([0] + list(xs), np.int32), (M, N))
        u = np.stack([np.zeros(M, np.float32)] + list(us), 1).astype(np.float32)
        return oracle.verify_tree(target, dl, parents, tok, u, 1.0, max_depth=1, variant=variant, threads=4)

    seqs = itertools.product(range(V), repeat=n) if replace else itertools.permutations(range(V), n)
    for xs in seqs:
        w, left = 1.0, 1.0
        for x in xs:                       # the drafter's draws
            w *= q[x] / left
            if not replace:
                left -= q[x]
        reach = 1.0                        # probability that siblings 1..j-1 were all rejected
        for j in range(n):
            us = [rej] * j + [grid] + [half] * (n - j - 1) + [half]
            a = (run(xs, us)["path_nodes"][:, 1] == j + 1).mean()
            law[xs[j]] += w * reach * a
            reach *= 1 - a
            if reach == 0.0:
                break
        if reach > 0.0:
            out = run(xs, [rej] * n + [grid])
            assert np.all(out["accepted_len"] == 0)
            law += w * reach * np.bincount(out["out_tokens"][:, 0], minlength=V) / M
    return law


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_sibling_walk_first_token_is_exactly_p(seed):
    rng = np.random.default_rng(40 + seed)
    V = 3
    lp = (rng.standard_normal(V) * 1.5).astype(np.float32)
    lq = (rng.standard_normal(V) * 1.5).astype(np.float32)
    p = _softmax64(lp)
    law = _tree_first_token_law(lp, lq, oracle.VARIANT_LOSSLESS)
    assert np.max(np.abs(law - p)) < 4.0 * V / M
    bad = _tree_first_token_law(lp, lq, oracle.TREE_VARIANT_NO_RESIDUAL_UPDATE)
    assert np.max(np.abs(bad - p)) > 5e-3


def test_tree_monte_carlo_second_token_follows_child_target():
    # deeper check: given the first emitted token came from accepting child c,
    # the second token is distributed as the child's own target p_c
    rng = np.random.default_rng(5)
    V, n = 5, 200_000
    lroot = (rng.standard_normal(V) * 1.2).astype(np.float32)
    lq = (rng.standard_normal(V) * 1.2).astype(np.float32)
    lchild = (rng.standard_normal(V) * 1.2).astype(np.float32)
    N = 3
    target = np.broadcast_to(np.stack([lroot, lchild, lchild]), (n, N, V))
    dl = np.broadcast_to(np.stack([lq, lq, lq]), (n, N, V))
    parents = np.broadcast_to(np.array([-1, 0, 0], np.int32), (n, N))
    q = _softmax64(lq)
    tok = np.zeros((n, N), np.int32)
    tok[:, 1:] = rng.choice(V, size=(n, 2), p=q)
    u = rng.random((n, N + 1), dtype=np.float32)
    out = oracle.verify_tree(target, dl, parents, tok, u, 1.0, max_depth=1, threads=8)
    first = out["out_tokens"][:, 0]
    p_root = _softmax64(lroot)
    np.testing.assert_allclose(np.bincount(first, minlength=V) / n, p_root, atol=5 * np.sqrt(0.25 / n))
    sel = out["accepted_len"] == 1
    second = out["out_tokens"][sel, 1]
    p_child = _softmax64(lchild)
    np.testing.assert_allclose(np.bincount(second, minlength=V) / sel.sum(), p_child,
                               atol=5 * np.sqrt(0.25 / sel.sum()))


def test_bad_trees_and_tokens_are_flagged():
    V, N = 8, 4
    target = np.zeros((5, N, V), np.float32)
    parents = np.array([[-1, 0, 0, 1],       # fine
                        [-1, 0, 2, 1],       # parent not earlier
                        [0, 0, 1, 2],        # root has a parent
                        [-1, 0, 1, 2],       # depth 3 > max_depth 2
                        [-1, 0, 0, 1]], np.int32)
    tok = np.array([[0, 1, 2, 3]] * 4 + [[0, 1, V, 3]], np.int32)
    u = np.full((5, N + 1), 0.5, np.float32)
    out = oracle.verify_tree(target, target, parents, tok, u, 1.0, max_depth=2)
    assert list(out["status"]) == [0, oracle.ST_BAD_TREE, oracle.ST_BAD_TREE, oracle.ST_BAD_TREE,
                                   oracle.ST_TOKEN_RANGE]
    assert list(out["n_emit"]) == [out["n_emit"][0], 0, 0, 0, 0]
    assert out["n_emit"][0] >= 1


def test_single_node_tree_draws_from_root_target():
    V, n = 6, 100_000
    rng = np.random.default_rng(9)
    l = (rng.standard_normal(V)).astype(np.float32)
    target = np.broadcast_to(l, (n, 1, V))
    out = oracle.verify_tree(target, target, np.full((n, 1), -1, np.int32), np.zeros((n, 1), np.int32),
                             rng.random((n, 2), dtype=np.float32), 1.0, max_depth=0, threads=8)
    assert np.all(out["n_emit"] == 1) and np.all(out["accepted_len"] == 0)
    np.testing.assert_allclose(np.bincount(out["out_tokens"][:, 0], minlength=V) / n, _softmax64(l),
                               atol=5 * np.sqrt(0.25 / n))


@pytest.mark.parametrize("seed", [0, 1])
def test_siblings_without_replacement_first_token_is_exactly_p(seed):
    """Three siblings drawn from q without replacement: the rule that removes
    each rejected sibling's token from q (and renormalises it) emits exactly
    p; the i.i.d. rule applied to such drafts does not."""
    rng = np.random.default_rng(70 + seed)
    V = 4
    lp = (rng.standard_normal(V) * 1.5).astype(np.float32)
    lq = (rng.standard_normal(V) * 1.5).astype(np.float32)
    p = _softmax64(lp)
    law = _tree_first_token_law(lp, lq, oracle.TREE_VARIANT_WITHOUT_REPLACEMENT, n=3, replace=False)
    assert np.max(np.abs(law - p)) < 6.0 * V / M
    bad = _tree_first_token_law(lp, lq, oracle.VARIANT_LOSSLESS, n=3, replace=False)
    assert np.max(np.abs(bad - p)) > 5e-3


def test_gumbel_top_draws_without_replacement():
    """The drafts that exercise the without-replacement rule: the first two of
    l + G (Gumbel-top-k) follow sequential sampling without replacement,
    P(x, y) = q(x) q(y) / (1 - q(x))."""
    V, n = 4, 200_000
    rng = np.random.default_rng(21)
    l = (rng.standard_normal(V) * 1.2).astype(np.float32)
    q = _softmax64(l)
    pairs = np.array([workloads.gumbel_top(rng, l, 1.0, 2) for _ in range(n)])
    assert np.all(pairs[:, 0] != pairs[:, 1])
    freq = np.zeros((V, V))
    np.add.at(freq, (pairs[:, 0], pairs[:, 1]), 1.0 / n)
    law = q[:, None] * q[None, :] / (1.0 - q[:, None])
    np.fill_diagonal(law, 0.0)
    assert np.max(np.abs(freq - law)) < 5 * np.sqrt(0.25 / n)
    with pytest.raises(ValueError):
        workloads.gumbel_top(rng, l, 1.0, V + 1)
