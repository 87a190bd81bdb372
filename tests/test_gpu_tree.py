"""GPU parity of tree verification against the oracle (greedy: bit for bit;
sampling: bit for bit except decisions within 1e-5 of their fp64 threshold),
with the default rule and with siblings drawn without replacement
(spec_verify_tree_ex, SPEC_TREE_SIBLINGS_WITHOUT_REPLACEMENT, against the
oracle's without-replacement variant)."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_02_gb300 import api, workloads
from tests.parity import check_chain_sample, check_tree, host, poison_like, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _run_tree(prob, max_depth=None, greedy=False, wor=False):
    T = -1.0 if greedy else prob["T"]
    md = prob["depth"] if max_depth is None else max_depth
    args = (to_dev(prob["target"]), None if greedy else to_dev(prob["draft_logits"]),
            to_dev(prob["parents"]), to_dev(prob["node_tok"]), to_dev(prob["uniforms"]), T, md)
    flags = api.TREE_SIBLINGS_WITHOUT_REPLACEMENT if wor else 0
    o = api.spec_verify_tree(*args, flags=flags)
    poison_like(o)
    o = api.spec_verify_tree(*args, flags=flags, out=o)
    torch.cuda.synchronize()
    return host(o)


def _oracle_tree(prob, max_depth=None, greedy=False, wor=False):
    return oracle.verify_tree(prob["target"], None if greedy else prob["draft_logits"], prob["parents"],
                              prob["node_tok"], prob["uniforms"], -1.0 if greedy else prob["T"],
                              prob["depth"] if max_depth is None else max_depth,
                              variant=oracle.TREE_VARIANT_WITHOUT_REPLACEMENT if wor else oracle.VARIANT_LOSSLESS,
                              threads=oracle.max_threads())


def test_tree60_full_size():
    """B=16 trees of 60 nodes, depth 6, <=10 children, V=128,256 bf16, T=1."""
    prob = workloads.tree60()
    g, r = _run_tree(prob), _oracle_tree(prob)
    print("near-threshold", check_tree(prob, g, r), "mean accepted", r["accepted_len"].mean())
    gg, rg = _run_tree(prob, greedy=True), _oracle_tree(prob, greedy=True)
    check_tree(dict(prob, T=-1.0), gg, rg)


@pytest.mark.parametrize("seed,B,N,depth,kids,V,dtype,T", [
    (1, 24, 12, 3, 4, 3000, "bf16", 1.0), (2, 24, 30, 5, 6, 20011, "fp32", 0.8),
    (3, 8, 1, 0, 1, 5000, "bf16", 1.0), (4, 12, 40, 8, 10, 70000, "bf16", 1.2),
    (5, 30, 6, 2, 5, 17, "fp32", 1.0), (6, 10, 100, 10, 12, 8192, "bf16", 1.0)])
def test_tree_parity_shapes(seed, B, N, depth, kids, V, dtype, T):
    prob = workloads.tree_problem(seed, B, N, depth, kids, V, dtype, T, target_std=1.2, noise_std=0.6,
                                  peaks=0)
    g, r = _run_tree(prob), _oracle_tree(prob)
    print("near-threshold", check_tree(prob, g, r))
    gg, rg = _run_tree(prob, greedy=True), _oracle_tree(prob, greedy=True)
    check_tree(dict(prob, T=-1.0), gg, rg)


def test_tree_greedy_walks_deep_branches():
    # the target's argmax follows the drafted tokens, so greedy walks go deep
    prob = workloads.tree_problem(7, 16, 30, 6, 4, 4096, "bf16", 1.0, target_std=1.0, peaks=0)
    t = workloads.bf16_to_f32(prob["target"]).copy()
    for b in range(16):
        for u in range(30):
            kids = [c for c in range(30) if prob["parents"][b, c] == u]
            if kids:
                t[b, u, prob["node_tok"][b, kids[0]]] += 20.0
    prob["target"] = workloads.bf16_bits(t)
    gg, rg = _run_tree(prob, greedy=True), _oracle_tree(prob, greedy=True)
    check_tree(dict(prob, T=-1.0), gg, rg)
    assert np.all(rg["accepted_len"] == 6)   # the first children form the depth-6 chain 0->1->...->6


def test_tree_chain_shape_matches_chain_kernel():
    prob = workloads.chain_problem(12, 32, 5, 9000, "bf16", 1.0, target_std=1.5, noise_std=0.5)
    B, k = 32, 5
    parents = np.tile(np.arange(-1, k, dtype=np.int32), (B, 1))
    node_tok = np.concatenate([np.zeros((B, 1), np.int32), prob["draft"]], 1)
    dl = np.concatenate([prob["draft_logits"], prob["draft_logits"][:, :1]], 1)
    u_tree = np.concatenate([np.zeros((B, 1), np.float32), prob["uniforms"]], 1)
    tree = host(api.spec_verify_tree(to_dev(prob["target"]), to_dev(dl), to_dev(parents), to_dev(node_tok),
                                     to_dev(u_tree), 1.0, k))
    chain = host(api.spec_verify_sample(to_dev(prob["target"]), to_dev(prob["draft_logits"]),
                                        to_dev(prob["draft"]), to_dev(prob["uniforms"]), 1.0))
    r = oracle.verify_sample(prob["target"], prob["draft_logits"], prob["draft"], prob["uniforms"], 1.0)
    check_chain_sample(prob, chain, r)
    check_chain_sample(prob, dict(accepted=tree["accepted_len"], n_emit=tree["n_emit"],
                                  out_tokens=tree["out_tokens"], status=tree["status"]), r)


def test_tree_bad_inputs_are_flagged():
    V, N = 512, 5
    prob = workloads.tree_problem(9, 6, N, 2, 3, V, "fp32", 1.0, peaks=0)
    prob["parents"][1, 3] = 3              # parent not earlier
    prob["parents"][2, 0] = 0              # root with a parent
    prob["node_tok"][3, 2] = V             # token out of range
    prob["parents"][4] = [-1, 0, 1, 2, 3]  # depth 4 > max_depth 2
    g, r = _run_tree(prob, max_depth=2), _oracle_tree(prob, max_depth=2)
    np.testing.assert_array_equal(g["status"], r["status"])
    assert list(g["status"][1:5]) == [2, 2, 1, 2]
    for b in range(1, 5):
        assert g["n_emit"][b] == 0 and np.all(g["out_tokens"][b] == -1) and np.all(g["path_nodes"][b] == -1)
    check_tree(prob, g, r)


# ------------------------------------------------ siblings without replacement

def test_tree60_without_replacement_full_size():
    """The 16 x 60-node, V=128,256 bf16 trees with siblings drafted without
    replacement, verified with the matching rule."""
    prob = workloads.tree_problem(workloads.SEED_BASE + 5, 16, 60, 6, 10, 128256, "bf16", 1.0,
                                  siblings="without_replacement")
    g, r = _run_tree(prob, wor=True), _oracle_tree(prob, wor=True)
    print("near-threshold", check_tree(prob, g, r, without_replacement=True), "mean accepted",
          r["accepted_len"].mean())


@pytest.mark.parametrize("seed,B,N,depth,kids,V,dtype,T", [
    (11, 24, 12, 3, 4, 3000, "bf16", 1.0), (12, 24, 30, 5, 6, 20011, "fp32", 0.8),
    (13, 30, 20, 2, 8, 17, "fp32", 1.0), (14, 12, 40, 4, 12, 70000, "bf16", 1.2),
    (15, 40, 9, 1, 8, 10, "fp32", 0.5), (16, 10, 100, 10, 12, 8192, "bf16", 1.0)])
def test_tree_without_replacement_parity(seed, B, N, depth, kids, V, dtype, T):
    """Small vocabularies with many siblings remove most of q's mass; the
    target sharpened towards one peak makes removals and rejections common."""
    prob = workloads.tree_problem(seed, B, N, depth, kids, V, dtype, T, target_std=1.5, noise_std=1.0,
                                  peaks=2 if V > 16 else 0, siblings="without_replacement")
    g, r = _run_tree(prob, wor=True), _oracle_tree(prob, wor=True)
    print("near-threshold", check_tree(prob, g, r, without_replacement=True))
    # greedy walks ignore the flag
    gg, rg = _run_tree(prob, greedy=True, wor=True), _oracle_tree(prob, greedy=True)
    check_tree(dict(prob, T=-1.0), gg, rg)


def test_without_replacement_rule_differs_from_default():
    """Same inputs, both rules: the walks differ on some requests (the rule is
    in effect), and each matches its own oracle variant."""
    prob = workloads.tree_problem(17, 64, 20, 2, 8, 12, "fp32", 1.0, target_std=1.5, noise_std=1.0, peaks=0,
                                  siblings="without_replacement")
    g0, r0 = _run_tree(prob), _oracle_tree(prob)
    g2, r2 = _run_tree(prob, wor=True), _oracle_tree(prob, wor=True)
    check_tree(prob, g0, r0)
    check_tree(prob, g2, r2, without_replacement=True)
    assert (r0["out_tokens"] != r2["out_tokens"]).any(axis=1).sum() >= 3


def test_without_replacement_duplicate_and_exhausted_tokens():
    """Siblings drawn i.i.d. over V=3 repeat tokens and can remove all of q's
    mass; the rule still applies: a removed token has q = 0 and is accepted
    iff its residual p is positive."""
    prob = workloads.tree_problem(18, 48, 16, 1, 15, 3, "fp32", 1.0, target_std=1.0, noise_std=1.5, peaks=0)
    g, r = _run_tree(prob, wor=True), _oracle_tree(prob, wor=True)
    check_tree(prob, g, r, without_replacement=True)


@pytest.mark.parametrize("wor", [False, True])
def test_tree_parity_large_logits_low_temperature(wor):
    """Tree walks on logits shifted to +40 at T = 0.05 (|max| / T above 800):
    the sweeps form every exponent as (x - max) / T."""
    prob = workloads.tree_problem(62, 8, 20, 4, 4, 20_000, "fp32", 0.05, target_std=0.15, draft_scale=1.0,
                                  noise_std=0.03, peaks=0,
                                  siblings="without_replacement" if wor else "iid")
    prob["target"] = prob["target"] + np.float32(40.0)
    prob["draft_logits"] = prob["draft_logits"] + np.float32(40.0)
    g, r = _run_tree(prob, wor=wor), _oracle_tree(prob, wor=wor)
    print("near-threshold", check_tree(prob, g, r, without_replacement=wor), "mean accepted",
          r["accepted_len"].mean())
