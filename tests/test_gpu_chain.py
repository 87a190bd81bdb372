"""GPU parity of chain verification (greedy and sampling) against the oracle.

Greedy outputs and accept counts are compared bit for bit.  Sampled
decisions follow the rule in tests/parity.py (near-threshold cases counted),
per-token probabilities within 1e-5 absolute.  Every test runs once on each
chain path (two-pass and fused; a fused call whose clusters cannot all be
resident runs two-pass).
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_02_gb300 import api, workloads
from tests.parity import check_chain_sample, host, poison_like, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.fixture(scope="module", autouse=True, params=["two_pass", "fused", "chunked"])
def chain_path(request, _built):
    api.set_chain_path({"two_pass": api.CHAIN_TWO_PASS, "fused": api.CHAIN_FUSED,
                         "chunked": api.CHAIN_CHUNKED}[request.param])
    yield request.param
    api.set_chain_path(api.CHAIN_AUTO)


def _greedy_drafts(target_bits_or_f32, rng, accept_prob=0.7):
    """Drafts that agree with the target's argmax for a random prefix."""
    t = workloads.logits_as_f64(target_bits_or_f32)
    am = t.argmax(-1).astype(np.int32)          # numpy argmax: first index of the max
    B, R, V = t.shape
    draft = am[:, :R - 1].copy()
    for b in range(B):
        for i in range(R - 1):
            if V > 1 and rng.random() > accept_prob:
                draft[b, i] = (draft[b, i] + 1 + rng.integers(V - 1)) % V
    return draft


def _run_greedy(target, draft, draft_len=None, max_emit=None):
    dev = "cuda"
    o = api.spec_verify_greedy(to_dev(target), to_dev(draft),
                               None if draft_len is None else to_dev(draft_len),
                               None if max_emit is None else to_dev(max_emit))
    # run again into poisoned buffers: every slot must be rewritten
    poison_like(o)
    o = api.spec_verify_greedy(to_dev(target), to_dev(draft),
                               None if draft_len is None else to_dev(draft_len),
                               None if max_emit is None else to_dev(max_emit), out=o)
    torch.cuda.synchronize()
    return host(o)


def _assert_greedy_equal(g, r):
    for key in ("accepted", "out_tokens", "n_emit", "status"):
        np.testing.assert_array_equal(g[key], r[key], err_msg=key)


@pytest.mark.parametrize("dtype,V,B,k", [("fp32", 2048, 4, 4), ("bf16", 2048, 16, 4),
                                         ("bf16", 248320, 2, 4), ("bf16", 128256, 8, 8),
                                         ("fp32", 32000, 8, 4), ("bf16", 1003, 9, 3),
                                         ("fp32", 16389, 5, 2), ("bf16", 1, 3, 2)])
def test_greedy_parity(dtype, V, B, k):
    rng = np.random.default_rng(V + B + k)
    prob = workloads.chain_problem(int(rng.integers(1 << 30)), B, k, V, dtype, target_std=2.0)
    draft = _greedy_drafts(prob["target"], rng)
    g = _run_greedy(prob["target"], draft)
    r = oracle.verify_greedy(prob["target"], draft)
    _assert_greedy_equal(g, r)
    assert g["accepted"].max() > 0 or V == 1 or B < 4


def test_greedy_ties_lowest_index():
    # bf16 rows with the maximum repeated at many places
    B, k, V = 6, 3, 70000
    rng = np.random.default_rng(3)
    t = np.zeros((B, k + 1, V), np.float32)
    for b in range(B):
        for i in range(k + 1):
            t[b, i] = rng.integers(-3, 3, V)
            t[b, i, rng.choice(V, 17, replace=False)] = 5.0
    bits = workloads.bf16_bits(t)
    draft = _greedy_drafts(bits, rng, 0.8)
    _assert_greedy_equal(_run_greedy(bits, draft), oracle.verify_greedy(bits, draft))
    # all-equal rows: argmax is index 0; -inf rows too
    t2 = np.zeros((2, 2, 5000), np.float32)
    t2[1] = -np.inf
    d2 = np.zeros((2, 1), np.int32)
    g = _run_greedy(t2, d2)
    _assert_greedy_equal(g, oracle.verify_greedy(t2, d2))
    assert list(g["out_tokens"][:, 1]) == [0, 0]


def test_greedy_lengths_caps_and_bad_tokens():
    rng = np.random.default_rng(5)
    B, k, V = 12, 5, 4096
    prob = workloads.chain_problem(77, B, k, V, "bf16", target_std=2.0)
    draft = _greedy_drafts(prob["target"], rng, 0.9)
    draft_len = rng.integers(0, k + 1, B).astype(np.int32)
    draft_len[0], draft_len[1] = -1, k + 1        # bad lengths
    draft[2, 0] = V                                # out of range
    draft[3, 1] = -5
    draft_len[3] = 3
    max_emit = rng.integers(0, k + 2, B).astype(np.int32)
    g = _run_greedy(prob["target"], draft, draft_len, max_emit)
    r = oracle.verify_greedy(prob["target"], draft, draft_len, max_emit)
    _assert_greedy_equal(g, r)
    assert list(g["status"][:4]) == [3, 3, 1, 1]


def test_greedy_strided_and_broadcast_layouts():
    rng = np.random.default_rng(9)
    B, k, V = 5, 3, 3001
    base = rng.standard_normal((B, k + 2, V + 3)).astype(np.float32)
    dev = to_dev(base)
    view = dev[:, 1:, :V]                           # row stride V+3 (unaligned), offset start
    tgt = base[:, 1:, :V]
    draft = _greedy_drafts(tgt, rng)
    o = api.spec_verify_greedy(view, to_dev(draft))
    torch.cuda.synchronize()
    _assert_greedy_equal(host(o), oracle.verify_greedy(np.ascontiguousarray(tgt), draft))
    # request stride 0: every request reads the same rows
    one = to_dev(tgt[:1])
    bview = one.expand(B, k + 1, V)
    o = api.spec_verify_greedy(bview, to_dev(draft))
    torch.cuda.synchronize()
    _assert_greedy_equal(host(o), oracle.verify_greedy(np.broadcast_to(tgt[:1], (B, k + 1, V)), draft))


def test_greedy_empty_batch_and_zero_k():
    t = to_dev(np.zeros((0, 3, 10), np.float32))
    o = api.spec_verify_greedy(t, torch.zeros((0, 2), dtype=torch.int32, device="cuda"))
    assert o["accepted"].numel() == 0
    x = np.random.default_rng(0).standard_normal((4, 1, 777)).astype(np.float32)
    g = _run_greedy(x, np.zeros((4, 0), np.int32))
    _assert_greedy_equal(g, oracle.verify_greedy(x, np.zeros((4, 0), np.int32)))


# ------------------------------------------------------------------ sampling

def _run_sample(prob, draft_len=None, max_emit=None, probs=True):
    args = dict(draft_len=None if draft_len is None else to_dev(draft_len),
                max_emit=None if max_emit is None else to_dev(max_emit), probs=probs)
    T = to_dev(prob["target"])
    D = to_dev(prob["draft_logits"])
    o = api.spec_verify_sample(T, D, to_dev(prob["draft"]), to_dev(prob["uniforms"]), prob["T"], **args)
    poison_like(o)
    o = api.spec_verify_sample(T, D, to_dev(prob["draft"]), to_dev(prob["uniforms"]), prob["T"], out=o,
                               **args)
    torch.cuda.synchronize()
    return host(o)


def _oracle_sample(prob, draft_len=None, max_emit=None):
    return oracle.verify_sample(prob["target"], prob["draft_logits"], prob["draft"], prob["uniforms"],
                                prob["T"], draft_len=draft_len, max_emit=max_emit,
                                threads=oracle.max_threads())


def test_sample_parity_small_chain():
    """The V=2048 fp32 chain, B=4, k=4, T=1 workload."""
    prob = workloads.chain_small()
    stats = check_chain_sample(prob, _run_sample(prob), _oracle_sample(prob))
    print("near-threshold", stats)


@pytest.mark.parametrize("seed,B,k,V,dtype,T", [(1, 128, 4, 2048, "fp32", 1.0), (2, 96, 6, 5000, "bf16", 0.7),
                                               (3, 64, 8, 1003, "bf16", 1.3), (4, 33, 1, 40000, "fp32", 1.0),
                                               (5, 40, 3, 9, "bf16", 1.0), (6, 16, 0, 3000, "bf16", 1.0)])
def test_sample_parity_many(seed, B, k, V, dtype, T):
    prob = workloads.chain_problem(seed, B, k, V, dtype, T, target_std=1.5,
                                   noise_std=np.linspace(0.2, 2.0, B).astype(np.float32))
    g, r = _run_sample(prob), _oracle_sample(prob)
    stats = check_chain_sample(prob, g, r)
    print("near-threshold", stats)
    if k > 0:
        assert 0 < r["accepted"].mean() < k


def test_sample_parity_vocab248k():
    """The V=248,320 bf16, B=1, k=4 workload at full size, several seeds."""
    for seed in range(4):
        prob = workloads.chain_vocab248k(workloads.SEED_BASE + 3 + 1000 * seed, B=2)
        check_chain_sample(prob, _run_sample(prob), _oracle_sample(prob))


def test_sample_parity_batch64():
    """The V=128,256 bf16, B=64, k=8, T=0.7 workload at full size."""
    prob = workloads.chain_batch64()
    stats = check_chain_sample(prob, _run_sample(prob), _oracle_sample(prob))
    print("near-threshold", stats)


def test_sample_lengths_caps_bad_tokens_and_no_prob_outputs():
    rng = np.random.default_rng(11)
    B, k, V = 24, 6, 3000
    prob = workloads.chain_problem(21, B, k, V, "bf16", 1.0, target_std=1.0, noise_std=0.5)
    draft_len = rng.integers(0, k + 1, B).astype(np.int32)
    draft_len[0] = -2
    prob["draft"][1, 0] = V + 1
    draft_len[1] = 2
    max_emit = rng.integers(0, k + 2, B).astype(np.int32)
    g = _run_sample(prob, draft_len, max_emit)
    r = _oracle_sample(prob, draft_len, max_emit)
    check_chain_sample(prob, g, r, draft_len=draft_len)
    assert g["status"][0] == 3 and g["status"][1] == 1
    g2 = _run_sample(prob, draft_len, max_emit, probs=False)
    for key in ("accepted", "out_tokens", "n_emit", "status"):
        np.testing.assert_array_equal(g2[key], g[key])


def test_sample_masked_logits():
    """-inf logits (masked tokens) in both rows."""
    prob = workloads.chain_problem(31, 16, 3, 4000, "fp32", 1.0, target_std=1.0, noise_std=0.7)
    rng = np.random.default_rng(0)
    for arr in (prob["target"], prob["draft_logits"]):
        mask = rng.random(arr.shape) < 0.3
        arr[mask] = -np.inf
    for b in range(16):
        for i in range(3):
            prob["draft"][b, i] = workloads.gumbel_draw(rng, prob["draft_logits"][b, i], 1.0)
    check_chain_sample(prob, _run_sample(prob), _oracle_sample(prob))


def test_total_variation_200k_on_gpu():
    """200,000 independent verifications of one V=2048 position on the GPU:
    the first emitted token is distributed as p (TV at sampling noise), and
    every decision matches the oracle's under the decision rule."""
    prob = workloads.chain_small()
    lp, lq, lb = prob["target"][0, 0], prob["draft_logits"][0, 0], prob["target"][0, 1]
    V, n = lp.size, 200_000
    p = oracle.softmax(lp)
    q = oracle.softmax(lq)
    rng = np.random.default_rng(4242)
    draft = rng.choice(V, size=(n, 1), p=q).astype(np.int32)
    u = rng.random((n, 2), dtype=np.float32)
    T = to_dev(np.stack([lp, lb]))[None].expand(n, 2, V)
    D = to_dev(lq)[None, None].expand(n, 1, V)
    o = host(api.spec_verify_sample(T, D, to_dev(draft), to_dev(u), 1.0))
    tv = 0.5 * np.abs(np.bincount(o["out_tokens"][:, 0], minlength=V) / n - p).sum()
    noise = 0.5 * np.sum(np.sqrt(2 * p * (1 - p) / (np.pi * n)))
    assert tv < 1.2 * noise
    big = dict(target=np.broadcast_to(np.stack([lp, lb]), (n, 2, V)),
               draft_logits=np.broadcast_to(lq[None], (n, 1, V)), draft=draft, uniforms=u, T=1.0)
    r = oracle.verify_sample(big["target"], big["draft_logits"], draft, u, 1.0, threads=oracle.max_threads())
    stats = check_chain_sample(big, o, r)
    print("TV", tv, "noise", noise, stats)


def test_workspace_reuse_and_graph_replay():
    prob = workloads.chain_problem(8, 8, 4, 20000, "bf16", 1.0, target_std=2.0, noise_std=1.0)
    r = _oracle_sample(prob)
    T, D = to_dev(prob["target"]), to_dev(prob["draft_logits"])
    x, u = to_dev(prob["draft"]), to_dev(prob["uniforms"])
    o = api.spec_verify_sample(T, D, x, u, 1.0)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        api.spec_verify_sample(T, D, x, u, 1.0, out=o)   # warm the workspace on this stream
        with torch.cuda.graph(g, stream=s):
            api.spec_verify_sample(T, D, x, u, 1.0, out=o)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(5):
        poison_like(o)
        g.replay()
        torch.cuda.synchronize()
        check_chain_sample(prob, host(o), r)


@pytest.mark.parametrize("seed,B,k,V,dtype,T", [(21, 400, 4, 3001, "bf16", 0.9), (22, 420, 3, 2500, "fp32", 1.0),
                                               (23, 2, 4, 600_000, "bf16", 1.0), (24, 200, 6, 40_003, "bf16", 1.1)])
def test_sample_parity_chunked_accept_path(seed, B, k, V, dtype, T, chain_path):
    """Shapes that take the chunked accept kernel: more requests than one
    wave of cluster-accept CTAs (two 512-thread CTAs per SM on 152 SMs), or
    V beyond 16 CTAs of 32,768 logits."""
    prob = workloads.chain_problem(seed, B, k, V, dtype, T, target_std=1.5,
                                   noise_std=np.linspace(0.3, 2.0, B).astype(np.float32))
    rng = np.random.default_rng(seed)
    draft_len = rng.integers(0, k + 1, B).astype(np.int32)
    max_emit = rng.integers(1, k + 2, B).astype(np.int32)
    api.trace_enable(True)
    api.trace_collect()
    try:
        g = _run_sample(prob, draft_len, max_emit)
        launched = api.trace_collect()
    finally:
        api.trace_enable(False)
    if chain_path == "two_pass":
        assert "chain_sample_accept" in launched, launched
    r = _oracle_sample(prob, draft_len, max_emit)
    stats = check_chain_sample(prob, g, r, draft_len=draft_len)
    print("near-threshold", stats)
    assert (r["accepted"] < draft_len).any() and (r["accepted"] == draft_len).any()


@pytest.mark.parametrize("seed,B,k,V,dtype,T", [(31, 160, 4, 3001, "bf16", 0.9), (32, 2, 4, 300_000, "bf16", 1.0),
                                               (33, 24, 5, 40_003, "fp32", 1.2)])
def test_sample_parity_cluster_accept_path(seed, B, k, V, dtype, T, chain_path):
    """Shapes whose two-pass path ends in the cluster accept kernel (every
    request's cluster resident at once, slices of at most 32,768 logits)."""
    prob = workloads.chain_problem(seed, B, k, V, dtype, T, target_std=1.5,
                                   noise_std=np.linspace(0.3, 2.0, B).astype(np.float32))
    rng = np.random.default_rng(seed)
    draft_len = rng.integers(0, k + 1, B).astype(np.int32)
    max_emit = rng.integers(1, k + 2, B).astype(np.int32)
    api.trace_enable(True)
    api.trace_collect()
    try:
        g = _run_sample(prob, draft_len, max_emit)
        launched = api.trace_collect()
    finally:
        api.trace_enable(False)
    if chain_path == "two_pass":
        assert "chain_sample_accept_cluster" in launched, launched
    r = _oracle_sample(prob, draft_len, max_emit)
    stats = check_chain_sample(prob, g, r, draft_len=draft_len)
    print("near-threshold", stats)
    if B >= 16:  # enough requests that some are rejected
        assert (r["accepted"] < draft_len).any()


@pytest.mark.parametrize("dtype,offset", [("fp32", 40.0), ("bf16", 40.0), ("fp32", -300.0)])
def test_sample_parity_large_logits_low_temperature(dtype, offset):
    """Logits shifted to +40 (or -300) at T = 0.05, so |max| / T is above
    1,000: every exponent must be formed as (x - max) / T.  Rounding max / T
    on its own would shift all of them by up to 6e-5 and put p off by more
    than the 1e-5 tolerance."""
    rng = np.random.default_rng(61)
    B, k, V, T = 24, 4, 30_000, 0.05
    base = workloads.chain_problem(61, B, k, V, "fp32", 1.0, target_std=0.15,
                                   noise_std=np.linspace(0.005, 0.05, B).astype(np.float32))
    cast = workloads.bf16_bits if dtype == "bf16" else (lambda a: np.ascontiguousarray(a, np.float32))
    prob = dict(base, target=cast(base["target"] + np.float32(offset)),
                draft_logits=cast(base["draft_logits"] + np.float32(offset)), T=T, dtype=dtype)
    for b in range(B):
        for i in range(k):
            prob["draft"][b, i] = workloads.gumbel_draw(rng, prob["draft_logits"][b, i], T)
    g, r = _run_sample(prob), _oracle_sample(prob)
    print("near-threshold", check_chain_sample(prob, g, r))
    assert 0 < r["accepted"].mean() < k
