"""GPU parity of the grid chain kernel (one cooperative launch, every
request's rows held in registers across the CTAs) against the oracle.

Every case asserts through the trace that the grid kernel ran.  The shapes
cover one to eight register slots per warp, one to 152 CTAs, slices that end
inside a 16-byte group (scalar path), unaligned and broadcast strides,
variable draft lengths, emission caps and bad tokens, masked logits, k = 0,
greedy ties, and repeated graph replays (the barrier counter must come back
to zero after every launch).
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_02_gb300 import api, workloads
from tests.parity import check_chain_sample, host, poison_like, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _grid_path():
    import __graft_entry__
    __graft_entry__.build()
    api.set_chain_path(api.CHAIN_GRID)
    yield
    api.set_chain_path(api.CHAIN_AUTO)


def _traced(fn):
    api.trace_enable(True)
    api.trace_collect()
    try:
        out = fn()
        torch.cuda.synchronize()
        launched = api.trace_collect()
    finally:
        api.trace_enable(False)
    return out, launched


def _sample(prob, draft_len=None, max_emit=None, T=None, D=None):
    args = dict(draft_len=None if draft_len is None else to_dev(draft_len),
                max_emit=None if max_emit is None else to_dev(max_emit))
    T = to_dev(prob["target"]) if T is None else T
    D = to_dev(prob["draft_logits"]) if D is None else D
    x, u = to_dev(prob["draft"]), to_dev(prob["uniforms"])
    o = api.spec_verify_sample(T, D, x, u, prob["T"], **args)
    poison_like(o)
    o, launched = _traced(lambda: api.spec_verify_sample(T, D, x, u, prob["T"], out=o, **args))
    assert "chain_grid_sample" in launched, launched
    assert len(launched) == 1, launched          # one launch does the whole call
    return host(o)


def _oracle(prob, draft_len=None, max_emit=None):
    return oracle.verify_sample(prob["target"], prob["draft_logits"], prob["draft"], prob["uniforms"], prob["T"],
                                draft_len=draft_len, max_emit=max_emit, threads=oracle.max_threads())


@pytest.mark.parametrize("seed,B,k,V,dtype,T", [
    (1, 1, 4, 248_320, "bf16", 1.0),     # 152 CTAs, 7 chunks per row slice, 3 slots
    (2, 4, 4, 2048, "fp32", 1.0),        # 16 CTAs, 1 chunk
    (3, 2, 4, 300_000, "bf16", 1.0),     # 8 slots
    (4, 3, 7, 32_000, "bf16", 0.7),      # 2 slots
    (5, 1, 2, 7, "fp32", 1.0),           # one CTA, a slice shorter than a group
    (6, 5, 3, 40_003, "bf16", 1.2),      # V ends inside a group: scalar loads
    (7, 8, 4, 20_000, "bf16", 0.9),
    (8, 16, 3, 4000, "fp32", 1.0),
    (9, 2, 0, 100_000, "bf16", 1.0)])    # k = 0: the draw from p_0 alone
def test_grid_sample_parity(seed, B, k, V, dtype, T):
    prob = workloads.chain_problem(seed, B, k, V, dtype, T, target_std=1.5,
                                   noise_std=np.linspace(0.3, 2.0, B).astype(np.float32))
    g, r = _sample(prob), _oracle(prob)
    print("near-threshold", check_chain_sample(prob, g, r))


def test_grid_headline_shape_many_seeds():
    """B=1, k=4, V=248,320 bf16 (t~N(0,3) with 5 peaks, d=0.8t+N(0,1)), 16 seeds:
    both rejections and full accepts occur."""
    acc = []
    for s in range(16):
        prob = workloads.chain_vocab248k(workloads.SEED_BASE + 3 + 7919 * s, B=1)
        g, r = _sample(prob), _oracle(prob)
        check_chain_sample(prob, g, r)
        acc.append(int(r["accepted"][0]))
    assert min(acc) < 4 and max(acc) == 4, acc


def test_grid_lengths_caps_bad_tokens():
    rng = np.random.default_rng(3)
    B, k, V = 20, 5, 6000
    prob = workloads.chain_problem(41, B, k, V, "bf16", 1.0, target_std=1.0, noise_std=0.5)
    draft_len = rng.integers(0, k + 1, B).astype(np.int32)
    draft_len[0], draft_len[2] = -1, k + 1
    prob["draft"][1, 0] = V
    draft_len[1] = 3
    max_emit = rng.integers(0, k + 2, B).astype(np.int32)
    g, r = _sample(prob, draft_len, max_emit), _oracle(prob, draft_len, max_emit)
    check_chain_sample(prob, g, r, draft_len=draft_len)
    assert list(g["status"][:3]) == [3, 1, 3]


def test_grid_masked_logits():
    prob = workloads.chain_problem(42, 8, 3, 9000, "fp32", 1.0, target_std=1.0, noise_std=0.7)
    rng = np.random.default_rng(1)
    for arr in (prob["target"], prob["draft_logits"]):
        arr[rng.random(arr.shape) < 0.4] = -np.inf
    for b in range(8):
        for i in range(3):
            prob["draft"][b, i] = workloads.gumbel_draw(rng, prob["draft_logits"][b, i], 1.0)
    check_chain_sample(prob, _sample(prob), _oracle(prob))


def test_grid_unaligned_and_broadcast_strides():
    rng = np.random.default_rng(5)
    B, k, V = 3, 2, 5001
    prob = workloads.chain_problem(43, B, k, V, "fp32", 1.0, target_std=1.5, noise_std=0.8)
    pad_t = np.zeros((B, k + 1, V + 3), np.float32)
    pad_t[:, :, 1:V + 1] = prob["target"]
    pad_d = np.zeros((B, k, V + 3), np.float32)
    pad_d[:, :, 1:V + 1] = prob["draft_logits"]
    T, D = to_dev(pad_t)[:, :, 1:V + 1], to_dev(pad_d)[:, :, 1:V + 1]   # rows 4 bytes off alignment
    check_chain_sample(prob, _sample(prob, T=T, D=D), _oracle(prob))
    one = dict(prob, target=np.broadcast_to(prob["target"][:1], prob["target"].shape),
               draft_logits=np.broadcast_to(prob["draft_logits"][:1], prob["draft_logits"].shape))
    one["draft"] = np.broadcast_to(prob["draft"][:1], prob["draft"].shape).copy()
    Tb = to_dev(prob["target"][:1]).expand(B, k + 1, V)
    Db = to_dev(prob["draft_logits"][:1]).expand(B, k, V)
    check_chain_sample(one, _sample(one, T=Tb, D=Db), _oracle(one))


def test_grid_graph_replay_and_path_switching():
    """Graph replays of the grid kernel, with two-pass calls on the same
    workspace in between: the barrier counter is left zero every time."""
    prob = workloads.chain_vocab248k(workloads.SEED_BASE + 77, B=2)
    r = _oracle(prob)
    T, D = to_dev(prob["target"]), to_dev(prob["draft_logits"])
    x, u = to_dev(prob["draft"]), to_dev(prob["uniforms"])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        o = api.spec_verify_sample(T, D, x, u, 1.0)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for _ in range(3):
                api.spec_verify_sample(T, D, x, u, 1.0, out=o)
    torch.cuda.current_stream().wait_stream(s)
    for rep in range(20):
        poison_like(o)
        with torch.cuda.stream(s):
            g.replay()
            if rep % 5 == 4:   # the two-pass path on the same stream and workspace
                api.set_chain_path(api.CHAIN_TWO_PASS)
                o2 = api.spec_verify_sample(T, D, x, u, 1.0)
                api.set_chain_path(api.CHAIN_GRID)
        torch.cuda.synchronize()
        check_chain_sample(prob, host(o), r)
        if rep % 5 == 4:
            check_chain_sample(prob, host(o2), r)
    ws = api.workspace(1, T.device, s)
    assert int(ws[:4].view(torch.int32).item()) == 0   # the counter at rest


# --------------------------------------------------------------------- greedy

def _greedy(target, draft, draft_len=None, max_emit=None):
    T = to_dev(target)
    args = (None if draft_len is None else to_dev(draft_len), None if max_emit is None else to_dev(max_emit))
    o = api.spec_verify_greedy(T, to_dev(draft), *args)
    poison_like(o)
    o, launched = _traced(lambda: api.spec_verify_greedy(T, to_dev(draft), *args, out=o))
    assert "chain_grid_greedy" in launched and len(launched) == 1, launched
    return host(o)


@pytest.mark.parametrize("dtype,V,B,k", [("bf16", 248_320, 1, 4), ("fp32", 2048, 4, 4), ("bf16", 1, 3, 2),
                                         ("bf16", 70_001, 6, 3), ("fp32", 9, 20, 5)])
def test_grid_greedy_parity(dtype, V, B, k):
    rng = np.random.default_rng(V + 17 * B)
    prob = workloads.chain_problem(int(rng.integers(1 << 30)), B, k, V, dtype, target_std=2.0)
    t = workloads.logits_as_f64(prob["target"])
    draft = t.argmax(-1)[:, :k].astype(np.int32)
    for b in range(B):
        for i in range(k):
            if V > 1 and rng.random() < 0.3:
                draft[b, i] = (draft[b, i] + 1) % V
    draft_len = rng.integers(0, k + 1, B).astype(np.int32)
    max_emit = rng.integers(0, k + 2, B).astype(np.int32)
    g = _greedy(prob["target"], draft, draft_len, max_emit)
    r = oracle.verify_greedy(prob["target"], draft, draft_len, max_emit)
    for key in ("accepted", "out_tokens", "n_emit", "status"):
        np.testing.assert_array_equal(g[key], r[key], err_msg=key)


def test_grid_greedy_ties_across_slices():
    """The maximum repeated in many CTAs' slices: the lowest index wins."""
    B, k, V = 2, 3, 200_000
    rng = np.random.default_rng(8)
    t = rng.integers(-3, 3, (B, k + 1, V)).astype(np.float32)
    for b in range(B):
        for i in range(k + 1):
            t[b, i, np.sort(rng.choice(V, 40, replace=False))] = 9.0
    bits = workloads.bf16_bits(t)
    draft = workloads.logits_as_f64(bits).argmax(-1)[:, :k].astype(np.int32)
    g = _greedy(bits, draft)
    r = oracle.verify_greedy(bits, draft)
    for key in ("accepted", "out_tokens", "n_emit", "status"):
        np.testing.assert_array_equal(g[key], r[key], err_msg=key)
    assert (g["accepted"] == k).all()


def test_grid_spec_sample_draws():
    """spec_sample (k = 0) on the grid path: tokens and probabilities."""
    rng = np.random.default_rng(12)
    B, V = 6, 50_000
    x = workloads.bf16_bits(rng.normal(0, 2, (B, V)).astype(np.float32))
    u = rng.random(B, dtype=np.float32)
    g, launched = _traced(lambda: api.spec_sample(to_dev(x), to_dev(u), 0.8))
    assert "chain_grid_sample" in launched, launched
    g = host(g)
    for b in range(B):
        r = oracle.verify_sample(np.ascontiguousarray(x[b:b + 1, None]), np.zeros((1, 0, V), x.dtype),
                                 np.zeros((1, 0), np.int32), u[b:b + 1, None], 0.8)
        p = oracle.softmax(x[b], 0.8)
        assert int(g["tokens"][b]) == int(r["out_tokens"][0, 0]) or abs(np.cumsum(p)[g["tokens"][b]] - u[b]) < 1e-5
        assert abs(g["probs"][b] - p[g["tokens"][b]]) <= 1e-5
