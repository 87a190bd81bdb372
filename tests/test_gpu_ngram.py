"""GPU parity of the n-gram drafter (bit for bit) and of the full greedy
speculative loop driven by the library (equals plain greedy decoding)."""
import itertools

import numpy as np
import pytest
import torch

import oracle
from oracle.analysis import greedy_generate, speculative_generate
from speculative_decoding_verification_02_gb300 import api, workloads
from tests.parity import host, poison_like, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _run(hist, lens, w, k):
    o = api.spec_ngram_draft(to_dev(hist), to_dev(lens), w, k)
    poison_like(o)
    o = api.spec_ngram_draft(to_dev(hist), to_dev(lens), w, k, out=o)
    torch.cuda.synchronize()
    return host(o)


def _eq(g, r):
    np.testing.assert_array_equal(g["draft"], r[0])
    np.testing.assert_array_equal(g["draft_len"], r[1])
    np.testing.assert_array_equal(g["status"], r[2])


def test_ngram_workload_64x4096():
    prob = workloads.ngram_problem(workloads.SEED_BASE + 2)
    g = _run(prob["history"], prob["hist_len"], 3, 4)
    r = oracle.ngram_draft(prob["history"], prob["hist_len"], 3, 4)
    _eq(g, r)
    assert (r[1] > 0).sum() >= 30


def test_ngram_exhaustive_small():
    seqs = [s for n in range(11) for s in itertools.product(range(2), repeat=n)]
    h = np.zeros((len(seqs), 10), np.int32)
    for b, s in enumerate(seqs):
        h[b, :len(s)] = s
    lens = np.array([len(s) for s in seqs], np.int32)
    for w, k in [(1, 1), (2, 3), (3, 4), (4, 2)]:
        _eq(_run(h, lens, w, k), oracle.ngram_draft(h, lens, w, k))


@pytest.mark.parametrize("H,V,w,k", [(10000, 50, 3, 8), (5000, 3, 5, 4), (20000, 32000, 2, 6), (3, 5, 3, 4),
                                     (5003, 7, 4, 3),      # odd stride: 16-byte and 4-byte aligned rows mixed
                                     (9000, 1000, 64, 8)])  # the longest window (a match is planted)
def test_ngram_long_and_ragged(H, V, w, k):
    rng = np.random.default_rng(H + V)
    B = 24
    h = rng.integers(0, V, (B, H)).astype(np.int32)
    lens = rng.integers(0, H + 1, B).astype(np.int32)
    lens[0], lens[1] = H, 0
    if H > 100:
        # a match only near the start of a long history: the walk must reach early tiles
        h[2, :] = np.arange(H) % 100000 + 100000
        h[2, 5:5 + w] = h[2, H - w:H]
        lens[2] = H
    lens[3] = H + 1                 # bad length
    if B > 4:
        lens[4] = -1
    g = _run(h, lens, w, k)
    _eq(g, oracle.ngram_draft(h, lens, w, k))
    assert g["status"][3] == 3


def test_speculative_greedy_on_gpu_equals_plain_greedy():
    """The draft -> verify -> append loop run on the library's kernels emits
    exactly the tokens plain greedy decoding emits."""
    V, k, window = 12, 4, 3

    def model(seed):
        def next_logits(seq):
            a = seq[-2] if len(seq) > 1 else V
            rng = np.random.default_rng(seed * 1_000_003 + a * (V + 1) + seq[-1])
            return rng.standard_normal(V).astype(np.float32)
        return next_logits

    def draft_fn(hist):
        o = api.spec_ngram_draft(to_dev(np.array([hist], np.int32)), to_dev(np.array([len(hist)], np.int32)),
                                 window, k)
        n = int(o["draft_len"].item())
        return list(o["draft"][0, :n].cpu().numpy())

    def verify_fn(rows, draft):
        o = api.spec_verify_greedy(to_dev(rows[None]), to_dev(np.array([draft], np.int32).reshape(1, -1)))
        n = int(o["n_emit"].item())
        return list(o["out_tokens"][0, :n].cpu().numpy())

    for seed in range(6):
        m = model(seed)
        prompt = [seed % V, (seed * 5 + 1) % V, (seed * 7 + 3) % V]
        plain = greedy_generate(m, prompt, 120, oracle.argmax)
        spec, acc = speculative_generate(m, prompt, 120, k, draft_fn, verify_fn)
        assert spec == plain
        assert max(acc) > 0
