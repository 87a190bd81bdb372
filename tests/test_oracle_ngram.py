"""Pins for the n-gram history-lookup drafter.

The oracle scans every start position.  The pins use a different route:
hand-worked cases, and for every short history over a 2- or 3-letter
alphabet, Python's own substring search (str.rfind over the history encoded
as text), which finds the rightmost earlier occurrence of the window.
"""
import itertools

import numpy as np
import pytest

import oracle
from speculative_decoding_verification_02_gb300 import workloads

# (history, window, k, expected draft)
CASES = [
    ([5, 6, 7, 8, 5, 6, 7], 3, 4, [8, 5, 6, 7]),        # one earlier copy, full continuation
    ([1, 2, 3, 9, 1, 2, 3, 4, 1, 2, 3], 3, 2, [4, 1]),  # two earlier copies: the later one wins
    ([1, 2, 3, 4], 3, 4, []),                             # no earlier copy
    ([7, 7, 7, 7], 3, 4, [7]),                            # overlapping copy, cut at the end
    ([1, 2, 3, 5, 1, 2, 3], 3, 8, [5, 1, 2, 3]),          # continuation cut at the history end
    ([1, 2, 3], 3, 4, []),                                # only the window itself
    ([], 3, 4, []),                                       # empty history
    ([4, 4], 1, 3, [4]),                                  # window of one token
]


@pytest.mark.parametrize("hist,w,k,expect", CASES)
def test_hand_cases(hist, w, k, expect):
    H = max(len(hist), 1)
    h = np.zeros((1, H), np.int32)
    h[0, :len(hist)] = hist
    d, n, st = oracle.ngram_draft(h, [len(hist)], w, k)
    assert st[0] == 0
    assert list(d[0, :n[0]]) == expect
    assert np.all(d[0, n[0]:] == -1)


def _by_rfind(seq, w, k):
    s = "".join(chr(ord("a") + t) for t in seq)
    n = len(s)
    if n <= w:
        return []
    i = s.rfind(s[n - w:], 0, n - 1)      # occurrence entirely inside s[0:n-1]
    return [] if i < 0 else list(seq[i + w:i + w + k])


@pytest.mark.parametrize("V,nmax", [(2, 10), (3, 7)])
@pytest.mark.parametrize("w,k", [(1, 1), (2, 3), (3, 4)])
def test_exhaustive_small_histories(V, nmax, w, k):
    seqs = [s for n in range(nmax + 1) for s in itertools.product(range(V), repeat=n)]
    H = nmax
    h = np.zeros((len(seqs), H), np.int32)
    for b, s in enumerate(seqs):
        h[b, :len(s)] = s
    lens = np.array([len(s) for s in seqs], np.int32)
    d, n, st = oracle.ngram_draft(h, lens, w, k)
    assert np.all(st == 0)
    for b, s in enumerate(seqs):
        assert list(d[b, :n[b]]) == _by_rfind(s, w, k), s


def test_planted_spans_are_found():
    prob = workloads.ngram_problem(workloads.SEED_BASE + 2)
    d, n, st = oracle.ngram_draft(prob["history"], prob["hist_len"], prob["window"], prob["k"])
    assert np.all(st == 0)
    planted = prob["planted_next"]
    hits = 0
    for b in range(prob["B"]):
        if planted[b, 0] >= 0:
            hits += list(d[b, :n[b]]) == [t for t in planted[b] if t >= 0][:n[b]] and n[b] > 0
    assert hits >= 0.9 * np.sum(planted[:, 0] >= 0)


def test_bad_lengths_are_flagged():
    h = np.arange(12, dtype=np.int32).reshape(2, 6)
    d, n, st = oracle.ngram_draft(h, [7, -1], 3, 2)
    assert list(st) == [oracle.ST_BAD_LENGTH] * 2 and list(n) == [0, 0]
    assert np.all(d == -1)
