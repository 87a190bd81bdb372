"""Pins for top-k / top-p filtered verification (the oracle's filter_row and
verify_sample with top_k / top_p).

- Hand-worked rows: top-k keeps every logit at or above the k-th largest
  (ties at the cut stay); top-p keeps the smallest descending prefix whose
  mass reaches top_p; top-k then top-p renormalises between the two (a case
  where the other order keeps a different set).
- Special cases: both filters off give softmax exactly; top_k = 1 and a tiny
  top_p keep only the maximum; the filtered row sums to 1.
- Invariants on random rows: the kept set is a prefix of the descending
  order, its mass reaches top_p, and the prefix one distinct value shorter
  does not.
- Losslessness: the first emitted token of a k = 1 chain whose draft was drawn
  from the filtered q is distributed exactly as the filtered p (each uniform
  scanned over a 2^16 grid); verifying such a draft against the unfiltered
  p is off.
"""
import numpy as np
import pytest

import oracle
from speculative_decoding_verification_02_gb300 import workloads

M = 1 << 16
U_REJECT = np.float32(1.0 - 2.0 ** -24)


def _softmax64(x):
    z = np.asarray(x, np.float64)
    e = np.exp(z - z.max())
    return e / e.sum()


def test_top_k_keeps_ties_at_the_cut():
    x = np.array([3, 1, 2, 2, 0, -1], np.float32)
    p = _softmax64(x)
    for k, keep in [(1, [0]), (2, [0, 2, 3]), (3, [0, 2, 3]), (4, [0, 1, 2, 3]), (6, [0, 1, 2, 3, 4, 5])]:
        pf, theta, kept = oracle.filter_row(x, top_k=k)
        want = np.zeros(6)
        want[keep] = p[keep] / p[keep].sum()
        np.testing.assert_allclose(pf, want, rtol=0, atol=1e-15)
        assert kept == len(keep) and theta == x[keep].min()


def test_top_p_smallest_prefix_reaching_the_mass():
    probs = np.array([0.5, 0.3, 0.15, 0.05])
    x = np.log(probs).astype(np.float32)
    p = _softmax64(x)
    for top_p, keep in [(0.49, [0]), (0.79, [0, 1]), (0.81, [0, 1, 2]), (0.96, [0, 1, 2, 3]), (1.0, [0, 1, 2, 3])]:
        pf, theta, kept = oracle.filter_row(x, top_p=top_p)
        want = np.zeros(4)
        want[keep] = p[keep] / p[keep].sum()
        np.testing.assert_allclose(pf, want, rtol=0, atol=1e-15)
        assert kept == len(keep)


def test_top_k_then_top_p_renormalises_between():
    probs = np.array([0.35, 0.25, 0.2, 0.2])
    x = np.log(probs).astype(np.float32)
    # top-k = 2 leaves [0.583, 0.417]: top-p = 0.55 keeps the first alone
    pf, _, kept = oracle.filter_row(x, top_k=2, top_p=0.55)
    assert kept == 1 and pf[0] == 1.0
    # top-p alone at 0.55 needs two tokens (0.35 + 0.25)
    _, _, kept = oracle.filter_row(x, top_p=0.55)
    assert kept == 2


def test_special_cases():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(300) * 2).astype(np.float32)
    for T in (0.7, 1.0, 1.5):
        pf, theta, kept = oracle.filter_row(x, T, 0, 1.0)
        np.testing.assert_allclose(pf, _softmax64(x.astype(np.float64) / T), rtol=1e-14, atol=1e-18)
        assert kept == 300 and theta == x.min()
        assert oracle.filter_row(x, T, 300, 1.0)[2] == 300      # top_k = V: off
    for args in [dict(top_k=1), dict(top_p=1e-6)]:
        pf, theta, kept = oracle.filter_row(x, **args)
        assert kept == 1 and pf[np.argmax(x)] == 1.0 and theta == x.max()
    bits = workloads.bf16_bits(x)
    pf, _, _ = oracle.filter_row(bits, 1.0, 40, 0.9)
    assert abs(pf.sum() - 1.0) < 1e-12


@pytest.mark.parametrize("seed", range(6))
def test_kept_set_invariants(seed):
    rng = np.random.default_rng(100 + seed)
    V = int(rng.integers(5, 400))
    x = np.round(rng.standard_normal(V) * 2, 1).astype(np.float32)    # repeated values
    T = float(rng.uniform(0.5, 2.0))
    top_k = int(rng.integers(0, V + 2))
    top_p = float(rng.uniform(0.05, 1.0))
    pf, theta, kept = oracle.filter_row(x, T, top_k, top_p)
    keep = x >= theta
    assert keep.sum() == kept and np.all(pf[~keep] == 0) and np.all(pf[keep] > 0)
    assert np.all(x[keep].min() >= x[~keep].max(initial=-np.inf))   # a prefix of the descending order
    p = _softmax64(x.astype(np.float64) / T)
    k_set = x >= (np.sort(x)[::-1][top_k - 1] if 0 < top_k < V else -np.inf)
    pk = p * k_set / p[k_set].sum()
    if top_p < 1:
        assert pk[keep].sum() >= top_p - 1e-12
        shorter = x > theta
        assert not shorter.any() or pk[shorter].sum() < top_p + 1e-12
    else:
        assert np.array_equal(keep, k_set)


def _filtered_first_token_law(lp, lq, top_k, top_p, draft_filter=True, verify_filter=True):
    """First emitted token of a k = 1 chain, the draft drawn from the filtered
    q (or the plain q), verification with or without the filter, each
    threshold scanned over a 2^16 grid."""
    V = lp.size
    grid = (np.arange(M, dtype=np.float64) / M).astype(np.float32)
    qd = oracle.filter_row(lq, 1.0, top_k, top_p)[0] if draft_filter else _softmax64(lq)
    vk, vp = (top_k, top_p) if verify_filter else (0, 1.0)
    law = np.zeros(V)
    for x in range(V):
        if qd[x] == 0:
            continue
        run = lambda u: oracle.verify_sample(np.broadcast_to(lp, (M, 2, V)), np.broadcast_to(lq, (M, 1, V)),
                                             np.full((M, 1), x, np.int32), u, T=1.0, top_k=vk, top_p=vp,
                                             threads=4)
        acc = run(np.stack([grid, np.full(M, 0.5, np.float32)], 1))["accepted"].mean()
        law[x] += qd[x] * acc
        if acc < 1.0:
            out = run(np.stack([np.full(M, U_REJECT, np.float32), grid], 1))
            assert np.all(out["accepted"] == 0)
            law += qd[x] * (1.0 - acc) * np.bincount(out["out_tokens"][:, 0], minlength=V) / M
    return law


@pytest.mark.parametrize("seed,top_k,top_p", [(0, 3, 1.0), (1, 0, 0.7), (2, 4, 0.8), (3, 2, 0.95)])
def test_filtered_verification_is_lossless_against_the_filtered_target(seed, top_k, top_p):
    rng = np.random.default_rng(40 + seed)
    V = 6
    lp = (rng.standard_normal(V) * 1.5).astype(np.float32)
    lq = (lp + rng.standard_normal(V)).astype(np.float32)
    pf = oracle.filter_row(lp, 1.0, top_k, top_p)[0]
    law = _filtered_first_token_law(lp, lq, top_k, top_p)
    assert np.max(np.abs(law - pf)) < 2.0 * V / M
    # verifying a filtered draft against the unfiltered target gives a different law
    off = _filtered_first_token_law(lp, lq, top_k, top_p, verify_filter=False)
    assert np.max(np.abs(off - pf)) > 1e-3


def test_drafter_top_k_draws_follow_the_top_k_softmax():
    """The input generator's drafter-side top-k draw (bench workload topkp64):
    only the top_k largest logits are drawn, each with its softmax
    probability renormalised over them (frequencies within 4 sigma)."""
    rng = np.random.default_rng(11)
    row = workloads.bf16_bits(np.array([0.5, 2.0, -1.0, 1.25, 3.0, 0.0], np.float32))
    T, top_k, n = 0.8, 3, 60_000
    draws = np.array([workloads.gumbel_draw_top_k(rng, row, T, top_k) for _ in range(n)])
    assert set(np.unique(draws)) <= {1, 3, 4}
    z = np.array([2.0, 1.25, 3.0]) / T
    p = np.exp(z - z.max())
    p /= p.sum()
    freq = np.array([(draws == v).mean() for v in (1, 3, 4)])
    assert np.all(np.abs(freq - p) <= 4 * np.sqrt(p * (1 - p) / n)), (freq, p)
    # a tie at the cut takes the lower position
    tie = workloads.bf16_bits(np.array([1.0, 5.0, 1.0, 1.0], np.float32))
    assert {workloads.gumbel_draw_top_k(rng, tie, 1.0, 2) for _ in range(200)} <= {0, 1}


def test_per_row_top_p_filters_each_row_with_its_own_mass():
    """verify_sample's per-row top_p: filled with top_p it is the scalar form
    bit for bit; a different value on one row changes that row's filter alone
    (its p(x) is the filtered row's at that mass, every other row's is
    unchanged)."""
    rng = np.random.default_rng(5)
    B, k, V, T = 3, 3, 40, 0.9
    t = (rng.standard_normal((B, k + 1, V)) * 2).astype(np.float32)
    d = (t[:, :k] + rng.standard_normal((B, k, V))).astype(np.float32)
    x = rng.integers(0, V, (B, k)).astype(np.int32)
    u = np.full((B, k + 1), 0.999, np.float32)
    u[:, 0] = 0.0                                     # position 0 accepted whenever p(x) > 0
    top_k, top_p = 15, 0.8
    a = oracle.verify_sample(t, d, x, u, T, top_k=top_k, top_p=top_p)
    b = oracle.verify_sample(t, d, x, u, T, top_k=top_k, top_p=top_p, top_p_rows=np.full((B, 2 * k + 1), top_p))
    for key in ("accepted", "out_tokens", "n_emit", "p_tok", "q_tok", "resid_mass"):
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)
    tp = np.full((B, 2 * k + 1), top_p)
    tp[1, 1] = 0.3                                    # target row 1 of request 1
    tp[2, k + 1 + 2] = 0.5                            # draft row 2 of request 2
    c = oracle.verify_sample(t, d, x, u, T, top_k=top_k, top_p=top_p, top_p_rows=tp)
    assert c["p_tok"][1, 1] == oracle.filter_row(t[1, 1], T, top_k, 0.3)[0][x[1, 1]]
    assert c["q_tok"][2, 2] == oracle.filter_row(d[2, 2], T, top_k, 0.5)[0][x[2, 2]]
    same = np.ones((B, k), bool)
    same[1, 1] = False
    np.testing.assert_array_equal(c["p_tok"][same], a["p_tok"][same])
    same = np.ones((B, k), bool)
    same[2, 2] = False
    np.testing.assert_array_equal(c["q_tok"][same], a["q_tok"][same])
    assert oracle.filter_row(t[1, 1], T, top_k, 0.3)[2] < oracle.filter_row(t[1, 1], T, top_k, top_p)[2]
