"""Pins for sampling chain verification.

T-d  with the same p, q at every position the acceptances are i.i.d. with
     alpha = sum min(p, q), so tokens per round average
     (1 - alpha^(k+1)) / (1 - alpha); alpha = 0.8, k = 1 gives 1.8.
T-e  the emitted first token is distributed exactly as p.  The oracle is a
     deterministic function of the uniforms, so scanning one uniform over a
     2^16-point grid (the others held to force the branch) measures each
     acceptance threshold and the residual draw to 2^-16; composing them over
     the draft token gives p to ~1e-4.  The resample-from-p negative control
     must instead show the bias min(p,q) - alpha p.
T-f  200,000 draws on a V=2048 row: the lossless rule's total-variation
     distance to p is at sampling-noise level; resampling from p after a
     rejection shows its closed-form bias; the naive "keep only if equal"
     rule accepts with probability sum p q.
"""
import numpy as np
import pytest

import oracle
from oracle.analysis import expected_tokens_per_round
from speculative_decoding_verification_02_gb300 import workloads

M = 1 << 16
U_REJECT = np.float32(1.0 - 2.0 ** -24)     # largest float32 below 1: rejects unless p >= q


def _softmax64(x):
    z = np.asarray(x, np.float64)
    e = np.exp(z - z.max())
    return e / e.sum()


def _rows(p, q):
    return np.log(p).astype(np.float32), np.log(q).astype(np.float32)


def test_closed_form_values():
    assert expected_tokens_per_round(0.8, 1) == pytest.approx(1.8, abs=1e-15)
    assert expected_tokens_per_round(0.0, 4) == 1.0
    assert expected_tokens_per_round(1.0, 4) == 5.0
    assert expected_tokens_per_round(0.5, 4) == pytest.approx(1.9375)


@pytest.mark.parametrize("k", [1, 2, 4, 8])
def test_tokens_per_round_match_closed_form(k):
    V, B = 8, 40_000
    rng = np.random.default_rng(100 + k)
    lp, lq = _rows(rng.dirichlet(np.ones(V)), rng.dirichlet(np.ones(V)))
    p, q = _softmax64(lp), _softmax64(lq)
    alpha = np.minimum(p, q).sum()
    target = np.broadcast_to(lp, (B, k + 1, V))
    draft_logits = np.broadcast_to(lq, (B, k, V))
    draft = rng.choice(V, size=(B, k), p=q).astype(np.int32)
    u = rng.random((B, k + 1), dtype=np.float32)
    out = oracle.verify_sample(target, draft_logits, draft, u, T=1.0, threads=4)
    tokens = out["n_emit"].astype(np.float64)
    sigma = tokens.std() / np.sqrt(B)
    assert abs(tokens.mean() - expected_tokens_per_round(alpha, k)) < 4 * sigma
    # the accepted count is geometric, truncated at k
    hist = np.bincount(out["accepted"], minlength=k + 1) / B
    expect = np.array([alpha ** j * (1 - alpha) for j in range(k)] + [alpha ** k])
    assert np.max(np.abs(hist - expect)) < 5 * np.sqrt(0.25 / B)


def _first_token_law(lp, lq, T, variant):
    """Exact law of the first emitted token, measured threshold by threshold."""
    V = lp.size
    grid = (np.arange(M, dtype=np.float64) / M).astype(np.float32)
    law = np.zeros(V)
    qd = _softmax64(lq.astype(np.float64) / T)
    for x in range(V):
        # acceptance threshold of draft token x: scan u0
        u = np.stack([grid, np.full(M, 0.5, np.float32)], 1)
        out = oracle.verify_sample(np.broadcast_to(lp, (M, 2, V)), np.broadcast_to(lq, (M, 1, V)),
                                   np.full((M, 1), x, np.int32), u, T=T, variant=variant, threads=4)
        acc = out["accepted"].mean()
        law[x] += qd[x] * acc
        if acc == 1.0:
            continue
        # the draw after a rejection: force the rejection, scan the last uniform
        u = np.stack([np.full(M, U_REJECT, np.float32), grid], 1)
        out = oracle.verify_sample(np.broadcast_to(lp, (M, 2, V)), np.broadcast_to(lq, (M, 1, V)),
                                   np.full((M, 1), x, np.int32), u, T=T, variant=variant, threads=4)
        assert np.all(out["accepted"] == 0)
        law += qd[x] * (1.0 - acc) * np.bincount(out["out_tokens"][:, 0], minlength=V) / M
    return law


@pytest.mark.parametrize("V,T,seed", [(2, 1.0, 0), (3, 1.0, 1), (4, 0.7, 2), (4, 1.0, 3)])
def test_first_token_is_exactly_p(V, T, seed):
    rng = np.random.default_rng(seed)
    lp = (rng.standard_normal(V) * 1.5).astype(np.float32)
    lq = (lp + rng.standard_normal(V)).astype(np.float32)
    p = _softmax64(lp.astype(np.float64) / T)
    q = _softmax64(lq.astype(np.float64) / T)
    law = _first_token_law(lp, lq, T, oracle.VARIANT_LOSSLESS)
    assert np.max(np.abs(law - p)) < 2.0 * V / M
    # negative control: resampling from p after a rejection gives
    # min(p, q) + (1 - alpha) p, off from p by min(p, q) - alpha p
    bad = _first_token_law(lp, lq, T, oracle.VARIANT_RESAMPLE_FROM_P)
    alpha = np.minimum(p, q).sum()
    assert np.max(np.abs(bad - (np.minimum(p, q) + (1 - alpha) * p))) < 2.0 * V / M
    assert np.max(np.abs(bad - p)) > 1e-3


def test_per_token_probabilities_and_residual_mass():
    prob = workloads.chain_small()
    out = oracle.verify_sample(prob["target"], prob["draft_logits"], prob["draft"], prob["uniforms"], prob["T"])
    for b in range(prob["B"]):
        for i in range(prob["k"]):
            p = _softmax64(prob["target"][b, i].astype(np.float64) / prob["T"])
            q = _softmax64(prob["draft_logits"][b, i].astype(np.float64) / prob["T"])
            x = prob["draft"][b, i]
            assert out["p_tok"][b, i] == pytest.approx(p[x], rel=1e-12, abs=1e-300)
            assert out["q_tok"][b, i] == pytest.approx(q[x], rel=1e-12, abs=1e-300)
        m = out["accepted"][b]
        if m < prob["k"]:
            p = _softmax64(prob["target"][b, m].astype(np.float64))
            q = _softmax64(prob["draft_logits"][b, m].astype(np.float64))
            assert out["resid_mass"][b] == pytest.approx(1.0 - np.minimum(p, q).sum(), abs=1e-12)
        else:
            assert out["resid_mass"][b] == 0.0


def _tv(counts, p):
    return 0.5 * np.abs(counts / counts.sum() - p).sum()


def test_total_variation_200k_draws():
    """'投机解码:为什么一个字都不改', section 改进方案: on V=2048 and 200,000
    draws the lossless rule sits at sampling noise, resampling from p does not."""
    prob = workloads.chain_small()
    lp, lq = prob["target"][0, 0], prob["draft_logits"][0, 0]
    lbonus = prob["target"][0, 1]
    V, n = lp.size, 200_000
    p, q = _softmax64(lp), _softmax64(lq)
    rng = np.random.default_rng(2048)
    draft = rng.choice(V, size=(n, 1), p=q).astype(np.int32)
    u = rng.random((n, 2), dtype=np.float32)
    target = np.broadcast_to(np.stack([lp, lbonus]), (n, 2, V))
    dl = np.broadcast_to(lq, (n, 1, V))
    noise = 0.5 * np.sum(np.sqrt(2 * p * (1 - p) / (np.pi * n)))   # E[TV] of n direct draws

    good = oracle.verify_sample(target, dl, draft, u, threads=8)
    tv_good = _tv(np.bincount(good["out_tokens"][:, 0], minlength=V), p)
    tv_direct = _tv(np.bincount(rng.choice(V, size=n, p=p), minlength=V), p)
    assert tv_good < 1.2 * noise and tv_direct < 1.2 * noise
    assert abs(tv_good - tv_direct) < 0.25 * noise

    wrong = oracle.verify_sample(target, dl, draft, u, variant=oracle.VARIANT_RESAMPLE_FROM_P, threads=8)
    alpha = np.minimum(p, q).sum()
    theory = 0.5 * np.abs(np.minimum(p, q) - alpha * p).sum()
    pw = np.minimum(p, q) + (1 - alpha) * p
    noise_w = 0.5 * np.sum(np.sqrt(2 * pw * (1 - pw) / (np.pi * n)))
    tv_wrong = _tv(np.bincount(wrong["out_tokens"][:, 0], minlength=V), p)
    assert abs(tv_wrong - theory) < 1.3 * noise_w
    assert tv_wrong > 3 * noise

    naive = oracle.verify_sample(target, dl, draft, u, variant=oracle.VARIANT_NAIVE_EQUAL, threads=8)
    rate = (naive["accepted"] > 0).mean()
    pq = float(np.sum(p * q))
    assert abs(rate - pq) < 5 * np.sqrt(pq * (1 - pq) / n)
