"""Host analysis helpers: the oracle's restatement pinned by the pages and by
simulation, and the library's native helpers (spec_expected_tokens,
spec_speedup, spec_best_k, spec_alpha_estimate) against the oracle.  No GPU
is needed: the helpers are host code.

Pins:
- the page's worked value: alpha = 0.8, draft cost c = 0, k = 1 gives exactly
  1.8 tokens per round ("投机解码", the third experiment);
- with c = 0 the speedup is the expected tokens per round, and a longer draft
  never hurts (best k = k_max); with c >= 1 no draft pays (best k = 0);
- a simulated decoder (Bernoulli(alpha) positions, draft forwards costing c
  each, one target forward per round) finds the same best k and its tokens
  per unit cost match the speedup within sampling error;
- the alpha estimate on a hand-counted example, and on simulated rounds
  (within 4 standard errors of the true alpha).
"""
import numpy as np
import pytest

from oracle.analysis import alpha_estimate, best_k, expected_tokens_per_round, speedup
from speculative_decoding_verification_02_gb300 import api


def _simulate(alpha, k, c, rounds, rng):
    """Tokens per unit of cost for a decoder whose positions are accepted
    independently with probability alpha (rounds stop at the first rejection)."""
    ok = rng.random((rounds, k)) < alpha if k else np.zeros((rounds, 0), bool)
    m = np.where(ok.all(axis=1), k, np.argmin(ok, axis=1)) if k else np.zeros(rounds, int)
    tokens = (m + 1).sum()
    cost = rounds * (k * c + 1.0)
    return tokens / cost, m


def test_page_value_and_zero_cost():
    assert speedup(0.8, 1, 0.0) == pytest.approx(1.8, abs=1e-12)
    for a in (0.0, 0.3, 0.75, 0.99, 1.0):
        for k in range(0, 9):
            assert speedup(a, k, 0.0) == pytest.approx(expected_tokens_per_round(a, k), rel=1e-12)
    assert best_k(0.6, 0.0, 12)[0] == 12
    assert best_k(0.95, 1.0, 12) == (0, 1.0)
    assert best_k(1.0, 1.0, 12) == (0, 1.0)      # every k ties at 1: the shorter draft


@pytest.mark.parametrize("alpha,c", [(0.6, 0.2), (0.8, 0.05), (0.5, 0.3)])
def test_simulated_decoder_agrees(alpha, c):
    rng = np.random.default_rng(int(alpha * 100 + c * 10))
    rates = []
    for k in range(0, 7):
        r, _ = _simulate(alpha, k, c, 200_000, rng)
        rates.append(r)
        assert r == pytest.approx(speedup(alpha, k, c), rel=0.01)
    assert int(np.argmax(rates)) == best_k(alpha, c, 6)[0]


def test_alpha_estimate_pins():
    assert alpha_estimate([0, 2, 4], k=4) == (0.75, 8)          # 6 accepted of 1 + 3 + 4 tested
    assert alpha_estimate([1, 3], draft_len=[1, 5]) == (0.8, 5)  # a full accept of L=1 tests 1
    rng = np.random.default_rng(5)
    for alpha in (0.3, 0.7, 0.9):
        _, m = _simulate(alpha, 4, 0.0, 50_000, rng)
        a, tests = alpha_estimate(m, k=4)
        assert abs(a - alpha) < 4 * np.sqrt(alpha * (1 - alpha) / tests)


def test_library_matches_oracle():
    rng = np.random.default_rng(7)
    for a in (0.0, 0.2, 0.5, 0.8, 0.97, 1.0):
        for k in (0, 1, 2, 4, 8, 16):
            assert api.expected_tokens(a, k) == pytest.approx(expected_tokens_per_round(a, k), rel=1e-12, abs=1e-12)
            for c in (0.0, 0.05, 0.3, 1.0, 2.5):
                assert api.speedup(a, k, c) == pytest.approx(speedup(a, k, c), rel=1e-12)
        for c in (0.0, 0.02, 0.1, 0.3, 1.0):
            kb, sb = api.best_k(a, c, 20)
            ko, so = best_k(a, c, 20)
            assert kb == ko and sb == pytest.approx(so, rel=1e-12)
    for _ in range(20):
        n, k = int(rng.integers(1, 50)), int(rng.integers(0, 9))
        L = rng.integers(0, k + 1, n)
        m = np.array([rng.integers(0, l + 1) for l in L])
        got = api.alpha_estimate(m, L, k)
        want = alpha_estimate(m, L, k)
        assert got[1] == want[1]
        assert (np.isnan(got[0]) and np.isnan(want[0])) or got[0] == pytest.approx(want[0], rel=1e-15)


def test_library_argument_checks():
    for bad in (lambda: api.expected_tokens(-0.1, 2), lambda: api.expected_tokens(0.5, -1),
                lambda: api.speedup(1.5, 2, 0.1), lambda: api.speedup(0.5, 2, -1.0),
                lambda: api.speedup(0.5, 2, float("nan")), lambda: api.best_k(0.5, 0.1, -1),
                lambda: api.alpha_estimate([3], [2], 4), lambda: api.alpha_estimate([-1], None, 4)):
        with pytest.raises(api.SpecError):
            bad()
    a, t = api.alpha_estimate([], None, 4)
    assert np.isnan(a) and t == 0
