"""Pins for the oracle's row-level building blocks: softmax(x/T), argmax,
inverse CDF and the residual norm(max(0, p - q)).

Each check compares the oracle with a closed form or a special case that does
not go through the oracle's own code: softmax of T*log(w) is w/sum(w), a
two-logit softmax is a logistic function, constant logits give the uniform
distribution, bf16 bit patterns decode to known values.
"""
import math

import numpy as np
import pytest

import oracle
from speculative_decoding_verification_02_gb300.workloads import bf16_bits, bf16_to_f32


def test_softmax_uniform_for_constant_logits():
    for V in (1, 2, 7, 2048):
        p = oracle.softmax(np.full(V, 3.25, np.float32), T=0.7)
        assert np.all(p == pytest.approx(1.0 / V, abs=1e-15))


@pytest.mark.parametrize("T", [0.5, 0.7, 1.0, 2.0])
def test_softmax_of_scaled_log_weights_is_the_weights(T):
    # softmax((T * log w) / T) = w / sum(w); the only error is fp32 rounding of T*log w
    rng = np.random.default_rng(7)
    w = rng.uniform(0.05, 1.0, size=64)
    x = (T * np.log(w)).astype(np.float32)
    expect = np.exp(x.astype(np.float64) / T)
    expect /= expect.sum()
    assert np.max(np.abs(oracle.softmax(x, T) - w / w.sum())) < 1e-6
    assert np.max(np.abs(oracle.softmax(x, T) - expect)) < 1e-15


def test_softmax_two_logits_is_logistic():
    for a, b, T in [(0.0, 1.0, 1.0), (2.5, -1.0, 0.7), (10.0, 10.0, 3.0)]:
        p = oracle.softmax(np.array([a, b], np.float32), T)
        p0 = 1.0 / (1.0 + math.exp((b - a) / T))
        assert p[0] == pytest.approx(p0, rel=1e-14)
        assert p[1] == pytest.approx(1.0 - p0, rel=1e-13, abs=1e-300)


def test_softmax_large_logits_stay_finite():
    p = oracle.softmax(np.array([1000.0, 1000.0, 0.0], np.float32), 1.0)
    assert p[0] == pytest.approx(0.5) and p[1] == pytest.approx(0.5) and p[2] < 1e-300


def test_softmax_reads_bf16_bits():
    # 0x3F80 = 1.0, 0x0000 = 0.0, 0xC000 = -2.0 in bf16
    bits = np.array([0x3F80, 0x0000, 0xC000], np.uint16)
    e = np.exp([1.0, 0.0, -2.0])
    np.testing.assert_allclose(oracle.softmax(bits, 1.0), e / e.sum(), rtol=1e-14)


def test_bf16_rounding_is_nearest_even():
    # 1 + 2^-8 is halfway between bf16 neighbours 1 and 1 + 2^-7: ties to even (1.0)
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.0, 3.0e38], np.float32)
    back = bf16_to_f32(bf16_bits(x))
    assert back[0] == 1.0 and back[1] == 1.0 and back[2] == np.float32(1.0 + 2 ** -6)
    assert back[3] == -2.0 and np.isfinite(back[4])


def test_argmax_lowest_index_on_ties():
    assert oracle.argmax(np.array([1, 5, 5, 2], np.float32)) == 1
    assert oracle.argmax(np.array([-0.0, 0.0], np.float32)) == 0   # -0 == +0: a tie
    assert oracle.argmax(np.array([7.0], np.float32)) == 0
    bits = bf16_bits(np.array([0.5, 3.0, -1.0, 3.0], np.float32))
    assert oracle.argmax(bits) == 1
    x = np.zeros(100_000, np.float32)
    x[[123, 99_999, 777]] = 2.0
    assert oracle.argmax(x) == 123


def test_inverse_cdf_definition():
    d = np.array([0.25, 0.25, 0.5])
    assert oracle.inverse_cdf(d, 0.0) == 0
    assert oracle.inverse_cdf(d, 0.1) == 0
    assert oracle.inverse_cdf(d, 0.25) == 1      # prefix must EXCEED u
    assert oracle.inverse_cdf(d, 0.7) == 2
    z = np.array([0.0, 0.5, 0.0, 0.5])
    assert oracle.inverse_cdf(z, 0.0) == 1       # zero-mass entries are never drawn
    assert oracle.inverse_cdf(z, 0.5) == 3
    # rounding fallback: u at or above the total -> last entry with mass
    assert oracle.inverse_cdf(np.array([0.5, 0.5, 0.0]), 1.0) == 1


def test_inverse_cdf_frequencies_match_distribution():
    d = np.array([0.1, 0.0, 0.6, 0.3])
    M = 4096
    hits = np.bincount([oracle.inverse_cdf(d, (j + 0.5) / M) for j in range(M)], minlength=4)
    np.testing.assert_allclose(hits / M, d, atol=1.0 / M)


@pytest.mark.parametrize("V", [2, 3, 5, 16])
def test_residual_identity(V):
    # min(p, q) + (1 - alpha) * norm(max(0, p - q)) = p, alpha = sum min(p, q)
    # ("投机解码:为什么一个字都不改", section 改进方案, Leviathan et al. App. A.1)
    rng = np.random.default_rng(V)
    for _ in range(50):
        p, q = rng.dirichlet(np.ones(V)), rng.dirichlet(np.ones(V))
        r, R = oracle.residual(p, q)
        alpha = np.minimum(p, q).sum()
        assert R == pytest.approx(1.0 - alpha, abs=1e-15)
        np.testing.assert_allclose(np.minimum(p, q) + R * r, p, atol=1e-15)
        assert np.all(r >= 0.0) and r.sum() == pytest.approx(1.0, abs=1e-14)
        assert np.all(r[p <= q] == 0.0)


def test_residual_of_equal_distributions_is_empty():
    p = np.array([0.2, 0.3, 0.5])
    r, R = oracle.residual(p, p)
    assert R == 0.0 and np.all(r == 0.0)
