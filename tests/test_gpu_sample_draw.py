"""GPU parity of spec_sample (the drafter-side draw x ~ softmax(row / T))
against the oracle's draw, on both chain paths and on every accept kernel
the shapes reach: the token is the oracle's except where u lies within 1e-5
of a CDF boundary (counted), and the returned probability is the oracle's
softmax at the drawn token within 1e-5.  200,000 draws from one row follow
the row's distribution (total variation at sampling noise).
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_02_gb300 import api, workloads
from tests.parity import TOL, _near_draw, host, to_dev

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


def _problem(seed, B, V, dtype, std=2.0, stride_pad=0):
    rng = np.random.default_rng(seed)
    x = rng.normal(0.0, std, (B, V + stride_pad)).astype(np.float32)
    x[:, rng.integers(0, V, 3)] += 6.0
    if dtype == "bf16":
        x = workloads.bf16_bits(x)
    u = rng.random(B, dtype=np.float32)
    return x, u


def _check(x, V, u, T, g):
    B = u.size
    near = 0
    for b in range(B):
        p = oracle.softmax(x[b, :V], T)
        r = oracle.verify_sample(np.ascontiguousarray(x[b:b + 1, None, :V]), np.zeros((1, 0, V), x.dtype),
                                 np.zeros((1, 0), np.int32), u[b:b + 1, None], T)
        rt, gt = int(r["out_tokens"][0, 0]), int(g["tokens"][b])
        if rt != gt:
            assert _near_draw(p, float(u[b]), rt, gt), (b, rt, gt)
            near += 1
        assert g["status"][b] == 0
        assert abs(g["probs"][b] - p[gt]) <= TOL, (b, g["probs"][b], p[gt])
    return near


@pytest.mark.parametrize("seed,B,V,dtype,T,pad", [(1, 1, 248_320, "bf16", 1.0, 0), (2, 64, 128_256, "bf16", 0.7, 0),
                                                  (3, 400, 3001, "fp32", 1.0, 0), (4, 3, 7, "fp32", 0.3, 0),
                                                  (5, 16, 32_000, "fp32", 1.3, 3), (6, 5, 1, "bf16", 1.0, 0),
                                                  (7, 9, 40_003, "bf16", 2.0, 1)])
def test_sample_parity(seed, B, V, dtype, T, pad):
    x, u = _problem(seed, B, V, dtype, stride_pad=pad)
    logits = to_dev(x)[:, :V]             # pad > 0: rows longer than V (odd strides take the scalar path)
    g = api.spec_sample(logits, to_dev(u), T)
    g["tokens"].fill_(-7), g["probs"].fill_(-7.0)
    g = host(api.spec_sample(logits, to_dev(u), T, out=g))
    near = _check(x, V, u, T, g)
    print("near-threshold draws", near)
    if V == 1:
        assert (g["tokens"] == 0).all() and np.allclose(g["probs"], 1.0)


def test_draws_follow_the_distribution():
    """200,000 draws from one V=2048 row with fresh uniforms: TV to the row's
    softmax at sampling noise (the row broadcast with a zero request stride)."""
    prob = workloads.chain_small()
    row = prob["draft_logits"][0, 0]
    V, n = row.size, 200_000
    q = oracle.softmax(row, 1.0)
    u = np.random.default_rng(99).random(n, dtype=np.float32)
    g = host(api.spec_sample(to_dev(row)[None].expand(n, V), to_dev(u), 1.0))
    tv = 0.5 * np.abs(np.bincount(g["tokens"], minlength=V) / n - q).sum()
    noise = 0.5 * np.sum(np.sqrt(2 * q * (1 - q) / (np.pi * n)))
    assert tv < 1.2 * noise, (tv, noise)
    assert np.abs(g["probs"] - q[g["tokens"]]).max() <= TOL
