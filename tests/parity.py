"""Helpers for comparing the CUDA library with the fp64 oracle.

Decision rule for sampled outputs: accept counts and emitted tokens must be
identical to the oracle's, except where the uniform lies within TOL of the
threshold the oracle computed in fp64 (for an accept test: u vs min(1, p/q);
for a draw: u vs the normalised CDF at the boundary between the two picks).
Such cases are counted and reported, not failed.  Per-token probabilities
must agree to TOL absolute.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

TOL = 1e-5


def to_dev(x, device="cuda"):
    """numpy fp32 / bf16-bits (uint16) / int32 / float32 -> torch tensor on device."""
    x = np.ascontiguousarray(x)
    if x.dtype == np.uint16:
        return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(x).to(device)


def host(o: dict) -> dict:
    return {k: v.cpu().numpy() for k, v in o.items()}


def poison_like(o: dict):
    """Fill output tensors with -7 so an unwritten slot cannot pass."""
    for v in o.values():
        v.fill_(-7)
    return o


def _near_draw(dist, u, a, b, tol=TOL):
    lo, hi = min(a, b), max(a, b)
    if lo < 0 or hi >= dist.size:
        return False
    cdf = np.cumsum(dist)
    return abs(u - cdf[lo]) < tol and abs(u - cdf[hi - 1]) < tol


def check_chain_sample(prob, gpu: dict, orc: dict, draft_len=None, tol=TOL) -> dict:
    """Asserts the decision rule; returns counters."""
    B, k, T = prob["target"].shape[0], prob["target"].shape[1] - 1, prob["T"]
    u = prob["uniforms"]
    near_accept = near_draw = 0
    np.testing.assert_array_equal(gpu["status"], orc["status"])
    for b in range(B):
        L = k if draft_len is None else int(draft_len[b])
        if orc["status"][b] != 0:
            assert gpu["n_emit"][b] == 0 and np.all(gpu["out_tokens"][b] == -1)
            continue
        pt, qt = orc["p_tok"][b], orc["q_tok"][b]
        if "p_tok" in gpu:
            assert np.all(np.abs(gpu["p_tok"][b, :L] - pt[:L]) <= tol), (b, gpu["p_tok"][b], pt)
            assert np.all(np.abs(gpu["q_tok"][b, :L] - qt[:L]) <= tol), (b, gpu["q_tok"][b], qt)
            assert np.all(gpu["p_tok"][b, L:] == -1.0) and np.all(gpu["q_tok"][b, L:] == -1.0)
        mg, mo = int(gpu["accepted"][b]), int(orc["accepted"][b])
        if mg != mo:
            i = min(mg, mo)
            thr = min(1.0, pt[i] / qt[i]) if qt[i] > 0 else 1.0
            assert abs(float(u[b, i]) - thr) < tol, f"request {b}: accepted {mg} vs oracle {mo}"
            near_accept += 1
            continue
        assert gpu["n_emit"][b] == orc["n_emit"][b]
        ne = int(orc["n_emit"][b])
        np.testing.assert_array_equal(gpu["out_tokens"][b, :mo], orc["out_tokens"][b, :mo])
        assert np.all(gpu["out_tokens"][b, ne:] == -1)
        if "resid_mass" in gpu:
            assert abs(gpu["resid_mass"][b] - orc["resid_mass"][b]) <= tol, b
        if mo < ne and gpu["out_tokens"][b, mo] != orc["out_tokens"][b, mo]:
            p = oracle.softmax(prob["target"][b, mo], T)
            if mo < L:
                q = oracle.softmax(prob["draft_logits"][b, mo], T)
                dist, R = oracle.residual(p, q)
                if R <= 0.0:
                    dist = p
            else:
                dist = p
            assert _near_draw(dist, float(u[b, k]), int(gpu["out_tokens"][b, mo]),
                              int(orc["out_tokens"][b, mo]), tol), f"request {b}: final token differs"
            near_draw += 1
    return dict(near_accept=near_accept, near_draw=near_draw)


def check_tree(prob, gpu: dict, orc: dict, tol=TOL, without_replacement=False) -> dict:
    """Tree outputs must match the oracle exactly, except when a decision on the
    oracle's own path was within tol of its fp64 threshold.  without_replacement:
    the walk also removes each rejected sibling's token from q."""
    B, N = prob["parents"].shape
    T = prob["T"]
    near = 0
    np.testing.assert_array_equal(gpu["status"], orc["status"])
    for b in range(B):
        same = (gpu["n_emit"][b] == orc["n_emit"][b] and
                np.array_equal(gpu["out_tokens"][b], orc["out_tokens"][b]) and
                np.array_equal(gpu["path_nodes"][b], orc["path_nodes"][b]) and
                gpu["accepted_len"][b] == orc["accepted_len"][b])
        if same:
            continue
        assert T > 0, f"greedy tree walk differs on request {b}"
        assert _tree_near_threshold(prob, b, gpu, orc, tol, without_replacement), f"tree request {b} differs"
        near += 1
    return dict(near=near)


def _tree_near_threshold(prob, b, gpu, orc, tol, without_replacement=False):
    """Replays the oracle's walk in fp64 up to the first divergence and checks
    that the diverging decision was within tol of its threshold."""
    par, tok, u = prob["parents"][b], prob["node_tok"][b], prob["uniforms"][b]
    N, T = par.size, prob["T"]
    node = 0
    depth = 0
    while True:
        p = oracle.softmax(prob["target"][b, node], T)
        kids = [c for c in range(node + 1, N) if par[c] == node]
        q = oracle.softmax(prob["draft_logits"][b, node], T) if kids else None
        nxt = -1
        for c in kids:
            x = tok[c]
            thr = min(1.0, p[x] / q[x]) if q[x] > 0 else float(p[x] > 0)
            if abs(float(u[c]) - thr) < tol:
                return True
            if u[c] < thr:
                nxt = c
                break
            r, R = oracle.residual(p, q)
            if R > 0:
                p = r
                if without_replacement:
                    q = q.copy()
                    q[x] = 0.0
                    Q = q.sum()
                    q = q / Q if Q > 0 else np.zeros_like(q)
        g_next = int(gpu["path_nodes"][b, depth + 1]) if depth + 1 < gpu["path_nodes"].shape[1] else -1
        if nxt < 0:
            a, bb = int(gpu["out_tokens"][b, depth]), int(orc["out_tokens"][b, depth])
            return g_next == -1 and _near_draw(p, float(u[N]), a, bb, tol)
        if g_next != nxt:
            return False
        node = nxt
        depth += 1
