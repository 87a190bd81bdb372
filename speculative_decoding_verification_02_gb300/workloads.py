"""Seeded synthetic inputs for the verification workloads.

This module is the one thing the oracle and the CUDA path share.  It holds
none of the verification arithmetic: it draws logits, trees, histories and
uniforms with numpy's counter-free PCG64 streams (bit-identical on x86 and
Arm), rounds logits to bf16 with round-to-nearest-even, and draws each draft
token from the draft distribution with the Gumbel-max trick (the drafter's
own sampling, which happens before verification and is not part of it).

Logits come back as numpy arrays: float32, or bf16 as its raw uint16 bits.

Workload recipes (stddev convention: N(mu, s) means standard deviation s):
  chain_small   B=4,  k=4, V=2048 fp32, t ~ N(0,2), d = t + N(0,0.5), T=1
  ngram         B=64, history 4096 int32 over V=32000, 4-8 planted repeated
                spans of length 8-32, half the requests end inside a copy of
                an earlier span; window 3, k=4; target N(0,1) fp32 [64,5,V]
  chain_vocab248k  B=1, k=4, V=248320 bf16, t ~ N(0,3) with 5 random ids
                per row raised by 8, d = 0.8 t + N(0,1), T=1
  chain_batch64 B=64, k=8, V=128256 bf16, t ~ N(0,2.5), d = t + N(0,s_b)
                with s_b = (0.3, 1, 2)[b mod 3], T=0.7
  tree60        B=16, N=60 nodes (root included), depth 6, <=10 children,
                V=128256 bf16 target/draft rows per node drawn as in
                chain_vocab248k, child tokens i.i.d. from the parent's q, T=1
  eagle2_candidates  B=16 candidate trees grown layer by layer as in
                EAGLE-2's expansion stage: the root gets `branch` children,
                then for depth-1 more layers `expand` nodes of the newest
                layer each get `branch` children (the expanded nodes are a
                random subset here); a node's confidences are the sorted
                first `branch` weights of a Dirichlet(0.5) draw over
                branch + 1 outcomes (the last standing for the rest of the
                vocabulary), tokens uniform over [0, V).  Defaults: depth 6,
                expand 10, branch 10 -> N = 511 nodes; m = 60 kept
"""
from __future__ import annotations

import numpy as np

SEED_BASE = 20260000


def _rngs(seed: int, n: int):
    return [np.random.Generator(np.random.PCG64(s)) for s in np.random.SeedSequence(seed).spawn(n)]


def bf16_bits(x) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return the bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16_to_f32(bits) -> np.ndarray:
    """Exact widening of bf16 bits to float32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def logits_as_f64(x) -> np.ndarray:
    x = np.asarray(x)
    return bf16_to_f32(x).astype(np.float64) if x.dtype == np.uint16 else x.astype(np.float64)


def _store(x32: np.ndarray, dtype: str) -> np.ndarray:
    return bf16_bits(x32) if dtype == "bf16" else np.ascontiguousarray(x32, dtype=np.float32)


def gumbel_draw(rng, logits_row, T: float) -> int:
    """One draw from softmax(logits/T) by Gumbel-max: argmax(l/T + G), G Gumbel(0,1)."""
    u = rng.random(logits_row.shape[-1])
    u = np.where(u <= 0.0, np.finfo(np.float64).tiny, u)
    return int(np.argmax(logits_as_f64(logits_row) / T - np.log(-np.log(u))))


def gumbel_draw_top_k(rng, logits_row, T: float, top_k: int) -> int:
    """A drafter that samples from its own top-k: Gumbel-max over exactly
    top_k logits, the largest (equal logits at the cut taken by position).
    Without ties at the cut this is a draw from the top-k filtered softmax."""
    l64 = logits_as_f64(logits_row)
    cand = np.argsort(-l64, kind="stable")[:top_k]
    u = rng.random(top_k)
    u = np.where(u <= 0.0, np.finfo(np.float64).tiny, u)
    return int(cand[np.argmax(l64[cand] / T - np.log(-np.log(u)))])


def gumbel_top(rng, logits_row, T: float, n: int) -> np.ndarray:
    """n draws from softmax(logits/T) without replacement, in draw order: the
    n largest of l/T + G (Gumbel-top-k), the largest first."""
    if n > logits_row.shape[-1]:
        raise ValueError("more draws without replacement than tokens")
    u = rng.random(logits_row.shape[-1])
    u = np.where(u <= 0.0, np.finfo(np.float64).tiny, u)
    keys = logits_as_f64(logits_row) / T - np.log(-np.log(u))
    return np.argsort(-keys, kind="stable")[:n].astype(np.int32)


def uniforms(rng, shape) -> np.ndarray:
    """Caller-supplied uniforms in [0, 1), float32."""
    u = rng.random(shape, dtype=np.float32)
    return np.minimum(u, np.float32(1.0) - np.float32(2.0 ** -24)).astype(np.float32)


# ------------------------------------------------------------------ chains

def chain_problem(seed: int, B: int, k: int, V: int, dtype: str = "bf16", T: float = 1.0,
                  target_std: float = 1.0, draft_scale: float = 1.0, noise_std=0.5,
                  peaks: int = 0, peak_height: float = 0.0) -> dict:
    """A chain-verification problem.

    target t ~ N(0, target_std) (plus `peaks` random ids per row raised by
    peak_height), draft d = draft_scale * t + N(0, noise_std[b]); draft
    tokens x_i ~ softmax(d_i / T); uniforms [B, k+1].
    """
    r_t, r_n, r_x, r_u, r_p = _rngs(seed, 5)
    noise = np.broadcast_to(np.asarray(noise_std, dtype=np.float32), (B,))
    target = np.empty((B, k + 1, V), dtype=np.uint16 if dtype == "bf16" else np.float32)
    draft_logits = np.empty((B, k, V), dtype=target.dtype)
    draft = np.empty((B, k), dtype=np.int32)
    for b in range(B):
        for i in range(k + 1):
            t = r_t.standard_normal(V, dtype=np.float32) * np.float32(target_std)
            if peaks:
                t[r_p.choice(V, size=peaks, replace=False)] += np.float32(peak_height)
            target[b, i] = _store(t, dtype)
            if i < k:
                d = np.float32(draft_scale) * t + r_n.standard_normal(V, dtype=np.float32) * noise[b]
                draft_logits[b, i] = _store(d, dtype)
                draft[b, i] = gumbel_draw(r_x, draft_logits[b, i], T)
    return dict(target=target, draft_logits=draft_logits, draft=draft,
                uniforms=uniforms(r_u, (B, k + 1)), T=float(T), B=B, k=k, V=V, dtype=dtype)


def chain_small(seed: int = SEED_BASE + 1) -> dict:
    return chain_problem(seed, 4, 4, 2048, "fp32", 1.0, target_std=2.0, noise_std=0.5)


def chain_vocab248k(seed: int = SEED_BASE + 3, B: int = 1) -> dict:
    return chain_problem(seed, B, 4, 248320, "bf16", 1.0, target_std=3.0, draft_scale=0.8,
                         noise_std=1.0, peaks=5, peak_height=8.0)


def chain_batch64(seed: int = SEED_BASE + 4, B: int = 64) -> dict:
    sig = np.array([(0.3, 1.0, 2.0)[b % 3] for b in range(B)], dtype=np.float32)
    return chain_problem(seed, B, 8, 128256, "bf16", 0.7, target_std=2.5, noise_std=sig)


def chain_batch64_topk(seed: int = SEED_BASE + 8, B: int = 64, top_k: int = 50) -> dict:
    """The batch64 rows with each draft token redrawn by a drafter sampling
    from its own top-k (for top-k / top-p filtered verification)."""
    p = chain_batch64(B=B)
    rng = np.random.default_rng(seed)
    for b in range(p["B"]):
        for i in range(p["k"]):
            p["draft"][b, i] = gumbel_draw_top_k(rng, p["draft_logits"][b, i], p["T"], top_k)
    return p


# ------------------------------------------------------------------- trees

def random_tree(rng, N: int, depth: int, max_children: int) -> np.ndarray:
    """Parent array of a random tree: node 0 is the root (-1), a chain 0->depth
    is laid first so the depth is exact, the other nodes hang off random
    nodes of depth < `depth` that still have fewer than `max_children`."""
    parents = np.full(N, -1, dtype=np.int32)
    dep = np.zeros(N, dtype=np.int32)
    nchild = np.zeros(N, dtype=np.int32)
    for i in range(1, min(depth, N - 1) + 1):
        parents[i], dep[i] = i - 1, i
        nchild[i - 1] += 1
    for i in range(depth + 1, N):
        cand = [u for u in range(i) if dep[u] < depth and nchild[u] < max_children]
        u = int(cand[rng.integers(len(cand))])
        parents[i], dep[i] = u, dep[u] + 1
        nchild[u] += 1
    return parents


def tree_problem(seed: int, B: int, N: int, depth: int, max_children: int, V: int,
                 dtype: str = "bf16", T: float = 1.0, target_std: float = 3.0,
                 draft_scale: float = 0.8, noise_std: float = 1.0, peaks: int = 5,
                 peak_height: float = 8.0, siblings: str = "iid") -> dict:
    """A tree-verification problem: per request a random tree, per node a target
    and a draft row, child tokens drawn from the parent's draft q: i.i.d.
    (siblings="iid"), or one after another without replacement, in id order
    (siblings="without_replacement")."""
    if siblings not in ("iid", "without_replacement"):
        raise ValueError(siblings)
    r_tree, r_t, r_n, r_x, r_u, r_p = _rngs(seed, 6)
    store = np.uint16 if dtype == "bf16" else np.float32
    target = np.empty((B, N, V), dtype=store)
    draft_logits = np.empty((B, N, V), dtype=store)
    parents = np.empty((B, N), dtype=np.int32)
    node_tok = np.empty((B, N), dtype=np.int32)
    for b in range(B):
        parents[b] = random_tree(r_tree, N, depth, max_children)
        for u in range(N):
            t = r_t.standard_normal(V, dtype=np.float32) * np.float32(target_std)
            if peaks:
                t[r_p.choice(V, size=peaks, replace=False)] += np.float32(peak_height)
            target[b, u] = _store(t, dtype)
            d = np.float32(draft_scale) * t + r_n.standard_normal(V, dtype=np.float32) * np.float32(noise_std)
            draft_logits[b, u] = _store(d, dtype)
        node_tok[b, 0] = int(r_x.integers(V))  # the last committed token
        Tq = T if T > 0 else 1.0
        if siblings == "iid":
            for c in range(1, N):
                node_tok[b, c] = gumbel_draw(r_x, draft_logits[b, parents[b, c]], Tq)
        else:
            for u in range(N):
                kids = np.flatnonzero(parents[b] == u)
                if kids.size:
                    node_tok[b, kids] = gumbel_top(r_x, draft_logits[b, u], Tq, kids.size)
    return dict(target=target, draft_logits=draft_logits, parents=parents, node_tok=node_tok,
                uniforms=uniforms(r_u, (B, N + 1)), T=float(T), B=B, N=N, V=V, depth=depth,
                dtype=dtype, siblings=siblings)


def tree60(seed: int = SEED_BASE + 5, B: int = 16) -> dict:
    return tree_problem(seed, B, 60, 6, 10, 128256, "bf16", 1.0)


# ------------------------------------------------------------------ n-gram

def ngram_problem(seed: int, B: int = 64, H: int = 4096, V: int = 32000, k: int = 4,
                  window: int = 3, spans=(4, 8), span_len=(8, 32), boost: float = 0.0,
                  hist_len=None) -> dict:
    """History-lookup workload.

    Histories are i.i.d. uniform tokens with planted repeated spans; half the
    requests end inside a copy of an earlier span, so their last `window`
    tokens reappear earlier.  `planted_next[b]` lists the tokens that follow
    the planted source (-1 where there is none).  With boost > 0 the target
    logits of the first U[0, k] positions are raised at those tokens, so the
    greedy verifier sees acceptances; with boost = 0 the target is pure
    N(0,1) noise.
    """
    r_h, r_s, r_t, r_b = _rngs(seed, 4)
    hist = r_h.integers(0, V, size=(B, H), dtype=np.int64).astype(np.int32)
    if hist_len is None:
        hist_len = np.full(B, H, dtype=np.int32)
    hist_len = np.asarray(hist_len, dtype=np.int32)
    planted_next = np.full((B, k), -1, dtype=np.int32)
    for b in range(B):
        n = int(hist_len[b])
        h = hist[b]
        if n < 4 * span_len[1]:
            continue
        for _ in range(int(r_s.integers(spans[0], spans[1] + 1))):
            L = int(r_s.integers(span_len[0], span_len[1] + 1))
            src = int(r_s.integers(0, n // 2 - L))
            dst = int(r_s.integers(n // 2, n - L))
            h[dst:dst + L] = h[src:src + L]
        if b % 2 == 0:
            L = int(r_s.integers(span_len[0], span_len[1] + 1))
            j = int(r_s.integers(window, L))          # copy the first j tokens of the span
            src = int(r_s.integers(0, n // 2 - L))
            h[n - j:n] = h[src:src + j]
            cont = h[src + j:src + j + k]
            planted_next[b, :len(cont)] = cont
    target = r_t.standard_normal((B, k + 1, V), dtype=np.float32)
    if boost > 0.0:
        for b in range(B):
            a = int(r_b.integers(0, k + 1))
            for i in range(a):
                if planted_next[b, i] >= 0:
                    target[b, i, planted_next[b, i]] += np.float32(boost)
    return dict(history=hist, hist_len=hist_len, target=target, window=window, k=k, V=V,
                planted_next=planted_next, B=B, H=H)


def eagle2_candidates(seed: int = SEED_BASE + 6, B: int = 16, depth: int = 6, expand: int = 10,
                      branch: int = 10, V: int = 128256) -> dict:
    """Candidate draft trees shaped like EAGLE-2's expansion stage (see the
    module docstring): parents [B, N] int32 (creation order, parents[0] =
    -1), conf [B, N] fp32 (conf[:, 0] = 1), node_tok [B, N] int32."""
    r_tree, r_conf, r_tok = _rngs(seed, 3)
    N = 1 + branch + (depth - 1) * expand * branch
    parents = np.full((B, N), -1, np.int32)
    conf = np.ones((B, N), np.float32)
    for b in range(B):
        nxt, layer = 1, [0]
        for d in range(depth):
            grow = layer if d == 0 else np.sort(r_tree.choice(layer, size=min(expand, len(layer)), replace=False))
            new = []
            for u in grow:
                w = np.sort(r_conf.dirichlet(np.full(branch + 1, 0.5))[:branch])[::-1].astype(np.float32)
                for c in w:
                    parents[b, nxt] = u
                    conf[b, nxt] = c
                    new.append(nxt)
                    nxt += 1
            layer = new
        assert nxt == N
    node_tok = r_tok.integers(0, V, (B, N)).astype(np.int32)
    return dict(parents=parents, conf=conf, node_tok=node_tok, V=V, depth=depth)
