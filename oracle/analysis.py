"""Host-side helpers of the oracle (plain Python) -- TEST INFRASTRUCTURE.

These restate the pages' bookkeeping, the closed form and the choice of k; they never touch
logits.  The decode loop takes its drafter and verifier as callables so the
same host loop can drive the oracle and, in the GPU tests, the library.
"""
from __future__ import annotations

from typing import Callable, Sequence

import numpy as np


def forward_bookkeeping(acceptances: Sequence[int], rounds: int | None = None):
    """(target forwards, tokens advanced) after the given rounds.

    "第 13 篇：推理引擎一次猜几个字" (section ④ 纸笔实验 and its REPL
    version): every round costs one target forward and advances the accepted
    count plus the one token the target supplies at the break point.
    """
    forwards = advanced = 0
    for m in list(acceptances)[:rounds]:
        forwards += 1
        advanced += m + 1
    return forwards, advanced


def expected_tokens_per_round(alpha: float, k: int) -> float:
    """(1 - alpha^(k+1)) / (1 - alpha): tokens per round when each of the k
    positions is accepted independently with probability alpha
    ("投机解码:为什么一个字都不改", replay/bookkeeping section)."""
    if alpha == 1.0:
        return float(k + 1)
    return (1.0 - alpha ** (k + 1)) / (1.0 - alpha)


def greedy_generate(next_logits: Callable[[list], np.ndarray], prompt: Sequence[int],
                    n_new: int, argmax: Callable) -> list:
    """Plain greedy decoding: one target call per token, take the argmax."""
    out = list(prompt)
    for _ in range(n_new):
        out.append(int(argmax(next_logits(out))))
    return out[len(prompt):]


def speculative_generate(next_logits: Callable[[list], np.ndarray], prompt: Sequence[int],
                         n_new: int, k: int, draft_fn: Callable, verify_fn: Callable):
    """The draft -> one verification -> append loop ("第 13 篇", section ③ 伪代码).

    draft_fn(history list) -> list of at most k proposed tokens.
    verify_fn(rows [L+1, V], draft list) -> tokens to append (accepted prefix
    plus the target's own token at the break point).
    Returns (generated tokens, per-round accepted counts).
    """
    out = list(prompt)
    accepted = []
    while len(out) - len(prompt) < n_new:
        draft = list(draft_fn(out))[:k]
        # one "forward" over the prefix and the draft: row i is the target's
        # next-token logits after prefix + draft[:i]
        rows = np.stack([next_logits(out + draft[:i]) for i in range(len(draft) + 1)])
        emitted = list(verify_fn(rows, draft))
        accepted.append(len(emitted) - 1)
        out.extend(emitted)
    return out[len(prompt):len(prompt) + n_new], accepted


def speedup(alpha: float, k: int, draft_cost: float) -> float:
    """Walltime speedup of speculative decoding over plain decoding when one
    draft forward costs `draft_cost` target forwards: a round runs k draft
    forwards and one target forward and yields the expected tokens per round
    ("投机解码:为什么一个字都不改", the bookkeeping experiments weighing the
    draft's cost against k)."""
    return expected_tokens_per_round(alpha, k) / (k * draft_cost + 1.0)


def best_k(alpha: float, draft_cost: float, k_max: int):
    """The draft length in 0..k_max with the largest speedup, by trying each
    (k = 0 is plain decoding, speedup 1; a tie keeps the smaller k)."""
    best, best_s = 0, 1.0
    for k in range(1, k_max + 1):
        s = speedup(alpha, k, draft_cost)
        if s > best_s:
            best, best_s = k, s
    return best, best_s


def alpha_estimate(accepted: Sequence[int], draft_len: Sequence[int] | None = None, k: int = 0):
    """Acceptance rate from observed rounds: a round that accepted m of L
    drafted tokens tested m + 1 positions if m < L (the last one rejected)
    and L if m = L; alpha = accepted positions / tested positions."""
    lens = [k] * len(accepted) if draft_len is None else list(draft_len)
    acc = sum(int(m) for m in accepted)
    tests = sum(int(m) + (1 if int(m) < int(L) else 0) for m, L in zip(accepted, lens))
    return (acc / tests if tests else float("nan")), tests
