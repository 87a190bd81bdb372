"""Pins for greedy chain verification and the decode-loop bookkeeping.

T-a  the four worked cases on the target path ABCDEFG (golden fixture);
T-b  speculative greedy decoding reproduces plain greedy decoding token for
     token (the pages report 16/16 on their models; here a synthetic
     deterministic model and many seeds);
T-c  forward/advance bookkeeping: acceptances [0, 2, 4] cost 3 forwards and
     advance 9 tokens.
"""
import numpy as np
import pytest

import oracle
from oracle.analysis import forward_bookkeeping, greedy_generate, speculative_generate
from tests.conftest import read_table

PATH_SYMBOLS = "ABCDEFG"


def _path_rows(prior, guess, V):
    """Target logits for each verified position: after a prefix of the path the
    target's choice is the path's next symbol; elsewhere the row is flat."""
    ids = {c: i for i, c in enumerate(PATH_SYMBOLS)}
    ids["X"] = len(PATH_SYMBOLS)
    rows = np.zeros((len(guess) + 1, V), np.float32)
    for i in range(len(guess) + 1):
        seq = prior + guess[:i]
        if PATH_SYMBOLS.startswith(seq) and len(seq) < len(PATH_SYMBOLS):
            rows[i, ids[PATH_SYMBOLS[len(seq)]]] = 5.0
    return rows, np.array([[ids[c] for c in guess]], np.int32), ids


@pytest.mark.parametrize("V", [8, 2048])
def test_worked_cases_on_path_ABCDEFG(V):
    meta, rows = read_table("greedy_worked_cases.txt")
    assert meta["target_path"] == PATH_SYMBOLS and len(rows) == 4
    for prior, guess, acc, added, new_out in rows:
        prior = "" if prior == "-" else prior
        acc = "" if acc == "-" else acc
        logits, draft, ids = _path_rows(prior, guess, V)
        remaining = len(PATH_SYMBOLS) - len(prior)       # "at the end of the path, add nothing"
        out = oracle.verify_greedy(logits[None], draft, max_emit=np.array([remaining]))
        emitted = "".join(PATH_SYMBOLS[t] for t in out["out_tokens"][0, :out["n_emit"][0]])
        assert prior + emitted == new_out, (prior, guess)
        assert out["accepted"][0] == len(acc)
        assert emitted == acc + ("" if added == "-" else added)
        assert out["status"][0] == 0
        assert np.all(out["out_tokens"][0, out["n_emit"][0]:] == -1)


def test_greedy_all_accepted_emits_the_bonus_and_first_mismatch_stops():
    V, k = 32, 4
    rng = np.random.default_rng(0)
    t = rng.standard_normal((3, k + 1, V)).astype(np.float32)
    am = t.argmax(-1)
    draft = am[:, :k].copy()
    draft[1, 2] = (draft[1, 2] + 1) % V                 # request 1 rejects at 2
    draft[2, 0] = (draft[2, 0] + 1) % V                 # request 2 rejects at 0
    out = oracle.verify_greedy(t, draft)
    assert list(out["accepted"]) == [4, 2, 0]
    assert list(out["n_emit"]) == [5, 3, 1]
    assert list(out["out_tokens"][0]) == list(am[0])
    assert list(out["out_tokens"][1]) == list(am[1, :3]) + [-1, -1]
    assert list(out["out_tokens"][2]) == [am[2, 0], -1, -1, -1, -1]


def test_greedy_variable_length_bad_token_and_empty_draft():
    V, k = 16, 3
    t = np.zeros((4, k + 1, V), np.float32)
    t[:, :, 5] = 1.0
    draft = np.full((4, k), 5, np.int32)
    draft[2, 1] = V                                     # out of range
    out = oracle.verify_greedy(t, draft, draft_len=np.array([0, 2, 3, 4]))
    assert list(out["status"]) == [0, 0, oracle.ST_TOKEN_RANGE, oracle.ST_BAD_LENGTH]
    assert list(out["accepted"]) == [0, 2, 0, 0]
    assert list(out["n_emit"]) == [1, 3, 0, 0]
    assert list(out["out_tokens"][0]) == [5, -1, -1, -1]


def _model(seed, V):
    """A deterministic toy 'target': next-token logits depend only on the last
    two tokens, so greedy decoding falls into cycles the n-gram drafter finds."""
    def next_logits(seq):
        a = seq[-2] if len(seq) > 1 else V
        b = seq[-1]
        rng = np.random.default_rng(seed * 1_000_003 + a * (V + 1) + b)
        return rng.standard_normal(V).astype(np.float32)
    return next_logits


def _oracle_draft(k, window):
    def draft_fn(hist):
        h = np.array([hist], np.int32)
        d, n, _ = oracle.ngram_draft(h, [len(hist)], window, k)
        return list(d[0, :n[0]])
    return draft_fn


def _oracle_verify(rows, draft):
    out = oracle.verify_greedy(rows[None], np.array([draft], np.int32).reshape(1, len(draft)))
    return list(out["out_tokens"][0, :out["n_emit"][0]])


@pytest.mark.parametrize("seed", range(12))
def test_speculative_greedy_equals_plain_greedy(seed):
    V, k, n_new = 12, 4, 160
    model = _model(seed, V)
    prompt = [seed % V, (seed * 5 + 1) % V, (seed * 7 + 3) % V]
    plain = greedy_generate(model, prompt, n_new, oracle.argmax)
    spec, accepted = speculative_generate(model, prompt, n_new, k, _oracle_draft(k, 3), _oracle_verify)
    assert spec == plain
    # the loop did real speculation: some rounds accepted drafts, some rejected
    assert max(accepted) > 0 and min(accepted) == 0
    # bookkeeping of the loop itself: every round advanced accepted + 1 tokens
    fw, adv = forward_bookkeeping(accepted)
    assert fw == len(accepted) and adv >= n_new and adv - (accepted[-1] + 1) < n_new


def test_bookkeeping_worked_example():
    # "第 13 篇：推理引擎一次猜几个字", ④ 纸笔实验 and its REPL version
    assert forward_bookkeeping([0, 2, 4]) == (3, 9)
    assert 9 - forward_bookkeeping([0, 2, 4])[0] == 6     # 9 token-by-token forwards saved 6
    assert forward_bookkeeping([0]) == (1, 1)
    assert forward_bookkeeping([2]) == (1, 3)
    assert forward_bookkeeping([4]) == (1, 5)
    assert forward_bookkeeping([0, 2, 4], rounds=2) == (2, 4)
