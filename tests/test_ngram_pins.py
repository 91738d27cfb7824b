"""Pins of the prompt-lookup drafter oracle (oracle/ngram_drafter.py)."""
import itertools

import numpy as np
import pytest

from oracle import ngram_drafter as ng

from _helpers import load_golden_text


def brute(history, K, n_min, n_max):
    """Every (n, s) whose n-gram at s equals the last n tokens, s before the
    suffix; the longest n, then the smallest s."""
    h = list(history)
    L = len(h)
    cands = [(n, s) for n in range(n_min, n_max + 1) for s in range(L) if n <= L - 1 and s + n <= L - 1
             and h[s:s + n] == h[L - n:]]
    if not cands:
        return [h[-1] if h else 0] * K, 0
    n, s = max(cands, key=lambda c: (c[0], -c[1]))
    prop = h[s + n:s + n + K]
    return prop + [prop[-1]] * (K - len(prop)), len(prop)


def test_hand_case_output_copies_prompt():
    """The page's scenario: an output that rewrites its prompt proposes the
    prompt's continuation of the output's tail."""
    g = load_golden_text("prompt_lookup.txt")
    vocab = {}
    tok = lambda words: [vocab.setdefault(w, len(vocab)) for w in words]
    prompt = g["prompt"]
    output = g["output"]
    hist = tok(prompt) + tok(output)
    K = int(g["K"][0])
    drafts, count = ng.propose(hist, K, 1, int(g["n_max"][0]))
    inv = {v: k for k, v in vocab.items()}
    assert [inv[int(t)] for t in drafts[:count]] == list(g["expect"])
    assert count == len(g["expect"])


def test_periodic_history_continues_the_period():
    hist = [7, 8, 9] * 4 + [7, 8]          # ... 7 8 9 7 8
    drafts, count = ng.propose(hist, 5, 1, 3)
    # suffix (9, 7, 8) first occurs at s = 2; what followed is 9 7 8 9 7
    assert count == 5 and drafts.tolist() == [9, 7, 8, 9, 7]


def test_all_distinct_history_has_no_proposal():
    hist = list(range(100, 130))
    drafts, count = ng.propose(hist, 4, 1, 3)
    assert count == 0 and drafts.tolist() == [129] * 4
    drafts, count = ng.propose([], 3, 1, 3)
    assert count == 0 and drafts.tolist() == [0, 0, 0]
    drafts, count = ng.propose([5], 3, 1, 3)
    assert count == 0 and drafts.tolist() == [5, 5, 5]


def test_longer_ngram_wins_over_earlier_shorter_match():
    # 1-gram "3" first occurs at 0, but the 2-gram "2 3" occurs at 4
    hist = [3, 9, 9, 9, 2, 3, 5, 6, 2, 3]
    drafts, count = ng.propose(hist, 2, 1, 3)
    assert count == 2 and drafts.tolist() == [5, 6]
    # with n_max = 1 the earliest 1-gram wins
    drafts, count = ng.propose(hist, 2, 1, 1)
    assert drafts.tolist() == [9, 9]


def test_proposal_cut_at_history_end_and_filled():
    hist = [1, 2, 3, 1, 2]                 # suffix (1, 2) at 0, continuation 3 1 2
    drafts, count = ng.propose(hist, 6, 1, 3)
    assert count == 3 and drafts.tolist() == [3, 1, 2, 2, 2, 2]


def test_n_min_excludes_short_matches():
    hist = [4, 5, 6, 4]
    assert ng.propose(hist, 2, 1, 3)[1] == 2      # 1-gram "4" at 0
    assert ng.propose(hist, 2, 2, 3)[1] == 0      # no 2-gram match


@pytest.mark.parametrize("n_min,n_max", [(1, 1), (1, 3), (2, 3)])
def test_exhaustive_brute_force_small_alphabet(n_min, n_max):
    K = 3
    for L in range(0, 8):
        for hist in itertools.product(range(3), repeat=L):
            d, c = ng.propose(list(hist), K, n_min, n_max)
            bd, bc = brute(list(hist), K, n_min, n_max)
            assert c == bc and d.tolist() == bd, (hist, d, c, bd, bc)


def test_invariants_on_random_histories():
    rng = np.random.default_rng(0)
    for trial in range(300):
        L = int(rng.integers(1, 200))
        V = int(rng.integers(2, 30))
        hist = rng.integers(0, V, size=L)
        n, s = ng.find_match(hist, 1, 4)
        d, c = ng.propose(hist, 5, 1, 4)
        if n == 0:
            assert c == 0
            continue
        assert np.array_equal(hist[s:s + n], hist[L - n:])
        assert c == min(5, L - s - n) and np.array_equal(d[:c], hist[s + n:s + n + c])
        # no longer key matches anywhere, and no earlier start for this key
        for m in range(n + 1, min(4, L - 1) + 1):
            for t in range(0, L - m):
                assert not np.array_equal(hist[t:t + m], hist[L - m:])
        for t in range(0, s):
            assert not np.array_equal(hist[t:t + n], hist[L - n:])


def test_batch_form_matches_rows():
    rng = np.random.default_rng(1)
    lens = np.array([0, 1, 17, 64, 5])
    hists = rng.integers(0, 4, size=(5, 64))
    d, c = ng.propose_batch(hists, lens, 4, 1, 3)
    for b in range(5):
        db, cb = ng.propose(hists[b, : lens[b]], 4, 1, 3)
        assert c[b] == cb and np.array_equal(d[b], db)
