"""CPU oracle of the prompt-lookup (n-gram) drafter.

TEST INFRASTRUCTURE, like the rest of ``oracle/``: only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may use it.

What the pages fix ([QH] quochung.cyou A.I article on speculative decoding,
"Vấn đề 3: Làm sao khi không muốn train drafter?"): with no trained drafter,
Prompt Lookup Decoding / n-gram matching looks for continuations that already
occurred in the initial prompt or in earlier output; it matches the tail of
the output being generated against that history and proposes what followed
the match; the proposal then goes to target verification.  It needs no
neural drafter, no weights and no extra memory, works well when the output
copies the input (code editing, summarisation, rewriting) and poorly in
open-ended chat.

Readings where the page is silent (the plainest ones it supports):

* history = the prompt followed by the output so far, one token sequence per
  sequence, length L;
* the matched key is a suffix of the history of n tokens, tried from n_max
  down to n_min; the first n with a match wins (longer context first);
* an occurrence is any start s < L - n (the suffix itself, s = L - n, is not
  an occurrence) with history[s:s+n] equal to the suffix; among them the
  earliest s wins: the page searches the prompt first, then later output;
* the proposal is history[s+n : s+n+K], cut at the end of the history, so it
  has count = min(K, L - s - n) >= 1 tokens;
* with no occurrence for any n, count = 0;
* the K output slots after the first count are filled with the last token of
  the proposal (the last history token when count = 0).  They are still
  drafts: greedy verification accepts a draft only where it equals the
  target's argmax, so a fill token costs nothing but its slot.

Pins (tests/test_ngram_pins.py): hand cases built on the page's scenario (an
output copying its prompt), periodic histories, all-distinct histories (no
proposal), exhaustive brute force over every history of length <= 7 on a
three-token alphabet, and the defining invariants on random histories.
"""
from __future__ import annotations

import numpy as np


def find_match(history, n_min: int, n_max: int):
    """(n, s) of the chosen occurrence, or (0, -1) when there is none."""
    h = np.asarray(history, dtype=np.int64)
    L = len(h)
    for n in range(min(n_max, L - 1), n_min - 1, -1):
        if n < 1:
            break
        suffix = h[L - n:]
        # candidate starts 0 .. L-n-1 (the suffix itself excluded)
        windows = np.lib.stride_tricks.sliding_window_view(h[: L - 1], n)   # starts 0 .. L-1-n
        hits = np.flatnonzero((windows == suffix).all(axis=1))
        if hits.size:
            return n, int(hits[0])
    return 0, -1


def propose(history, K: int, n_min: int, n_max: int):
    """(drafts [K] int64, count) for one history."""
    h = np.asarray(history, dtype=np.int64)
    n, s = find_match(h, n_min, n_max)
    if n == 0:
        count = 0
        prop = np.zeros(0, dtype=np.int64)
    else:
        prop = h[s + n: s + n + K]
        count = len(prop)
    out = np.empty(K, dtype=np.int64)
    out[:count] = prop
    fill = prop[-1] if count else (h[-1] if len(h) else 0)
    out[count:] = fill
    return out, count


def propose_batch(histories, lengths, K: int, n_min: int, n_max: int):
    """Batch form: ``histories`` [B][max_len] (rows padded past their length)."""
    B = len(lengths)
    drafts = np.empty((B, K), dtype=np.int64)
    counts = np.empty(B, dtype=np.int64)
    for b in range(B):
        drafts[b], counts[b] = propose(np.asarray(histories[b])[: int(lengths[b])], K, n_min, n_max)
    return drafts, counts
