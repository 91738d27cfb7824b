"""CPU oracle of the KV-cache commit that follows the verify step.

TEST INFRASTRUCTURE, like the rest of ``oracle/``: only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may use it.

What the pages fix ([NALAR] "Speculative Decoding: Memverifikasi Token Draft
secara Paralel", section "Verifikasi mengubah jalur cache", with the prefix
rule of "Penolakan memotong prefix yang diterima"): the target pass writes
cache state for every candidate position before anyone knows which survive;
after verification the entries of the discarded suffix must not become part
of the committed decoding state, and the next round must see target state
that matches the committed prefix only.  A separate autoregressive draft
model's cache must be advanced consistently with the accepted prefix and the
correction token.  Truncation, staged writes and index management are all
named as acceptable ways to get there.

Reading taken here (the plainest one the section supports):

* The target pass of one round consumes K+1 inputs per sequence: the last
  committed token t and the drafts x_0..x_{K-1}, at positions L..L+K, where L
  is the committed length before the round.  It produces K+1 cache entries
  (S = K+1 staged entries).  With n drafts accepted the committed inputs are
  t, x_0..x_{n-1}: the first n+1 entries survive.  The correction / bonus
  token has no entry yet; it is the next round's t.
* The draft model, drafting K tokens, consumed t, x_0..x_{K-2}: S = K staged
  entries, of which min(n+1, K) survive (with all K accepted, x_{K-1} was
  never fed to the draft model, which is then one entry behind).
* One rule covers both caches: keep = min(n+1, S); a sequence the verify
  step flagged as bad (n = -1) keeps nothing.
* Cache layout: a paged pool ``pool[layer][page][slot][entry]`` of fixed-size
  entries, and a block table ``block_table[b][p]`` giving the page that holds
  positions p*page_size .. (p+1)*page_size - 1 of sequence b.
* Staged mode: the pass wrote its S entries to ``staged[layer][b][i]``;
  committing copies the kept ones to positions L..L+keep-1 through the block
  table and advances the length.  In-place mode: the pass already wrote the
  entries at their positions; committing only advances the length, which is
  the index-based truncation of the rejected suffix.
* A sequence whose kept positions would need a page outside the pool or a
  block-table column past its end is left untouched (no copy, no length
  change) and reported.

Pins (tests/test_kv_commit_pins.py): the section's worked prefix example
(three drafts accepted, the fourth rejected), equality with the cache built
by feeding the committed tokens one at a time to a toy model (several rounds,
target and draft caches), untouched bytes outside the committed range, the
bad-row and capacity cases.
"""
from __future__ import annotations

import numpy as np


def kept_entries(num_accepted, S: int) -> np.ndarray:
    """keep_b = min(n_b + 1, S), 0 for a bad row (n_b < 0)."""
    n = np.asarray(num_accepted, dtype=np.int64)
    return np.where(n < 0, 0, np.minimum(n + 1, S)).astype(np.int64)


def commit(num_accepted, seq_len, block_table, pool, staged, page_size: int):
    """Commit one round.

    ``pool`` uint8 [layers][num_pages][page_size][E] is updated in place from
    ``staged`` uint8 [layers][B][S][E] (in-place mode is
    :func:`commit_in_place`).  Returns (new_seq_len, bad) with ``bad[b]``
    True for a sequence that could not be committed (left untouched)."""
    layers, B, S, E = staged.shape
    keep = kept_entries(num_accepted, S)
    new_len, bad = _lengths(keep, seq_len, block_table, pool.shape[1], page_size)
    for b in range(B):
        if bad[b]:
            continue
        for i in range(int(keep[b])):
            pos = int(seq_len[b]) + i
            page = int(block_table[b][pos // page_size])
            slot = pos % page_size
            for layer in range(layers):
                pool[layer, page, slot, :] = staged[layer, b, i, :]
    return new_len, bad


def commit_in_place(num_accepted, seq_len, block_table, num_pages: int, page_size: int, S: int):
    """Index-based truncation: only the lengths move."""
    keep = kept_entries(num_accepted, S)
    return _lengths(keep, seq_len, block_table, num_pages, page_size)


def _lengths(keep, seq_len, block_table, num_pages: int, page_size: int):
    B = len(keep)
    max_pages = block_table.shape[1]
    new_len = np.array(seq_len, dtype=np.int64).copy()
    bad = np.zeros(B, dtype=bool)
    for b in range(B):
        L = int(seq_len[b])
        k = int(keep[b])
        if L < 0:
            bad[b] = True
            continue
        if k == 0:
            continue
        last = L + k - 1
        if last // page_size >= max_pages:
            bad[b] = True
            continue
        pages = {int(block_table[b][p // page_size]) for p in range(L, L + k)}
        if any(pg < 0 or pg >= num_pages for pg in pages):
            bad[b] = True
            continue
        new_len[b] = L + k
    return new_len, bad


def gather_sequence(pool, block_table, b: int, length: int, page_size: int) -> np.ndarray:
    """The committed entries of sequence b, positions 0..length-1, as
    [layers][length][E] (what the next round's attention would read)."""
    out = np.empty((pool.shape[0], length, pool.shape[3]), dtype=pool.dtype)
    for pos in range(length):
        out[:, pos, :] = pool[:, int(block_table[b][pos // page_size]), pos % page_size, :]
    return out
