"""Pins of the KV-cache commit oracle (oracle/kv_commit.py) to things other
than itself: the pages' worked prefix example, and the cache a plain
one-token-at-a-time decode would have built, for a toy model whose cache
entry is a fixed function of (cache, layer, token, position)."""
import numpy as np
import pytest

from oracle import kv_commit

from _helpers import load_golden


def toy_entry(cache_id: int, layer: int, token: int, pos: int, E: int) -> np.ndarray:
    """A cache entry that identifies what produced it: E bytes from a
    splitmix64 stream seeded by (cache, layer, token, pos)."""
    cache_id, layer, token, pos = int(cache_id), int(layer), int(token), int(pos)
    x = (cache_id * 1_000_003 + layer * 7919 + token * 104_729 + pos * 15_485_863) & 0xFFFFFFFFFFFFFFFF
    out = np.empty(E, dtype=np.uint8)
    for i in range(0, E, 8):
        x = (x + 0x9E3779B97F4A7C15) & 0xFFFFFFFFFFFFFFFF
        z = x
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & 0xFFFFFFFFFFFFFFFF
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & 0xFFFFFFFFFFFFFFFF
        z ^= z >> 31
        out[i:i + 8] = np.frombuffer(int(z).to_bytes(8, "little"), dtype=np.uint8)[: min(8, E - i)]
    return out


def sequential_cache(cache_id, tokens, length, layers, E):
    """What feeding tokens[0..length-1] one at a time would leave: [layers][length][E]."""
    out = np.empty((layers, length, E), dtype=np.uint8)
    for pos in range(length):
        for layer in range(layers):
            out[layer, pos] = toy_entry(cache_id, layer, tokens[pos], pos, E)
    return out


class PagedCache:
    """A paged pool with a shuffled block table (pages are not contiguous)."""

    def __init__(self, B, layers, E, page_size, max_pages, rng):
        self.page_size, self.layers, self.E = page_size, layers, E
        self.num_pages = B * max_pages + 3
        perm = rng.permutation(self.num_pages)
        self.block_table = perm[: B * max_pages].reshape(B, max_pages).astype(np.int64)
        self.pool = rng.integers(0, 256, size=(layers, self.num_pages, page_size, E), dtype=np.uint8)


def speculative_round(cache_id, cache, tokens, seq_len, drafts, n, correction, S):
    """One round for one cache: stage the pass's S entries, commit with n
    accepted, return the new committed token lists and lengths."""
    B = len(tokens)
    staged = np.zeros((cache.layers, B, S, cache.E), dtype=np.uint8)
    for b in range(B):
        L = int(seq_len[b])
        # the pass consumes the pending token tokens[b][L] and then the drafts
        inputs = [tokens[b][L]] + list(drafts[b])
        for i in range(S):
            for layer in range(cache.layers):
                staged[layer, b, i] = toy_entry(cache_id, layer, inputs[i], L + i, cache.E)
    new_len, bad = kv_commit.commit(n, seq_len, cache.block_table, cache.pool, staged, cache.page_size)
    assert not bad.any()
    return new_len


@pytest.mark.parametrize("page_size", [1, 3, 16])
def test_commit_equals_sequential_decode_over_rounds(page_size):
    """After every round, target and draft caches hold exactly the entries a
    non-speculative decode of the committed tokens would hold."""
    rng = np.random.default_rng(11)
    B, K, layers, E, rounds = 3, 4, 2, 24, 5
    max_pages = (2 + rounds * (K + 1) + page_size) // page_size + 1
    target = PagedCache(B, layers, E, page_size, max_pages, rng)
    draft = PagedCache(B, layers, E, page_size, max_pages, rng)
    # committed: two prompt tokens with entries, plus the pending token
    tokens = [list(rng.integers(0, 50, size=3)) for _ in range(B)]
    t_len = np.full(B, 2, dtype=np.int64)
    d_len = np.full(B, 2, dtype=np.int64)
    for cache, cid in ((target, 0), (draft, 1)):
        for b in range(B):
            for pos in range(2):
                page = cache.block_table[b][pos // page_size]
                for layer in range(layers):
                    cache.pool[layer, page, pos % page_size] = toy_entry(cid, layer, tokens[b][pos], pos, E)
    for r in range(rounds):
        drafts = rng.integers(0, 50, size=(B, K))
        n = rng.integers(0, K + 1, size=B)
        n[r % B] = K if r % 2 else 0          # both extremes occur
        correction = rng.integers(0, 50, size=B)
        # the draft model had consumed the pending token and x_0..x_{K-2}; its
        # committed length must first catch up with the target's (an all-accept
        # round leaves it one behind): feed the missing committed tokens
        for b in range(B):
            while d_len[b] < t_len[b]:
                pos = int(d_len[b])
                page = draft.block_table[b][pos // page_size]
                for layer in range(layers):
                    draft.pool[layer, page, pos % page_size] = toy_entry(1, layer, tokens[b][pos], pos, E)
                d_len[b] += 1
        new_t = speculative_round(0, target, tokens, t_len, drafts, n, correction, K + 1)
        new_d = speculative_round(1, draft, tokens, d_len, drafts[:, : K - 1], n, correction, K)
        for b in range(B):
            tokens[b] = tokens[b][: int(t_len[b]) + 1] + list(drafts[b][: n[b]]) + [int(correction[b])]
            assert new_t[b] == t_len[b] + n[b] + 1
            assert new_d[b] == d_len[b] + min(n[b] + 1, K)
        t_len, d_len = new_t, new_d
        for b in range(B):
            assert len(tokens[b]) == t_len[b] + 1          # one pending token, no entry
            got = kv_commit.gather_sequence(target.pool, target.block_table, b, int(t_len[b]), page_size)
            assert np.array_equal(got, sequential_cache(0, tokens[b], int(t_len[b]), layers, E))
            got = kv_commit.gather_sequence(draft.pool, draft.block_table, b, int(d_len[b]), page_size)
            assert np.array_equal(got, sequential_cache(1, tokens[b], int(d_len[b]), layers, E))


def test_pages_prefix_example():
    """Three drafts accepted, the fourth rejected: the committed target cache
    holds the pending token and x_1..x_3; x_4 and x_5 leave no entry."""
    g = load_golden("prefix_cut.txt")
    k, n = int(g["k"][0]), int(g["accepted"][0])
    kept = [int(v) for v in g["kept_drafts"]]
    dropped = [int(v) for v in g["dropped_drafts"]]
    rng = np.random.default_rng(5)
    cache = PagedCache(1, 1, 16, 4, 4, rng)
    before = cache.pool.copy()
    tokens = [[7]]                       # empty history, pending token 7
    drafts = np.array([[101, 102, 103, 104, 105][:k]])
    new_len = speculative_round(0, cache, tokens, np.array([0]), drafts, np.array([n]), None, k + 1)
    assert new_len[0] == 1 + len(kept)
    got = kv_commit.gather_sequence(cache.pool, cache.block_table, 0, int(new_len[0]), 4)
    committed_inputs = [7] + [int(drafts[0][i - 1]) for i in kept]
    assert np.array_equal(got, sequential_cache(0, committed_inputs, len(committed_inputs), 1, 16))
    # nothing of a dropped draft reached the pool: every byte past the
    # committed range is what was there before
    for i in dropped:
        pos = i                           # draft x_i sits at position i (pending token at 0)
        page = cache.block_table[0][pos // 4]
        assert np.array_equal(cache.pool[0, page, pos % 4], before[0, page, pos % 4])


def test_untouched_outside_committed_range_and_bad_rows():
    rng = np.random.default_rng(3)
    B, S, layers, E, ps = 4, 5, 2, 16, 4
    cache = PagedCache(B, layers, E, ps, 6, rng)
    before = cache.pool.copy()
    staged = rng.integers(0, 256, size=(layers, B, S, E), dtype=np.uint8)
    seq_len = np.array([0, 5, 20, 3])
    n = np.array([-1, 4, 4, 2])          # bad row, all accepted, capacity overflow, two accepted
    new_len, bad = kv_commit.commit(n, seq_len, cache.block_table, cache.pool, staged, ps)
    assert bad.tolist() == [False, False, True, False]
    assert new_len.tolist() == [0, 10, 20, 6]
    written = set()
    for b, L, k in ((1, 5, 5), (3, 3, 3)):
        for i in range(k):
            pos = L + i
            written.add((int(cache.block_table[b][pos // ps]), pos % ps))
            assert np.array_equal(cache.pool[:, cache.block_table[b][pos // ps], pos % ps], staged[:, b, i])
    for page in range(cache.num_pages):
        for slot in range(ps):
            if (page, slot) not in written:
                assert np.array_equal(cache.pool[:, page, slot], before[:, page, slot])


def test_in_place_truncation_lengths():
    bt = np.arange(8).reshape(2, 4)
    new_len, bad = kv_commit.commit_in_place(np.array([2, 3]), np.array([10, 12]), bt, 8, 4, 4)
    assert new_len.tolist() == [13, 16] and not bad.any()
    # position 16 would need block-table column 4, past the table's end
    new_len, bad = kv_commit.commit_in_place(np.array([3]), np.array([13]), bt[:1], 8, 4, 5)
    assert bad.tolist() == [True] and new_len.tolist() == [13]
    # a page id outside the pool
    bt2 = np.array([[0, 1, 99, 2]])
    new_len, bad = kv_commit.commit_in_place(np.array([1]), np.array([7]), bt2, 8, 4, 5)
    assert bad.tolist() == [True]
    assert kv_commit.kept_entries([-1, 0, 3, 9], 5).tolist() == [0, 1, 4, 5]
