"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test ties one oracle function to something other than itself: a worked
example printed on the pages (fixtures under tests/golden/), a closed form, a
brute-force enumeration, a textbook special case, or a chi-square test of the
exactness property over 10^6 draws.  The negative controls plant mistakes in
the oracle (on the CPU) and check that the pins catch them.
"""
import itertools
import os

import numpy as np
import pytest
import torch
from scipy import stats

import oracle
from oracle import spec_oracle
from speculative_decoding_verification_67_gb300 import synth

from _helpers import load_golden

def draw_drafts(q_rows, n, seed):
    """n independent draft tokens per row of q (Gumbel-max, seeded)."""
    g = torch.Generator().manual_seed(seed)
    logits = torch.log(torch.as_tensor(q_rows, dtype=torch.float64))
    logits = logits.unsqueeze(0).expand(n, *logits.shape)
    return synth.gumbel_max_tokens(logits, 1.0, g).numpy()


def run_fixed_distributions(p_rows, q_rows, n, seed, chunk=200_000):
    """Run the oracle's sampling round n times on fixed per-slot distributions
    (p_rows [K+1, V], q_rows [K, V]); returns (tokens [n, K+1], num_accepted [n])."""
    p_rows = np.asarray(p_rows, dtype=np.float64)
    q_rows = np.asarray(q_rows, dtype=np.float64)
    K = q_rows.shape[0]
    rng = np.random.default_rng(seed)
    toks, ns = [], []
    for c0 in range(0, n, chunk):
        m = min(chunk, n - c0)
        zp = np.broadcast_to(np.log(p_rows), (m,) + p_rows.shape)
        zq = np.broadcast_to(np.log(q_rows), (m,) + q_rows.shape)
        x = draw_drafts(q_rows, m, seed + 1 + c0) if K > 0 else np.zeros((m, 0), dtype=np.int64)
        u = rng.random((m, K + 1))
        res = oracle.verify_sampling(zp, zq, x, u, 1.0)
        toks.append(res["tokens"])
        ns.append(res["num_accepted"])
    return np.concatenate(toks), np.concatenate(ns)


def chi2_stat(counts, probs):
    counts = np.asarray(counts, dtype=np.float64)
    exp = counts.sum() * np.asarray(probs, dtype=np.float64)
    keep = exp > 0
    assert counts[~keep].sum() == 0, "mass on a zero-probability outcome"
    return float(((counts[keep] - exp[keep]) ** 2 / exp[keep]).sum()), int(keep.sum()) - 1


CHI2_ALPHA = 1e-3


def chi2_ok(counts, probs):
    s, df = chi2_stat(counts, probs)
    return s <= stats.chi2.ppf(1 - CHI2_ALPHA, df), s, df


# ---------------------------------------------------------------------------
# the 60/30/10 worked example
# ---------------------------------------------------------------------------
def test_worked_example_accept_ratios():
    g = load_golden("paris_london_rome.txt")
    a = oracle.accept_probability(g["p"], g["q"])
    np.testing.assert_allclose(g["p"] / g["q"], g["ratio"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(a, g["accept_prob"], rtol=0, atol=1e-15)


def test_worked_example_counts_and_residual():
    g = load_golden("paris_london_rome.txt")
    n = g["trials"][0]
    a = oracle.accept_probability(g["p"], g["q"])
    np.testing.assert_allclose(n * g["q"], g["proposed"], atol=1e-9)
    np.testing.assert_allclose(n * g["q"] * a, g["accepted"], atol=1e-9)
    assert abs(n * oracle.acceptance_rate(g["p"], g["q"]) - g["accepted_total"][0]) < 1e-9
    assert abs(n * (1 - oracle.acceptance_rate(g["p"], g["q"])) - g["rejected_total"][0]) < 1e-9
    r = oracle.residual(g["p"], g["q"])
    np.testing.assert_allclose(r, g["residual"], atol=1e-15)
    np.testing.assert_allclose(r / r.sum(), g["residual_normalised"], atol=1e-12)
    # every rejection is corrected to Paris, whatever the uniform
    for u in (0.0, 0.3, 0.999999):
        y, *_ = oracle.inverse_cdf(r, u)
        assert y[0] == 0
    final = g["accepted"] + g["rejected_total"][0] * r / r.sum()
    np.testing.assert_allclose(final, g["final"], atol=1e-9)
    np.testing.assert_allclose(final, g["target_counts"], atol=1e-9)
    wrong = g["accepted"] + g["rejected_total"][0] * g["p"]
    np.testing.assert_allclose(g["rejected_total"][0] * g["p"], g["wrong_fix_added"], atol=1e-9)
    np.testing.assert_allclose(wrong, g["wrong_fix_final"], atol=1e-9)


def test_worked_example_monte_carlo():
    """10^6 rounds with K=1 through the oracle's own round: about 900 of every
    1000 proposals are accepted and the output follows 60/30/10."""
    g = load_golden("paris_london_rome.txt")
    p, q = g["p"], g["q"]
    p_rows = np.stack([p, p])          # slot 0 and the bonus row
    n = 1_000_000
    toks, ns = run_fixed_distributions(p_rows, q[None, :], n, seed=11)
    rate = (ns == 1).mean()
    sigma = np.sqrt(0.9 * 0.1 / n)
    assert abs(rate - 0.9) < 5 * sigma
    ok, s, df = chi2_ok(np.bincount(toks[:, 0], minlength=3), p)
    assert ok, (s, df)
    # the rejected rounds are all corrected to Paris
    assert (toks[ns == 0, 0] == 0).all()


def test_wrong_fix_is_caught(monkeypatch):
    """Planted mistake: resample rejections from p instead of the residual.
    The output then follows 56/33/11 and the chi-square test rejects it."""
    g = load_golden("paris_london_rome.txt")
    p, q = g["p"], g["q"]
    monkeypatch.setattr(spec_oracle, "residual", lambda p_row, q_row: np.asarray(p_row, dtype=np.float64))
    toks, _ = run_fixed_distributions(np.stack([p, p]), q[None, :], 1_000_000, seed=12)
    counts = np.bincount(toks[:, 0], minlength=3)
    ok, s, df = chi2_ok(counts, p)
    assert not ok
    np.testing.assert_allclose(counts / counts.sum(), g["wrong_fix_final"] / 1000, atol=3e-3)


# ---------------------------------------------------------------------------
# the 45/25/20 example
# ---------------------------------------------------------------------------
def test_dep_nong_lanh_greedy_and_sampling():
    g = load_golden("dep_nong_lanh.txt")
    p = g["p"]
    V = len(p)
    zp = np.log(p)[None, None, :].repeat(2, axis=1)       # B=1, K=1 (+ bonus row)
    res = oracle.verify_greedy(zp, np.array([[int(g["greedy_choice"][0])]]))
    assert res["argmax"][0, 0] == int(g["greedy_choice"][0])
    assert res["num_accepted"][0] == 1
    # sampling against a uniform draft: acceptance sum min(p, 1/5) = 0.70
    q = np.full(V, 1.0 / V)
    assert abs(oracle.acceptance_rate(p, q) - 0.70) < 1e-12
    n = 1_000_000
    toks, ns = run_fixed_distributions(np.stack([p, p]), q[None, :], n, seed=13)
    assert abs((ns == 1).mean() - 0.70) < 5 * np.sqrt(0.7 * 0.3 / n)
    ok, s, df = chi2_ok(np.bincount(toks[:, 0], minlength=V), p)
    assert ok, (s, df)


# ---------------------------------------------------------------------------
# exactness: chi-square over 10^6 rounds at V=16, K=4
# ---------------------------------------------------------------------------
def _random_pq(V, K, seed):
    rng = np.random.default_rng(seed)
    p = np.exp(rng.normal(size=(K + 1, V)))
    p /= p.sum(axis=1, keepdims=True)
    q = np.exp(rng.normal(size=(K, V)))
    q /= q.sum(axis=1, keepdims=True)
    return p, q


def _slot_counts(toks, ns, K, V):
    """Per slot j: counts of the token emitted at slot j among rounds that
    reached slot j (n >= j)."""
    out = []
    for j in range(K + 1):
        reached = ns >= j
        out.append(np.bincount(toks[reached, j], minlength=V))
    return out


def test_exactness_chi_square_v16_k4():
    V, K = 16, 4
    p, q = _random_pq(V, K, seed=21)
    n = 1_000_000
    toks, ns = run_fixed_distributions(p, q, n, seed=22)
    for j, counts in enumerate(_slot_counts(toks, ns, K, V)):
        ok, s, df = chi2_ok(counts, p[j])
        assert ok, (j, s, df)
    # closed-form acceptance at slot 0: sum_x min(p0, q0)
    a0 = oracle.acceptance_rate(p[0], q[0])
    rate0 = (ns >= 1).mean()
    assert abs(rate0 - a0) < 5 * np.sqrt(a0 * (1 - a0) / n)
    # prefix structure: P(n >= j) = prod_{i<j} sum min(p_i, q_i)
    for j in range(1, K + 1):
        expect = np.prod([oracle.acceptance_rate(p[i], q[i]) for i in range(j)])
        assert abs((ns >= j).mean() - expect) < 5 * np.sqrt(expect * (1 - expect) / n) + 1e-12


def test_exactness_negative_control_v16(monkeypatch):
    V, K = 16, 4
    p, q = _random_pq(V, K, seed=21)
    monkeypatch.setattr(spec_oracle, "residual", lambda p_row, q_row: np.asarray(p_row, dtype=np.float64))
    toks, ns = run_fixed_distributions(p, q, 1_000_000, seed=23)
    counts = _slot_counts(toks, ns, K, V)[0]
    ok, s, df = chi2_ok(counts, p[0])
    assert not ok


def test_accept_rule_planted_mistake_is_caught(monkeypatch):
    """Planted mistake: accept with p/q unclipped swapped for q/p."""
    V, K = 16, 1
    p, q = _random_pq(V, K, seed=24)
    monkeypatch.setattr(spec_oracle, "accept_probability",
                        lambda p_x, q_x: np.minimum(1.0, np.asarray(q_x) / np.asarray(p_x)))
    toks, ns = run_fixed_distributions(p, q, 400_000, seed=25)
    ok, s, df = chi2_ok(np.bincount(toks[:, 0], minlength=V), p[0])
    assert not ok


# ---------------------------------------------------------------------------
# brute force: every accept / reject path at V=4, K=2
# ---------------------------------------------------------------------------
def _enumerate_paths(p, q):
    """Exact probability of every outcome (n, emitted tokens) of one round,
    by walking the paths one at a time: draft x0 ~ q0, accept with
    min(1, p0/q0); then x1 ~ q1, accept with min(1, p1/q1); a rejection at
    slot j emits a token of max(0, p_j - q_j) normalised; two accepts emit a
    bonus token of p2."""
    V = p.shape[1]
    out = {}

    def add(key, w):
        out[key] = out.get(key, 0.0) + w

    res = [np.maximum(0.0, p[j] - q[j]) for j in range(2)]
    res = [r / r.sum() for r in res]
    for x0 in range(V):
        a0 = min(1.0, p[0, x0] / q[0, x0])
        for y in range(V):
            add((0, y), q[0, x0] * (1 - a0) * res[0][y])
        for x1 in range(V):
            a1 = min(1.0, p[1, x1] / q[1, x1])
            w = q[0, x0] * a0 * q[1, x1]
            for y in range(V):
                add((1, x0, y), w * (1 - a1) * res[1][y])
                add((2, x0, x1, y), w * a1 * p[2, y])
    return out


def test_brute_force_paths_v4_k2():
    V, K = 4, 2
    p, q = _random_pq(V, K, seed=31)
    paths = _enumerate_paths(p, q)
    assert len(paths) == 4 + 16 + 64
    assert abs(sum(paths.values()) - 1.0) < 1e-12
    # the enumeration itself reproduces p at slot 0 (the exactness identity)
    slot0 = np.zeros(V)
    for key, w in paths.items():
        slot0[key[1]] += w
    np.testing.assert_allclose(slot0, p[0], atol=1e-12)

    n = 1_000_000
    toks, ns = run_fixed_distributions(p, q, n, seed=32)
    keys = sorted(paths)
    index = {k: i for i, k in enumerate(keys)}
    counts = np.zeros(len(keys))
    for nb in range(K + 1):
        sel = ns == nb
        sub = toks[sel, :nb + 1]
        uniq, c = np.unique(sub, axis=0, return_counts=True)
        for row, cnt in zip(uniq, c):
            counts[index[(nb,) + tuple(int(t) for t in row)]] += cnt
    ok, s, df = chi2_ok(counts, np.array([paths[k] for k in keys]))
    assert ok, (s, df)


def test_brute_force_branch_regions_are_exact():
    """Deterministic check: uniforms chosen inside a branch's region reproduce
    that branch exactly, for every branch of the V=4, K=2 enumeration."""
    V, K = 4, 2
    p, q = _random_pq(V, K, seed=33)
    zp = np.log(p)[None]
    zq = np.log(q)[None]
    res = [np.maximum(0.0, p[j] - q[j]) for j in range(2)]

    def mid_of(dist, y):
        c = np.cumsum(dist / dist.sum())
        lo = c[y - 1] if y > 0 else 0.0
        return 0.5 * (lo + c[y])

    for x0, x1 in itertools.product(range(V), repeat=2):
        a0 = min(1.0, p[0, x0] / q[0, x0])
        a1 = min(1.0, p[1, x1] / q[1, x1])
        x = np.array([[x0, x1]])
        for y in range(V):
            if a0 < 1.0 and res[0][y] > 0:   # reject at slot 0, emit y
                u = np.array([[0.5 * (a0 + 1), 0.5, mid_of(res[0], y)]])
                r = oracle.verify_sampling(zp, zq, x, u, 1.0)
                assert r["num_accepted"][0] == 0 and r["tokens"][0, 0] == y
            if a0 > 0 and a1 < 1.0 and res[1][y] > 0:   # accept, reject, emit y
                u = np.array([[0.5 * a0, 0.5 * (a1 + 1), mid_of(res[1], y)]])
                r = oracle.verify_sampling(zp, zq, x, u, 1.0)
                assert r["num_accepted"][0] == 1
                assert list(r["tokens"][0]) == [x0, y, -1]
            if a0 > 0 and a1 > 0:   # accept both, bonus y
                u = np.array([[0.5 * a0, 0.5 * a1, mid_of(p[2], y)]])
                r = oracle.verify_sampling(zp, zq, x, u, 1.0)
                assert r["num_accepted"][0] == 2
                assert list(r["tokens"][0]) == [x0, x1, y]


# ---------------------------------------------------------------------------
# greedy
# ---------------------------------------------------------------------------
def _rows_with_argmax(ids, V):
    z = np.zeros((1, len(ids), V))
    for j, t in enumerate(ids):
        z[0, j, int(t)] = 1.0
    return z


def test_greedy_worked_rounds():
    g = load_golden("greedy_rounds.txt")
    V = int(g["vocab"][0])
    for r in ("r1", "r2"):
        zp = _rows_with_argmax(g[f"{r}_target_argmax"], V)
        x = g[f"{r}_drafts"].astype(np.int64)[None]
        res = oracle.verify_greedy(zp, x)
        assert res["num_accepted"][0] == int(g[f"{r}_num_accepted"][0])
        assert list(res["tokens"][0]) == [int(t) for t in g[f"{r}_tokens"]]


def test_greedy_ties_go_to_lowest_id():
    z = np.zeros((1, 2, 10))
    z[0, 0, [3, 7]] = 5.0
    z[0, 1, [9, 2, 4]] = 1.0
    res = oracle.verify_greedy(z, np.array([[7]]))
    assert res["argmax"][0, 0] == 3 and res["num_accepted"][0] == 0
    assert list(res["tokens"][0]) == [3, -1]
    res = oracle.verify_greedy(z, np.array([[3]]))
    assert list(res["tokens"][0]) == [3, 2]


def test_sampling_with_one_hot_target_reduces_to_greedy():
    """With p one-hot at its argmax, the sampling rule accepts a draft iff it
    is the argmax and otherwise corrects to the argmax, for any q > 0 and u."""
    rng = np.random.default_rng(41)
    B, K, V = 64, 4, 12
    g = rng.integers(0, V, size=(B, K + 1))
    zp = np.zeros((B, K + 1, V))
    zp[np.arange(B)[:, None], np.arange(K + 1)[None, :], g] = 1e4   # exp(-1e4) == 0
    zq = rng.normal(size=(B, K, V))
    x = np.where(rng.random((B, K)) < 0.7, g[:, :K], rng.integers(0, V, size=(B, K)))
    u = rng.random((B, K + 1))
    s = oracle.verify_sampling(zp, zq, x, u, 1.0)
    gr = oracle.verify_greedy(zp, x)
    np.testing.assert_array_equal(s["tokens"], gr["tokens"])
    np.testing.assert_array_equal(s["num_accepted"], gr["num_accepted"])


# ---------------------------------------------------------------------------
# LM head, softmax, inverse CDF
# ---------------------------------------------------------------------------
def test_lm_head_brute_force_tiny():
    rng = np.random.default_rng(51)
    M, d, V = 2, 3, 5
    h = rng.normal(size=(M, d))
    W = rng.normal(size=(V, d))
    z = oracle.lm_head(h, W)
    for m in range(M):
        for v in range(V):
            acc = 0.0
            for k in range(d):
                acc += h[m, k] * W[v, k]
            assert abs(z[m, v] - acc) < 1e-12


def test_lm_head_identity_slice_and_one_hot():
    rng = np.random.default_rng(52)
    M, d, V = 3, 8, 5
    h = rng.normal(size=(M, d))
    W = np.eye(d)[:V]                    # W[v] = e_v: logits are the first V features
    np.testing.assert_array_equal(oracle.lm_head(h, W), h[:, :V])
    W2 = rng.normal(size=(V, d))
    for k in range(d):
        e = np.zeros((1, d))
        e[0, k] = 1.0
        np.testing.assert_array_equal(oracle.lm_head(e, W2)[0], W2[:, k])
    # chunked upcast gives the same answer as one piece
    W3 = rng.normal(size=(37, d)).astype(np.float32)
    np.testing.assert_allclose(oracle.lm_head(h, W3, vocab_chunk=8),
                               h @ W3.astype(np.float64).T, rtol=0, atol=1e-12)


def test_softmax_temperature_closed_form():
    rng = np.random.default_rng(53)
    p = np.exp(rng.normal(size=20))
    p /= p.sum()
    np.testing.assert_allclose(oracle.softmax_t(np.log(p), 1.0), p, rtol=1e-12)
    for T in (0.5, 0.8, 2.0):
        pt = p ** (1.0 / T)
        np.testing.assert_allclose(oracle.softmax_t(np.log(p), T), pt / pt.sum(), rtol=1e-12)
    # shift invariance: adding a constant to the logits changes nothing
    np.testing.assert_allclose(oracle.softmax_t(np.log(p) + 123.0, 0.7),
                               oracle.softmax_t(np.log(p), 0.7), rtol=1e-12)


def test_inverse_cdf_boundaries():
    r = np.array([0.125, 0.25, 0.125, 0.5])       # dyadic: C = 0.125, 0.375, 0.5, 1 exactly
    for u, y in ((0.0, 0), (0.1, 0), (0.125, 1), (0.3749, 1), (0.375, 2), (0.5, 3), (0.999, 3)):
        got, lo, hi, S = oracle.inverse_cdf(r, u)
        assert got[0] == y, (u, got)
        assert lo[0] >= -1e-15 and hi[0] > 0 and abs(S[0] - 1.0) < 1e-15
    # zero-mass tokens are never drawn
    r = np.array([0.0, 0.5, 0.0, 0.5, 0.0])
    for u in np.linspace(0, 0.999, 50):
        got, *_ = oracle.inverse_cdf(r, u)
        assert got[0] in (1, 3)
    # unnormalised input: only proportions matter
    np.testing.assert_array_equal(oracle.inverse_cdf(7 * np.array([0.1, 0.2, 0.3, 0.4]), 0.35)[0],
                                  oracle.inverse_cdf(np.array([0.1, 0.2, 0.3, 0.4]), 0.35)[0])


def test_inverse_cdf_frequencies_follow_the_distribution():
    """Inverse CDF on uniform u reproduces the 45/25/20 frequencies (a die)."""
    p = load_golden("dep_nong_lanh.txt")["p"]
    u = np.random.default_rng(54).random(200_000)
    y, *_ = oracle.inverse_cdf(np.broadcast_to(p, (len(u), len(p))), u)
    ok, s, df = chi2_ok(np.bincount(y, minlength=len(p)), p)
    assert ok, (s, df)


# ---------------------------------------------------------------------------
# edge cases of the round
# ---------------------------------------------------------------------------
def test_k0_is_a_bonus_only_round():
    p = np.array([0.2, 0.5, 0.3])
    zp = np.log(p)[None, None, :]
    for u, y in ((0.1, 0), (0.5, 1), (0.9, 2)):
        r = oracle.verify_sampling(zp, np.zeros((1, 0, 3)), np.zeros((1, 0), dtype=np.int64),
                                   np.array([[u]]), 1.0)
        assert r["num_accepted"][0] == 0 and list(r["tokens"][0]) == [y]


def test_all_accepted_takes_the_bonus_row():
    p = np.array([[0.5, 0.5, 0.0], [0.1, 0.1, 0.8]])
    q = np.array([[0.5, 0.5, 0.0]])
    with np.errstate(divide="ignore"):
        zp, zq = np.log(p)[None], np.log(q)[None]
    r = oracle.verify_sampling(zp, zq, np.array([[1]]), np.array([[0.99, 0.5]]), 1.0)
    assert r["num_accepted"][0] == 1 and list(r["tokens"][0]) == [1, 2]


def test_temperature_scales_both_distributions():
    """The round at temperature T equals the round at T=1 on logits z/T."""
    rng = np.random.default_rng(61)
    B, K, V = 16, 3, 50
    zp = rng.normal(size=(B, K + 1, V))
    zq = zp[:, :K] + 0.5 * rng.normal(size=(B, K, V))
    x = rng.integers(0, V, size=(B, K))
    u = rng.random((B, K + 1))
    a = oracle.verify_sampling(zp, zq, x, u, 0.8)
    b = oracle.verify_sampling(zp / 0.8, zq / 0.8, x, u, 1.0)
    np.testing.assert_array_equal(a["tokens"], b["tokens"])
    np.testing.assert_allclose(a["accept_prob"], b["accept_prob"], rtol=1e-12)
