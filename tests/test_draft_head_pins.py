"""Pins of the draft-step oracle (oracle/draft_head.py): the draft token
follows softmax(z / T), T = 0 is the argmax, the step is the verify step's
bonus path with no drafts, and a round drafted by it keeps the target
distribution."""
import numpy as np
import pytest
from scipy import stats

import oracle
from oracle import draft_head


def chi2(counts, probs):
    exp = counts.sum() * probs
    keep = exp > 0
    assert counts[~keep].sum() == 0
    return float(((counts[keep] - exp[keep]) ** 2 / exp[keep]).sum()), int(keep.sum()) - 1


@pytest.mark.parametrize("T", [0.7, 1.5])
def test_draws_follow_the_tempered_softmax(T):
    rng = np.random.default_rng(int(T * 10))
    V, n = 16, 200_000
    z = rng.normal(0, 1.5, size=V)
    q = np.exp(z / T - (z / T).max())
    q /= q.sum()
    u = rng.random(n)
    res = draft_head.draft_step_from_logits(np.broadcast_to(z, (n, V)), u, T)
    counts = np.bincount(res["tokens"], minlength=V).astype(np.float64)
    s, df = chi2(counts, q)
    assert s < stats.chi2.ppf(1 - 1e-3, df), (s, df)
    # a wrong temperature is caught by the same test
    qw = np.exp(z - z.max())
    qw /= qw.sum()
    assert chi2(counts, qw)[0] > stats.chi2.ppf(1 - 1e-3, df)


def test_greedy_is_the_argmax_with_lowest_id_ties():
    z = np.array([[0.1, 2.0, 2.0, -1.0], [5.0, 1.0, 5.0, 5.0], [-3.0, -2.0, -1.0, -0.5]])
    res = draft_head.draft_step_from_logits(z, None, 0.0)
    assert res["tokens"].tolist() == [1, 0, 3]
    assert res["top2_gap"].tolist() == [0.0, 0.0, 0.5]


def test_step_equals_the_bonus_path_without_drafts():
    rng = np.random.default_rng(7)
    B, d, V, T = 5, 32, 300, 0.8
    h = rng.normal(size=(B, d))
    W = rng.normal(size=(V, d)) / np.sqrt(d)
    u = rng.random(B)
    step = draft_head.draft_step(h, W, u, T)
    z = oracle.lm_head(h, W)
    ver = oracle.verify_sampling(z.reshape(B, 1, V), np.zeros((B, 0, V)), np.zeros((B, 0), dtype=np.int64),
                                 u.reshape(B, 1), T)
    assert np.array_equal(step["tokens"], ver["tokens"][:, 0])
    assert np.allclose(step["logits"], h @ W.T, rtol=1e-13, atol=1e-12)


def test_round_drafted_by_the_step_keeps_the_target_distribution():
    """K = 2 draft steps (fixed draft logits per slot), then the verify step:
    the token emitted at slot 0 is ~ p_0, and at slot 1 (given slot 0 was
    accepted) ~ p_1."""
    rng = np.random.default_rng(3)
    V, K, n = 8, 2, 300_000
    zq = rng.normal(0, 1.2, size=(K, V))
    zp = zq[[0, 1, 1]] + rng.normal(0, 0.6, size=(K + 1, V))
    T = 1.0
    u_draft = rng.random((n, K))
    x = np.stack([draft_head.draft_step_from_logits(np.broadcast_to(zq[j], (n, V)), u_draft[:, j], T)["tokens"]
                  for j in range(K)], axis=1)
    u = rng.random((n, K + 1))
    res = oracle.verify_sampling(np.broadcast_to(zp, (n, K + 1, V)), np.broadcast_to(zq, (n, K, V)), x, u, T)
    p = np.exp(zp - zp.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    c0 = np.bincount(res["tokens"][:, 0], minlength=V).astype(np.float64)
    s, df = chi2(c0, p[0])
    assert s < stats.chi2.ppf(1 - 1e-3, df), (s, df)
    sel = res["num_accepted"] >= 1
    c1 = np.bincount(res["tokens"][sel, 1], minlength=V).astype(np.float64)
    s, df = chi2(c1, p[1])
    assert s < stats.chi2.ppf(1 - 1e-3, df), (s, df)
