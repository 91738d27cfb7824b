"""Pins of the tree-verification oracle (oracle/tree_verify.py)."""
import numpy as np
import pytest
from scipy import stats

import oracle
from oracle import tree_verify as tv

CRIT = lambda df: stats.chi2.ppf(1 - 1e-3, df)


def chi2(counts, probs):
    counts = np.asarray(counts, dtype=np.float64)
    exp = counts.sum() * np.asarray(probs, dtype=np.float64)
    keep = exp > 0
    assert counts[~keep].sum() == 0, "mass on a zero-probability outcome"
    return float(((counts[keep] - exp[keep]) ** 2 / exp[keep]).sum()), int(keep.sum()) - 1


def test_chain_tree_is_the_chain_rule():
    """par_i = i - 1: node j+1 is draft slot j, its test uses u[j+1]; the
    final draw uses u[0].  The result equals the chain rule exactly."""
    rng = np.random.default_rng(0)
    for trial in range(200):
        B, K, V = 3, int(rng.integers(0, 6)), int(rng.integers(2, 9))
        T = float(rng.choice([0.5, 1.0, 1.7]))
        zp = rng.normal(0, 1.5, size=(B, K + 1, V))
        zq = rng.normal(0, 1.5, size=(B, K, V))
        x = rng.integers(0, V, size=(B, K))
        u = rng.random((B, K + 1))
        ref = oracle.verify_sampling(zp, zq, x, u, T)
        N = K + 1
        tok = np.zeros((B, N), dtype=np.int64)
        tok[:, 1:] = x
        par = np.tile(np.arange(-1, N - 1), (B, 1))
        zq_t = np.zeros((B, N, V))
        zq_t[:, :K] = zq                      # node j's children are drawn from the draft row of slot j
        ut = np.zeros((B, N))
        ut[:, 1:] = u[:, :K]
        ut[:, 0] = u[:, K]
        res = tv.verify_tree(zp, zq_t, tok, par, ut, T)
        assert np.array_equal(res["num_accepted"], ref["num_accepted"])
        assert np.array_equal(res["tokens"], ref["tokens"])


def test_residual_update_matches_the_lambda_closed_form():
    rng = np.random.default_rng(1)
    for _ in range(50):
        V = 12
        p = rng.dirichlet(np.ones(V))
        q = rng.dirichlet(np.ones(V))
        r = p.copy()
        for k in range(1, 5):
            res = np.maximum(0.0, r - q)
            if res.sum() == 0:
                break
            r = res / res.sum()
            assert np.allclose(r, tv.lambda_residual(p, q, k), atol=1e-12)


def two_level_tree(rng, n, V, k1, k2, q_root, q_child, iid=True):
    """Root with k1 children drawn from q_root; every child with k2 children
    drawn from q_child[its token].  Node order: root, level 1, level 2."""
    N = 1 + k1 + k1 * k2
    par = np.empty((n, N), dtype=np.int64)
    tok = np.zeros((n, N), dtype=np.int64)
    par[:, 0] = -1
    par[:, 1:1 + k1] = 0
    for i in range(k1):
        par[:, 1 + k1 + i * k2: 1 + k1 + (i + 1) * k2] = 1 + i

    def draw(qrow, m, k):
        if iid:
            return np.stack([rng.choice(V, size=m, p=qrow) for _ in range(k)], axis=1)
        # k distinct tokens in sampling order without replacement
        out = np.empty((m, k), dtype=np.int64)
        for s in range(m):
            out[s] = rng.choice(V, size=k, replace=False, p=qrow)
        return out

    tok[:, 1:1 + k1] = draw(q_root, n, k1)
    for i in range(k1):
        for t in range(V):
            sel = tok[:, 1 + i] == t
            if sel.any():
                tok[sel, 1 + k1 + i * k2: 1 + k1 + (i + 1) * k2] = draw(q_child[t], int(sel.sum()), k2)
    return tok, par


def run_two_level(seed, n, iid=True, k1=3, k2=2, V=6):
    rng = np.random.default_rng(seed)
    p_root = rng.dirichlet(np.ones(V) * 0.8)
    q_root = rng.dirichlet(np.ones(V) * 0.8)
    P2 = rng.dirichlet(np.ones(V) * 0.8, size=V)       # target row after token t
    Q2 = rng.dirichlet(np.ones(V) * 0.8, size=V)       # draft row after token t
    P3 = rng.dirichlet(np.ones(V) * 0.8, size=(V, V))  # target row after (t1, t2)
    tok, par = two_level_tree(rng, n, V, k1, k2, q_root, Q2, iid)
    N = tok.shape[1]
    zp = np.empty((n, N, V))
    zq = np.full((n, N, V), 0.0)
    zp[:, 0] = np.log(p_root)
    zq[:, 0] = np.log(q_root)
    for i in range(1, 1 + k1):
        zp[:, i] = np.log(P2[tok[:, i]])
        zq[:, i] = np.log(Q2[tok[:, i]])
    for i in range(1 + k1, N):
        zp[:, i] = np.log(P3[tok[:, par[0, i]], tok[:, i]])
    u = rng.random((n, N))
    res = tv.verify_tree(zp, zq, tok, par, u, 1.0)
    return res, p_root, P2


def test_emitted_tokens_follow_the_target():
    """Every emitted token ~ the target's next-token distribution given the
    emitted prefix: y1 ~ p_root; y2 | y1 = a ~ P2[a]."""
    n = 60_000
    res, p_root, P2 = run_two_level(5, n)
    y1 = res["tokens"][:, 0]
    s, df = chi2(np.bincount(y1, minlength=6), p_root)
    assert s < CRIT(df), (s, df)
    two = res["num_accepted"] >= 1
    for a in range(6):
        sel = two & (y1 == a)
        if sel.sum() < 500:
            continue
        s, df = chi2(np.bincount(res["tokens"][sel, 1], minlength=6), P2[a])
        assert s < CRIT(df), (a, s, df)


def test_children_without_replacement_break_the_claim():
    """Negative control: siblings drawn as distinct tokens are not i.i.d.
    draft samples, and the rule no longer reproduces the target."""
    n = 60_000
    res, p_root, _ = run_two_level(5, n, iid=False, k1=3)
    s, df = chi2(np.bincount(res["tokens"][:, 0], minlength=6), p_root)
    assert s > CRIT(df), (s, df)


def test_greedy_walk_on_hand_trees():
    V = 5
    # root argmax 2; children: node1 token 4, node2 token 2 (accepted), node3 token 2
    # node2's row argmax 0; its children: node4 token 1, node5 token 0 (accepted, a leaf)
    # node5's row argmax 3 -> bonus 3
    par = np.array([[-1, 0, 0, 0, 2, 2]])
    tok = np.array([[0, 4, 2, 2, 1, 0]])
    zp = np.full((1, 6, V), -1.0)
    zp[0, 0, 2] = 5.0
    zp[0, 2, 0] = 5.0
    zp[0, 5, 3] = 5.0
    zp[0, 3, 1] = 5.0                   # node3 is never visited (node2 comes first)
    res = tv.verify_tree(zp, None, tok, par, None, 0.0)
    assert res["num_accepted"].tolist() == [2]
    assert res["path"][0, :3].tolist() == [2, 5, -1]
    assert res["tokens"][0].tolist() == [2, 0, 3, -1, -1, -1]
    # no child matches at the root: only the root's argmax is emitted
    zp2 = zp.copy()
    zp2[0, 0] = [0.0, 9.0, 9.0, 0.0, 0.0]      # tie -> lowest id 1, no child carries 1
    res = tv.verify_tree(zp2, None, tok, par, None, 0.0)
    assert res["num_accepted"].tolist() == [0] and res["tokens"][0, 0] == 1


def test_invalid_trees_are_flagged():
    zp = np.zeros((3, 3, 4))
    u = np.full((3, 3), 0.5)
    par = np.array([[-1, 0, 0], [-1, 1, 0], [0, 0, 1]])      # ok / parent not before node / root has parent
    tok = np.array([[0, 1, 2], [0, 1, 2], [0, 1, 2]])
    res = tv.verify_tree(zp, zp, tok, par, u, 1.0)
    assert res["num_accepted"].tolist()[1:] == [-1, -1] and res["num_accepted"][0] >= 0
    tok2 = np.array([[0, 1, 9], [0, 1, 2], [0, 1, 2]])       # token outside [0, V)
    res = tv.verify_tree(zp, zp, tok2, np.tile(par[:1], (3, 1)), u, 1.0)
    assert res["num_accepted"][0] == -1 and (res["tokens"][0] == -1).all()
