"""CPU oracle of tree-shaped candidate verification.

TEST INFRASTRUCTURE, like the rest of ``oracle/``: only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may use it.

What the pages fix: [NALAR] "Speculative Decoding: Memverifikasi Token Draft
secara Paralel", section "Sampling eksak memerlukan aturan koreksi", names
tree-shaped candidates among the variants of the method and says that each
variant needs its own distribution claim: exactness of the chain rule does
not carry over by itself.  The acceptance ratio min(1, p/q) and the positive
residual max(0, p - q) of the same section, and the accepted-prefix rule of
"Penolakan memotong prefix yang diterima", are the building blocks.

Reading taken here (the plainest exact construction from those blocks; the
pages give no tree algorithm):

* a tree of N nodes per sequence: node 0 is the root (the position of the
  last committed token), node i >= 1 carries draft token t_i and a parent
  par_i < i;
* z_p row i: the target's logits after the path to node i (one row per node,
  from one tree-attention target pass); z_q row i: the draft distribution
  from which node i's children were drawn; p_i = softmax(z_p_i / T),
  q_i = softmax(z_q_i / T);
* the children of a node are independent draws from that node's q (with
  repetition allowed) -- the condition under which the rule below is exact;
* walk from the root.  At node c, working distribution r = p_c.  Try the
  children in ascending node index: child k with token x is accepted iff
  u_k < min(1, r(x) / q_c(x)); on rejection r <- max(0, r - q_c) / (its sum)
  (if that sum is 0, r is left as it was).  On acceptance the walk moves to
  the child (r restarts at the child's p).  When every child of c was
  rejected, the emitted token is y ~ r; when the accepted node has no
  children, y ~ p of that node (the bonus).  y is drawn by the inverse CDF
  of the chain rule on u_0;
* output: the tokens of the accepted nodes in walk order, then y; the
  accepted node indices (the cache entries to keep); their count n;
* q(x) = 0 with r(x) > 0 accepts, both zero rejects (as in the chain rule);
* T = 0: a child is accepted iff its token is the argmax of the current
  node's target row (ties to the lowest token id; the first such child in
  index order), y = the argmax of the last node's row;
* invalid input (a parent not in [0, i), a token outside [0, V)) marks the
  sequence: n = -1, every output -1.

Claim and pins (tests/test_tree_pins.py): a chain (par_i = i - 1) gives
exactly the chain rule's result for the same uniforms; every emitted token is
distributed as the target's next-token distribution given the emitted prefix
(chi-square at V = 6 on a two-level tree whose children are i.i.d. draft
samples); children drawn without replacement break it (negative control);
the greedy walk on hand-built trees; the residual update agrees with the
closed form r_k ~ max(0, p - lambda_k q), lambda_{k+1} = lambda_k + sum(max(0,
p - lambda_k q)).
"""
from __future__ import annotations

import numpy as np

from . import spec_oracle


def children_of(parents):
    """Children lists in ascending node index (None if the tree is invalid)."""
    N = len(parents)
    kids = [[] for _ in range(N)]
    if N == 0 or int(parents[0]) != -1:
        return None
    for i in range(1, N):
        pi = int(parents[i])
        if pi < 0 or pi >= i:
            return None
        kids[pi].append(i)
    return kids


def _walk_sampling(p, q, tokens, kids, u):
    """One sequence: p, q [N, V] probabilities; returns (path, y, margins)."""
    cur, path, accept_margins = 0, [], []
    zero_mass = False
    while True:
        r = p[cur]
        accepted = None
        for c in kids[cur]:
            x = int(tokens[c])
            qx, rx = q[cur][x], r[x]
            if qx > 0:
                a = min(1.0, rx / qx)
            else:
                a = 1.0 if rx > 0 else 0.0
            accept_margins.append(abs(u[c] - a))
            if u[c] < a:
                accepted = c
                break
            res = np.maximum(0.0, r - q[cur])
            S = res.sum()
            if S > 0:
                r = res / S
            else:
                zero_mass = True
        if accepted is None:
            dist = r
            break
        path.append(accepted)
        cur = accepted
        if not kids[cur]:
            dist = p[cur]
            break
    y, lo, hi, _ = spec_oracle.inverse_cdf(dist[None, :], np.array([u[0]]))
    return path, int(y[0]), dict(accept=accept_margins, draw_lo=float(lo[0]), draw_hi=float(hi[0]),
                                 draw_mass=float(dist[int(y[0])]), zero_mass=zero_mass)


def _walk_greedy(zp, tokens, kids):
    cur, path, gaps = 0, [], []
    while True:
        row = zp[cur]
        best = int(np.argmax(row))
        top2 = np.sort(row)[-2:] if len(row) > 1 else np.array([row[0], row[0]])
        gaps.append(float(top2[1] - top2[0]))
        nxt = next((c for c in kids[cur] if int(tokens[c]) == best), None)
        if nxt is None:
            return path, best, gaps
        path.append(nxt)
        cur = nxt


def verify_tree(z_p, z_q, tokens, parents, uniforms, temperature: float) -> dict:
    """Tree verification for a batch: z_p [B, N, V], z_q [B, N, V] (None at
    T = 0), tokens [B, N], parents [B, N], uniforms [B, N] (None at T = 0).

    Returns tokens [B, N] (accepted path tokens, y, then -1), path [B, N]
    (accepted node indices, then -1), num_accepted [B], and per sequence the
    margins (accept: |u - a| of every test made; draw_lo/draw_hi/draw_mass of
    the final draw) or, at T = 0, the top-2 gaps of the visited rows."""
    z_p = np.asarray(z_p, dtype=np.float64)
    B, N, V = z_p.shape
    out_tok = np.full((B, N), -1, dtype=np.int64)
    out_path = np.full((B, N), -1, dtype=np.int64)
    n_acc = np.full(B, -1, dtype=np.int64)
    info = []
    greedy = temperature == 0.0
    if not greedy:
        p_all = spec_oracle.softmax_t(z_p, temperature)
        q_all = spec_oracle.softmax_t(np.asarray(z_q, dtype=np.float64), temperature)
    for b in range(B):
        kids = children_of(parents[b])
        toks = np.asarray(tokens[b])
        if kids is None or any(int(toks[i]) < 0 or int(toks[i]) >= V for i in range(1, N)):
            info.append(None)
            continue
        if greedy:
            path, y, gaps = _walk_greedy(z_p[b], toks, kids)
            info.append(dict(top2_gap=gaps))
        else:
            path, y, m = _walk_sampling(p_all[b], q_all[b], toks, kids, np.asarray(uniforms[b], dtype=np.float64))
            info.append(m)
        n = len(path)
        n_acc[b] = n
        out_path[b, :n] = path
        out_tok[b, :n] = toks[path]
        out_tok[b, n] = y
    return dict(tokens=out_tok, path=out_path, num_accepted=n_acc, info=info)


def lambda_residual(p, q, k: int):
    """The closed form of k successive residual updates of p against the
    same q: max(0, p - lambda_k q) normalised, lambda_1 = 1,
    lambda_{j+1} = lambda_j + sum(max(0, p - lambda_j q))."""
    lam = 1.0
    for _ in range(k - 1):
        lam += np.maximum(0.0, p - lam * q).sum()
    r = np.maximum(0.0, p - lam * q)
    return r / r.sum()
