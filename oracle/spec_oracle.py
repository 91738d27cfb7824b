"""CPU oracle of the target-side verify-and-accept step of speculative decoding.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import or run
this module.  The product path (the C-ABI library and its Python binding)
never calls it and must fail loudly when its CUDA library is missing.

Everything is plain numpy in float64.  The steps follow the pages:

* [QH]  quochung.cyou, A.I category article on speculative decoding
        (sections "Hidden state", "Chọn token: greedy vs sampling",
        "Một vòng speculative decoding", "Modified rejection sampling" with its
        sub-sections "Giải pháp", "Khi reject thì lấy token từ đâu?",
        "Toàn bộ thuật toán cho một token", "Áp dụng thuật toán").
* [NALAR] "Speculative Decoding: Memverifikasi Token Draft secara Paralel"
        (sections "Sampling eksak memerlukan aturan koreksi",
        "Penolakan memotong prefix yang diterima").
* [MLC] "57 Speculative Decoding" (ml-canon-ru), section "Идея и механизм"
        and the acceptance / residual / exactness equations under
        "Приёмка и почему распределение НЕ портится".

Readings where the pages are silent:
  - temperature: p = softmax(z / T) for target and draft alike; T = 0 is the
    greedy limit (argmax, ties to the lowest token id);
  - accept iff u < a (strict; [QH] prints u <= a, [MLC] prints random() < a;
    equal in measure);
  - q(x) = 0 with p(x) > 0 accepts, both zero rejects;
  - the correction / bonus draw is the inverse CDF over ascending token ids:
    y = smallest v with C_v > u * S, C_v = sum_{t <= v} r_t, S = sum r; if
    rounding leaves no such v, y = the largest v with r_v > 0;
  - a rejection whose residual mass is exactly zero (impossible in exact
    arithmetic) draws from p at that position instead;
  - rows per sequence: target rows j = 0..K, row j scores draft slot j,
    row K is the bonus distribution; uniforms [B][K+1]: K accept uniforms
    and one draw uniform shared by the correction and the bonus draw (only
    one of them happens per round).

Pins (tests/test_oracle_pins.py): the 60/30/10 worked example (ratios,
1000-trial counts, residual, final counts and the wrong-fix counterexample),
the 45/25/20 example, closed-form acceptance sum_x min(p, q), chi-square of
the output against p over 10^6 draws at V=16, brute-force path enumeration
at V=4, K=2, the greedy worked rounds, one-hot reduction of sampling to
greedy, and LM-head special cases (identity slice, one-hot hidden state).
No function here is left without a pin.
"""
from __future__ import annotations

import numpy as np


# ---------------------------------------------------------------------------
# S1: LM head ([QH] "Hidden state": the last hidden state, 4096 or 8192
# values, goes through the LM head to a score for every vocabulary token).
# ---------------------------------------------------------------------------
def lm_head(hidden, W, vocab_chunk: int = 4096) -> np.ndarray:
    """z[m, v] = sum_k hidden[m, k] * W[v, k], in float64.

    ``hidden`` [M, d] and ``W`` [V, d] hold the bf16 values exactly (any float
    dtype); they are upcast to float64 here, one vocabulary chunk of W at a
    time so that a large head needs only a bounded float64 copy."""
    h = np.asarray(hidden, dtype=np.float64)
    V = W.shape[0]
    z = np.empty((h.shape[0], V), dtype=np.float64)
    for v0 in range(0, V, vocab_chunk):
        Wc = np.asarray(W[v0:v0 + vocab_chunk], dtype=np.float64)
        z[:, v0:v0 + Wc.shape[0]] = h @ Wc.T
    return z


# ---------------------------------------------------------------------------
# S2: temperature softmax ([QH] "Forward pass": the scores form a probability
# distribution whose entries sum to 100%; "Chọn token": sampling, possibly at
# a low temperature).
# ---------------------------------------------------------------------------
def softmax_t(z, temperature: float) -> np.ndarray:
    """softmax(z / T) along the last axis, float64, max-shifted."""
    x = np.asarray(z, dtype=np.float64) / float(temperature)
    x = x - x.max(axis=-1, keepdims=True)
    e = np.exp(x)
    return e / e.sum(axis=-1, keepdims=True)


# ---------------------------------------------------------------------------
# S3: acceptance probability ([QH] "Giải pháp": accept_probability(token) =
# min(1, p(token) / q(token)); [NALAR] a(x) = min(1, p(x)/q(x)); [MLC] alpha(x)).
# ---------------------------------------------------------------------------
def accept_probability(p_x, q_x) -> np.ndarray:
    p_x = np.asarray(p_x, dtype=np.float64)
    q_x = np.asarray(q_x, dtype=np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(q_x > 0, p_x / np.where(q_x > 0, q_x, 1.0), np.where(p_x > 0, np.inf, 0.0))
    return np.minimum(1.0, ratio)


# ---------------------------------------------------------------------------
# S5: residual distribution ([QH] "Khi reject thì lấy token từ đâu?":
# residual(token) = max(0, p(token) - q(token)), then normalised;
# [NALAR] r(x) proportional to max(0, p(x) - q(x)); [MLC] norm(max(0, p - q))).
# ---------------------------------------------------------------------------
def residual(p_row, q_row) -> np.ndarray:
    """Unnormalised residual max(0, p - q) (normalisation is the draw's job)."""
    return np.maximum(0.0, np.asarray(p_row, dtype=np.float64) - np.asarray(q_row, dtype=np.float64))


# ---------------------------------------------------------------------------
# S6: the draw ([QH] "Toàn bộ thuật toán cho một token": sample the correction
# from normalize(max(0, p - q)); "Chọn token": sampling is a die with one face
# per unit of probability).  Inverse CDF in ascending token id on one supplied
# uniform is the reading taken for "sample".
# ---------------------------------------------------------------------------
def inverse_cdf(r, u):
    """Draw from the (unnormalised, non-negative) rows ``r`` [N, V] with
    uniforms ``u`` [N] in [0, 1).

    Returns (y, lo_margin, hi_margin, S): y = smallest v with C_v > u*S where
    C_v is the running sum of r in ascending v; the margins are the distances
    (t - C_{y-1}) / S and (C_y - t) / S of t = u*S from the two CDF boundaries
    that enclose it (C_{-1} = 0)."""
    r = np.atleast_2d(np.asarray(r, dtype=np.float64))
    u = np.atleast_1d(np.asarray(u, dtype=np.float64))
    C = np.cumsum(r, axis=-1)
    S = C[:, -1]
    t = u * S
    above = C > t[:, None]
    found = above.any(axis=-1)
    y = np.argmax(above, axis=-1)
    if not found.all():
        # rounding left t at or beyond the total: take the last token with mass
        V = r.shape[1]
        last_pos = V - 1 - np.argmax((r > 0)[:, ::-1], axis=-1)
        y = np.where(found, y, last_pos)
    rows = np.arange(r.shape[0])
    c_hi = C[rows, y]
    c_lo = np.where(y > 0, C[rows, np.maximum(y - 1, 0)], 0.0)
    with np.errstate(divide="ignore", invalid="ignore"):
        lo = np.where(S > 0, (t - c_lo) / S, 0.0)
        hi = np.where(S > 0, (c_hi - t) / S, 0.0)
    return y, lo, hi, S


# ---------------------------------------------------------------------------
# S3-S7: one verify round ([QH] "Áp dụng thuật toán": left to right over the
# drafts, stop at the first rejection, resample it from the residual and
# drop the rest; if all K are accepted, one bonus token from the target
# distribution after the last draft.  [NALAR] "Penolakan memotong prefix
# yang diterima"; [MLC] "Идея и механизм").
# ---------------------------------------------------------------------------
def verify_sampling(z_p, z_q, draft_tokens, uniforms, temperature: float) -> dict:
    """The sampling (T > 0) verify round for a batch of sequences.

    z_p [B, K+1, V] target logits (row j scores draft slot j, row K = bonus),
    z_q [B, K, V] draft logits, draft_tokens [B, K] ints, uniforms [B, K+1]
    (u[:, :K] accept tests, u[:, K] the draw).

    Returns a dict of numpy arrays:
      tokens [B, K+1] (accepted drafts, then the correction or bonus token,
      then -1), num_accepted [B], and diagnostics: p_x, q_x, accept_prob [B, K],
      logZ_p [B, K+1], logZ_q [B, K] (log-normalisers of z/T), accept_margin
      [B, K] = |u_j - a_j|, residual_mass [B] (sum of the drawn row; 1 for the
      bonus), draw_lo / draw_hi [B] (normalised distances of u*S from the CDF
      boundaries around the drawn token), draw_mass [B] (normalised mass of
      the drawn token), from_p_fallback [B] (zero-mass rejections)."""
    z_p = np.asarray(z_p, dtype=np.float64)
    z_q = np.asarray(z_q, dtype=np.float64)
    x = np.asarray(draft_tokens, dtype=np.int64)
    u = np.asarray(uniforms, dtype=np.float64)
    B, K1, V = z_p.shape
    K = K1 - 1
    T = float(temperature)
    assert T > 0.0
    assert z_q.shape == (B, K, V) and x.shape == (B, K) and u.shape == (B, K + 1)

    p = softmax_t(z_p, T)
    q = softmax_t(z_q, T) if K > 0 else np.zeros((B, 0, V))
    zp_s = z_p / T
    zq_s = z_q / T
    logZ_p = zp_s.max(axis=-1) + np.log(np.exp(zp_s - zp_s.max(axis=-1, keepdims=True)).sum(axis=-1))
    logZ_q = (zq_s.max(axis=-1) + np.log(np.exp(zq_s - zq_s.max(axis=-1, keepdims=True)).sum(axis=-1))
              if K > 0 else np.zeros((B, 0)))

    bi = np.arange(B)[:, None]
    ji = np.arange(K)[None, :]
    p_x = p[bi, ji, x] if K > 0 else np.zeros((B, 0))
    q_x = q[bi, ji, x] if K > 0 else np.zeros((B, 0))
    a = accept_probability(p_x, q_x)

    # first rejection, left to right
    num_accepted = np.full(B, K, dtype=np.int64)
    still = np.ones(B, dtype=bool)
    for j in range(K):
        accept_j = u[:, j] < a[:, j]
        rejected_here = still & ~accept_j
        num_accepted[rejected_here] = j
        still &= accept_j

    rows = np.arange(B)
    n = num_accepted
    rejected = n < K
    # residual row at the first rejection; the bonus row p_K when all K pass
    if K > 0:
        jr = np.minimum(n, K - 1)
        r_rej = residual(p[rows, jr], q[rows, jr])
    else:
        r_rej = np.zeros((B, V))
    r = np.where(rejected[:, None], r_rej, p[:, K])
    from_p = rejected & ~(r.sum(axis=-1) > 0.0)
    r = np.where(from_p[:, None], p[rows, np.minimum(n, K)], r)
    y, lo, hi, S = inverse_cdf(r, u[:, K])

    # emit: accepted drafts, then the drawn token, then -1
    pos = np.arange(K + 1)[None, :]
    x_pad = np.concatenate([x, np.full((B, 1), -1, dtype=np.int64)], axis=1)
    tokens = np.where(pos < n[:, None], x_pad, -1)
    tokens[rows, n] = y
    with np.errstate(divide="ignore", invalid="ignore"):
        draw_mass = np.where(S > 0, r[rows, y] / S, 0.0)
    return dict(tokens=tokens, num_accepted=n, p_x=p_x, q_x=q_x, accept_prob=a,
                logZ_p=logZ_p, logZ_q=logZ_q, accept_margin=np.abs(u[:, :K] - a),
                residual_mass=S, draw_lo=lo, draw_hi=hi, draw_mass=draw_mass,
                from_p_fallback=from_p)


# ---------------------------------------------------------------------------
# S8: greedy verify ([QH] "Chọn token": greedy takes the highest-probability
# token; "Một vòng speculative decoding" Bước 3: compare left to right, the
# first mismatch is replaced by the target's token and the tail discarded;
# Blockwise Parallel Decoding: draft = target argmax -> accept, else reject).
# ---------------------------------------------------------------------------
def argmax_lowest(z) -> np.ndarray:
    """argmax along the last axis, ties to the lowest index."""
    z = np.asarray(z, dtype=np.float64)
    return np.argmax(z, axis=-1)


def verify_greedy(z_p, draft_tokens) -> dict:
    """T = 0 round: accept the longest prefix of drafts that equal the target
    argmax of their row, then emit the target argmax of the next row (row K,
    the bonus, when every draft matched).

    Returns tokens [B, K+1], num_accepted [B], argmax [B, K+1] and top2_gap
    [B, K+1] (difference of the two largest logits of each row)."""
    z_p = np.asarray(z_p, dtype=np.float64)
    x = np.asarray(draft_tokens, dtype=np.int64)
    B, K1, V = z_p.shape
    K = K1 - 1
    g = argmax_lowest(z_p)
    num_accepted = np.full(B, K, dtype=np.int64)
    still = np.ones(B, dtype=bool)
    for j in range(K):
        match = x[:, j] == g[:, j]
        num_accepted[still & ~match] = j
        still &= match
    rows = np.arange(B)
    pos = np.arange(K + 1)[None, :]
    x_pad = np.concatenate([x, np.full((B, 1), -1, dtype=np.int64)], axis=1)
    tokens = np.where(pos < num_accepted[:, None], x_pad, -1)
    tokens[rows, num_accepted] = g[rows, num_accepted]
    if V >= 2:
        part = np.partition(z_p, V - 2, axis=-1)
        top2_gap = part[..., V - 1] - part[..., V - 2]
    else:
        top2_gap = np.full((B, K1), np.inf)
    return dict(tokens=tokens, num_accepted=num_accepted, argmax=g, top2_gap=top2_gap)


# ---------------------------------------------------------------------------
# Whole step from hidden states ([QH] "Một vòng speculative decoding" Bước 2:
# the target scores all candidate positions in one pass; the verify round
# then runs on those scores).
# ---------------------------------------------------------------------------
def spec_verify(hidden, W, draft_logits, draft_tokens, uniforms, temperature: float,
                B: int, K: int) -> dict:
    """hidden [B*(K+1), d], W [V, d], draft_logits [B*K, V] (T > 0),
    draft_tokens [B, K], uniforms [B, K+1] (T > 0)."""
    z = lm_head(hidden, W)
    V = z.shape[1]
    z_p = z.reshape(B, K + 1, V)
    if temperature == 0.0:
        res = verify_greedy(z_p, draft_tokens)
    else:
        z_q = np.asarray(draft_logits, dtype=np.float64).reshape(B, K, V)
        res = verify_sampling(z_p, z_q, draft_tokens, uniforms, temperature)
    res["target_logits"] = z
    return res


def acceptance_rate(p, q) -> float:
    """Closed form of the per-position acceptance probability, sum_x min(p, q)
    ([QH] "Giải pháp": 900 of 1000 proposals accepted = sum of min(p, q))."""
    return float(np.minimum(np.asarray(p, dtype=np.float64), np.asarray(q, dtype=np.float64)).sum())
