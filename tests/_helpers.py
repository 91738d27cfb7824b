"""Shared test helpers: run the oracle on the same seeded inputs as the CUDA
path and compare the two under the stated tolerances.

Tolerances (fp32 kernels against the fp64 oracle):
  * LM-head logits: |z_gpu - z_oracle| <= 1e-3 (absolute);
  * probabilities and log-normalisers of the debug output: relative 1e-5;
  * accept decisions: identical, except where the oracle's |u_j - a_j| < 1e-4
    (the decision is within rounding of its threshold; counted);
  * the drawn token: identical, except where u lies within DRAW_BAND of a
    boundary of the drawn token's CDF step, measured relative to that step's
    width (counted); the band is relative because an f32 CDF step is only
    resolved to a fraction of its own width, however small the step;
  * greedy: bit-exact, except rows whose two largest oracle logits are closer
    than twice the measured logit error (counted; only there may the f32
    argmax legitimately differ).

When the target logits come from the GPU's own f32 LM head (the whole step)
they differ from the oracle's fp64 logits by the head's rounding (measured,
~2e-6 at most), which moves each CDF boundary by a random amount far below a
token's step but not always below 1e-4 of it.  There a draw outside the
relative band may differ ("moved by the logits"); it is admissible when its
uniform lies within 1e-4 (in units of u) of the decision threshold -- the
literal band of the stated tolerance -- and every such difference is counted:
all differing draws together must stay under 0.1 % of the draws.  With
identical logits (the from-logits entry points) no such exemption applies.
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch

import oracle

LOGIT_ATOL = 1e-3
PROB_RTOL = 1e-5
ACCEPT_BAND = 1e-4
DRAW_BAND = 1e-4


def t32(T: float) -> float:
    """The temperature as the C ABI receives it (an f32), for the oracle."""
    return float(np.float32(T))


def np64(t) -> np.ndarray:
    return t.detach().to("cpu").double().numpy() if t is not None else None


def np_int(t) -> np.ndarray:
    return t.detach().to("cpu").numpy().astype(np.int64)


def oracle_sampling_from_logits(zp, zq, x, u, B, K, V, T):
    return oracle.verify_sampling(np.asarray(zp).reshape(B, K + 1, V), np.asarray(zq).reshape(B, K, V),
                                  x, u, T)


def compare_sampling(tok_gpu, n_gpu, ref, K, band_accept=ACCEPT_BAND, band_draw=DRAW_BAND, own_logits=False):
    """Compare GPU tokens / accept counts with the oracle's result dict.

    ``own_logits``: the GPU computed its own target logits (the whole step);
    a draw outside the relative band may then differ if its uniform lies
    within ``band_draw`` (absolute) of the threshold (module docstring).

    Returns a dict of counts: ``band_cases`` = sequences whose uniform lies in
    the band of a decision they reached (accept: |u - a| < 1e-4; draw: within
    1e-4 of the drawn token's step from one of its boundaries); ``mismatches``
    = sequences whose result differs (``moved_by_logits`` of them outside the
    relative band).  Raises AssertionError on a mismatch no band explains."""
    tok_gpu = np.asarray(tok_gpu)
    n_gpu = np.asarray(n_gpu)
    B = len(n_gpu)
    stats = dict(sequences=B, draws=B, accept_tests=0, accept_exempt=0, draw_exempt=0,
                 draw_mismatch_exempt=0, accept_mismatch_exempt=0, band_cases=0, mismatches=0, moved_by_logits=0)
    for b in range(B):
        n_o = int(ref["num_accepted"][b])
        n_g = int(n_gpu[b])
        assert n_g >= 0, f"sequence {b} flagged invalid by the GPU"
        tests = min(n_o, n_g, K - 1) + 1 if K > 0 else 0
        stats["accept_tests"] += tests
        margins = ref["accept_margin"][b, :tests] if K > 0 else np.zeros(0)
        near = bool((margins < band_accept).any())
        stats["accept_exempt"] += int(near)
        stats["band_cases"] += int(near)
        if n_g != n_o:
            assert near, (f"sequence {b}: accepted {n_g} on the GPU vs {n_o} in the oracle; "
                          f"accept margins {margins}")
            stats["accept_mismatch_exempt"] += 1
            stats["mismatches"] += 1
            continue
        np.testing.assert_array_equal(tok_gpu[b, :n_o], ref["tokens"][b, :n_o])
        assert (tok_gpu[b, n_o + 1:] == -1).all()
        width = ref["draw_mass"][b]
        margin = min(ref["draw_lo"][b], ref["draw_hi"][b])
        draw_near = margin < band_draw * width
        stats["draw_exempt"] += int(draw_near)
        stats["band_cases"] += int(draw_near and not near)
        if tok_gpu[b, n_o] != ref["tokens"][b, n_o]:
            stats["mismatches"] += 1
            if draw_near:
                stats["draw_mismatch_exempt"] += 1
            else:
                assert own_logits and margin < band_draw, (
                    f"sequence {b}: drew {tok_gpu[b, n_o]} on the GPU vs {ref['tokens'][b, n_o]} in the oracle; "
                    f"margin {margin:.3e} of a step {width:.3e}")
                stats["moved_by_logits"] += 1
    return stats


def add_stats(total: dict, st: dict) -> dict:
    for k, v in st.items():
        total[k] = total.get(k, 0) + v
    return total


def compare_debug(dbg_gpu, ref, n_gpu, K, T=1.0, logit_err=0.0, rtol=PROB_RTOL):
    """Probabilities and log-normalisers reported by the GPU against the oracle.

    With identical logits (logit_err = 0) the bound is rel 1e-5.  When the
    target logits come from the GPU's own LM head they differ from the
    oracle's by up to logit_err (measured, <= 1e-3), which moves log p by at
    most 2*logit_err/T and log Z_p by at most logit_err/T; the bound widens
    by exactly that.  Draft-side quantities (q, log Z_q) are inputs and keep
    rel 1e-5."""
    dbg = np.asarray(dbg_gpu, dtype=np.float64)
    B = dbg.shape[0]
    dp = 2.0 * logit_err / T
    if K > 0:
        np.testing.assert_allclose(dbg[:, :K, 0], ref["p_x"], rtol=rtol + dp, atol=0)
        np.testing.assert_allclose(dbg[:, :K, 1], ref["q_x"], rtol=rtol, atol=0)
        np.testing.assert_allclose(dbg[:, :K, 2], ref["accept_prob"], rtol=rtol + dp, atol=0)
        np.testing.assert_allclose(dbg[:, :K, 4], ref["logZ_q"], rtol=rtol, atol=1e-6)
    np.testing.assert_allclose(dbg[:, :, 3], ref["logZ_p"], rtol=rtol, atol=1e-6 + logit_err / T)
    n = np.asarray(n_gpu)
    for b in range(B):
        if n[b] == ref["num_accepted"][b]:
            np.testing.assert_allclose(dbg[b, n[b], 5], ref["residual_mass"][b], rtol=rtol, atol=1e-9 + dp)


def compare_greedy(tok_gpu, n_gpu, ref, logit_err=0.0):
    """Greedy results must be identical.  The only admissible difference is a
    row whose two largest oracle logits are within 2*logit_err (+1e-12) of
    each other, where the GPU's f32 logits (off by at most logit_err) may
    order them the other way; such sequences are counted."""
    tok_gpu = np.asarray(tok_gpu)
    n_gpu = np.asarray(n_gpu)
    B = len(n_gpu)
    band = 2.0 * logit_err + 1e-12
    near_rows, mismatched = 0, 0
    for b in range(B):
        n_o = int(ref["num_accepted"][b])
        rows = ref["top2_gap"][b, :min(n_o, max(int(n_gpu[b]), 0)) + 1]
        near = bool((rows <= band).any())
        near_rows += int(near)
        same = int(n_gpu[b]) == n_o and np.array_equal(tok_gpu[b], ref["tokens"][b])
        if not same:
            assert near, (f"sequence {b}: GPU {tok_gpu[b].tolist()} (n={int(n_gpu[b])}) vs oracle "
                          f"{ref['tokens'][b].tolist()} (n={n_o}); top-2 gaps {rows}")
            mismatched += 1
    return dict(sequences=B, near_ties=near_rows, mismatched_near_ties=mismatched)


def logits_error(z_gpu: np.ndarray, z_ref: np.ndarray) -> dict:
    d = z_gpu - z_ref
    return dict(max_abs=float(np.abs(d).max()), mean=float(d.mean()), rms=float(np.sqrt((d * d).mean())))


def cuda_inputs(inputs: dict) -> dict:
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inputs.items()}


GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_golden(name):
    """A fixture under tests/golden/: lines "key value value ...", '#' comments."""
    out = {}
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            out[key] = np.array([float(v) for v in vals])
    return out


def load_golden_text(name):
    """Like :func:`load_golden`, values kept as strings."""
    out = {}
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            out[key] = vals
    return out
