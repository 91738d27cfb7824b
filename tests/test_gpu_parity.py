"""Parity of the CUDA path (through the C ABI) with the fp64 CPU oracle.

Every case draws seeded synthetic inputs once, runs the library and the
oracle on the same bytes, and compares under the tolerances of _helpers.
Small cases span several tiles and a ragged tail; the full-size cases run the
B1 and headline workloads in the launch configuration the benchmark times
(the larger workloads, every sequence, and the repeated headline draws are in
test_gpu_full_size.py).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_67_gb300 as sv
from speculative_decoding_verification_67_gb300 import synth

from _helpers import (DRAW_BAND, LOGIT_ATOL, compare_debug, compare_greedy, compare_sampling, logits_error, np64, np_int,
                      t32)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from speculative_decoding_verification_67_gb300 import _build
    _build.build()
    sv.library()


def _run_head_case(w, seed=None, keep_debug=True):
    inp = synth.make_inputs(w, device="cuda", seed=seed)
    B, K, d, V, T = w.B, w.K, w.d, w.V, w.temperature
    logits = torch.empty((B * (K + 1), V), dtype=torch.float32, device="cuda") if T > 0 else None
    dbg = torch.zeros((B, K + 1, sv.SPEC_DEBUG_FIELDS), dtype=torch.float32, device="cuda")
    tok, n = sv.spec_verify(inp["hidden"], inp["W"], inp["draft_logits"], inp["draft_tokens"], inp["uniforms"], T,
                            out_target_logits=logits, out_debug=dbg if keep_debug else None)
    torch.cuda.synchronize()
    return inp, tok, n, logits, dbg


# ---------------------------------------------------------------- LM head
@pytest.mark.parametrize("M,d,V", [(1, 64, 128), (6, 4096, 1000), (7, 200, 1000), (40, 512, 3001),
                                   (100, 1024, 2500), (300, 256, 777), (576, 512, 1500), (1280, 128, 700)])
def test_lm_head_matches_oracle(M, d, V):
    g = torch.Generator(device="cuda").manual_seed(1000 + M + d + V)
    h = torch.randn((M, d), generator=g, device="cuda").to(torch.bfloat16)
    W = (torch.randn((V, d), generator=g, device="cuda") / math.sqrt(d)).to(torch.bfloat16)
    z = sv.spec_lm_head(h, W)
    torch.cuda.synchronize()
    ref = oracle.lm_head(np64(h), np64(W))
    err = logits_error(np64(z), ref)
    print(f"\nlm_head M={M} d={d} V={V}: {err}")
    assert err["max_abs"] <= LOGIT_ATOL, err


def test_lm_head_identity_slice_is_exact():
    M, d, V = 40, 256, 200
    h = torch.randn((M, d), device="cuda").to(torch.bfloat16)
    W = torch.eye(d, device="cuda")[:V].to(torch.bfloat16).contiguous()
    z = sv.spec_lm_head(h, W)
    torch.cuda.synchronize()
    assert torch.equal(z, h[:, :V].float())
    e = torch.zeros((d, d), device="cuda")
    e.fill_diagonal_(1.0)
    W2 = torch.randn((V, d), device="cuda").to(torch.bfloat16)
    z2 = sv.spec_lm_head(e.to(torch.bfloat16), W2)
    torch.cuda.synchronize()
    assert torch.equal(z2, W2.float().t())


def test_lm_head_is_deterministic():
    w = synth.custom("det", B=8, K=4, d=1024, V=5000, temperature=0.8)
    inp = synth.make_inputs(w, device="cuda")
    a = sv.spec_lm_head(inp["hidden"], inp["W"])
    b = sv.spec_lm_head(inp["hidden"], inp["W"])
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("B,K,T,d", [(2, 3, 0.9, 512),      # 16-column precise head, stream-K split tiles
                                     (8, 4, 0.8, 512),      # 48 columns
                                     (40, 7, 1.1, 512),     # large-batch head (two chunks of 160), draft-row pass
                                     (16, 4, 0.9, 4096),    # large-batch head, draft rows on its side warps
                                     (40, 7, 0.0, 512)])    # large-batch greedy (transposed argmax epilogue)
def test_whole_step_is_deterministic(B, K, T, d):
    """The same inputs twice through the whole step (LM head, statistics,
    decision, draw): identical logits, tokens, counts and debug fields.  The
    schedules fix every summation order (stream-K splits, per-CTA running
    partials, the merges), so nothing may depend on timing."""
    w = synth.custom("det_step", B=B, K=K, d=d, V=7001, temperature=T, seed=B + K)
    inp = synth.make_inputs(w, device="cuda")
    outs = []
    for _ in range(2):
        logits = torch.empty((B * (K + 1), w.V), dtype=torch.float32, device="cuda") if T > 0 else None
        dbg = torch.zeros((B, K + 1, sv.SPEC_DEBUG_FIELDS), dtype=torch.float32, device="cuda")
        tok, n = sv.spec_verify(inp["hidden"], inp["W"], inp["draft_logits"], inp["draft_tokens"], inp["uniforms"], T,
                                out_target_logits=logits, out_debug=dbg)
        torch.cuda.synchronize()
        outs.append((tok.clone(), n.clone(), dbg.clone(), None if logits is None else logits.clone()))
    (t1, n1, d1, z1), (t2, n2, d2, z2) = outs
    assert torch.equal(t1, t2) and torch.equal(n1, n2) and torch.equal(d1, d2)
    if z1 is not None:
        assert torch.equal(z1, z2)


# ---------------------------------------------------------------- sampling from logits
def _from_logits_case(B, K, V, T, seed, std=2.0, noise=0.5):
    g = torch.Generator(device="cuda").manual_seed(seed)
    zp = torch.randn((B * (K + 1), V), generator=g, device="cuda") * std
    zq = (zp.view(B, K + 1, V)[:, :K] + noise * torch.randn((B, K, V), generator=g, device="cuda")).reshape(B * K, V)
    x = synth.gumbel_max_tokens(zq, T, g).view(B, K).contiguous() if K > 0 else \
        torch.zeros((B, 0), dtype=torch.int32, device="cuda")
    u = torch.rand((B, K + 1), generator=g, device="cuda")
    return zp.contiguous(), zq.contiguous(), x, u


@pytest.mark.parametrize("B,K,V,T", [(1, 4, 1000, 1.0), (64, 4, 1000, 1.0), (33, 7, 8193, 0.8),
                                     (16, 0, 5000, 1.0), (8, 32, 3000, 1.3), (200, 3, 1001, 0.7),
                                     # rows of 4096-token chunks: 9 chunks on 5 CTAs (the last CTA's
                                     # second chunk empty), 25 on 13, 32 on 16, and 35 (no cluster)
                                     (3, 4, 36000, 0.9), (3, 3, 100000, 1.0), (2, 4, 131072, 0.8),
                                     (2, 3, 140000, 1.0),
                                     # 40 x 35 chunks exceed any residency (8 CTAs x 152 SMs): several
                                     # chunks per CTA, the last group of a row shorter
                                     (40, 1, 140000, 0.9)])
def test_verify_from_logits_matches_oracle(B, K, V, T):
    zp, zq, x, u = _from_logits_case(B, K, V, T, seed=B * 131 + K * 7 + V)
    dbg = torch.zeros((B, K + 1, sv.SPEC_DEBUG_FIELDS), device="cuda")
    tok, n = sv.spec_verify_from_logits(zp, zq, x, u, T, out_debug=dbg)
    torch.cuda.synchronize()
    ref = oracle.verify_sampling(np64(zp).reshape(B, K + 1, V), np64(zq).reshape(B, K, V), np_int(x), np64(u), t32(T))
    st = compare_sampling(np_int(tok), np_int(n), ref, K)
    print(f"\nfrom_logits B={B} K={K} V={V} T={T}: {st}")
    compare_debug(np64(dbg), ref, np_int(n), K, T)


# Statistics passes with at least four (row, 4096-token) units per SM and rows
# on 16-byte boundaries stream through the bulk-copy ring (two warps a stage);
# smaller ones use the many-warp form.  The ring's cases: a last chunk of 4
# tokens (a partial block of one vector), exact chunks, a last chunk of one
# whole 1024-token block.
@pytest.mark.parametrize("B,K,V,T", [(64, 4, 16388, 0.9), (48, 4, 12288, 1.1), (40, 3, 33792, 1.0),
                                     (32, 8, 20484, 0.7)])
def test_statistics_pass_streaming_form(B, K, V, T):
    zp, zq, x, u = _from_logits_case(B, K, V, T, seed=B * 7 + V)
    units = (B * (K + 1) + B * K) * ((V + 4095) // 4096)
    assert units >= 4 * torch.cuda.get_device_properties(0).multi_processor_count and V % 4 == 0
    outs = []
    for _ in range(2):
        dbg = torch.zeros((B, K + 1, sv.SPEC_DEBUG_FIELDS), device="cuda")
        tok, n = sv.spec_verify_from_logits(zp, zq, x, u, T, out_debug=dbg)
        torch.cuda.synchronize()
        outs.append((tok.clone(), n.clone(), dbg.clone()))
    assert all(torch.equal(outs[0][i], outs[1][i]) for i in range(3))   # deterministic
    tok, n, dbg = outs[0]
    ref = oracle.verify_sampling(np64(zp).reshape(B, K + 1, V), np64(zq).reshape(B, K, V), np_int(x), np64(u), t32(T))
    st = compare_sampling(np_int(tok), np_int(n), ref, K)
    print(f"\nstreaming statistics B={B} K={K} V={V} T={T}: {st}")
    compare_debug(np64(dbg), ref, np_int(n), K, T)


def test_statistics_pass_streaming_form_nonfinite():
    """A NaN target logit and an infinite draft logit in the ring form mark
    only their sequences; the others match the oracle."""
    B, K, V, T = 64, 4, 16388, 1.0
    zp, zq, x, u = _from_logits_case(B, K, V, T, seed=77)
    zp[5 * (K + 1) + 1, 16385] = float("nan")      # in the last, 4-token chunk
    zq[9 * K + 2, 4097] = float("inf")             # in a whole chunk
    ws = torch.empty(sv.from_logits_workspace_bytes(B, K, V, T), dtype=torch.uint8, device="cuda")
    tok, n = sv.spec_verify_from_logits(zp, zq, x, u, T, workspace=ws)
    assert sv.read_error(ws) & sv.DEVERR_NONFINITE
    n, tok = np_int(n), np_int(tok)
    assert n[5] == -1 and n[9] == -1 and (tok[5] == -1).all() and (tok[9] == -1).all()
    keep = [b for b in range(B) if b not in (5, 9)]
    z3, q3 = np64(zp).reshape(B, K + 1, V)[keep], np64(zq).reshape(B, K, V)[keep]
    ref = oracle.verify_sampling(z3, q3, np_int(x)[keep], np64(u)[keep], t32(T))
    compare_sampling(tok[keep], n[keep], ref, K)


def _degenerate_case(kind, B=16, K=4, V=300, T=1.0, seed=0):
    """Target / draft logit rows of a degenerate shape, drafts drawn from q
    (Gumbel-max in float64), uniforms U[0, 1)."""
    g = torch.Generator().manual_seed(seed)
    if kind == "v1":
        V = 1
        zp = torch.zeros((B * (K + 1), V), dtype=torch.float64)
        zq = torch.zeros((B * K, V), dtype=torch.float64)
    elif kind == "uniform":
        zp = torch.zeros((B * (K + 1), V), dtype=torch.float64)
        zq = torch.zeros((B * K, V), dtype=torch.float64)
    elif kind == "p_equals_q":
        zp = torch.randn((B * (K + 1), V), generator=g, dtype=torch.float64) * 2
        zq = zp.view(B, K + 1, V)[:, :K].reshape(B * K, V).clone()
    elif kind == "spikes":
        # target and draft each put (all but) all mass on one token, different ones
        zp = torch.full((B * (K + 1), V), -1e30, dtype=torch.float64)
        zq = torch.full((B * K, V), -1e30, dtype=torch.float64)
        zp[torch.arange(B * (K + 1)), torch.randint(0, V, (B * (K + 1),), generator=g)] = 0.0
        zq[torch.arange(B * K), torch.randint(0, V, (B * K,), generator=g)] = 0.0
    else:  # random logits at an extreme temperature
        zp = torch.randn((B * (K + 1), V), generator=g, dtype=torch.float64) * 2
        zq = (zp.view(B, K + 1, V)[:, :K].reshape(B * K, V)
              + 0.5 * torch.randn((B * K, V), generator=g, dtype=torch.float64))
    zp, zq = zp.float(), zq.float()
    x = synth.gumbel_max_tokens(zq.double(), T, g).view(B, K)
    u = torch.rand((B, K + 1), generator=g, dtype=torch.float32)
    return zp.cuda(), zq.cuda(), x.cuda(), u.cuda(), V


@pytest.mark.parametrize("kind,T", [("v1", 1.0), ("uniform", 1.0), ("p_equals_q", 0.7), ("spikes", 1.0),
                                    ("random", 0.05), ("random", 25.0)])
def test_degenerate_distributions(kind, T):
    """V = 1; uniform rows (every draw is a tie of equal steps); p equal to q
    (everything accepted, the bonus drawn); one-hot target and draft on
    different tokens (every draft rejected, the residual is the target's
    spike); extreme temperatures."""
    zp, zq, x, u, V = _degenerate_case(kind, T=T, seed=len(kind))
    B, K = x.shape
    tok, n = sv.spec_verify_from_logits(zp, zq, x, u, T)
    torch.cuda.synchronize()
    ref = oracle.verify_sampling(np64(zp).reshape(B, K + 1, V), np64(zq).reshape(B, K, V), np_int(x), np64(u), t32(T))
    compare_sampling(np_int(tok), np_int(n), ref, K)
    if kind in ("v1", "uniform", "p_equals_q"):
        assert (np_int(n) == K).all()
    if kind == "spikes":
        spike = np.argmax(np64(zp).reshape(B, K + 1, V)[:, 0], axis=1)
        same = np_int(x)[:, 0] == spike
        assert (np_int(n)[~same] == 0).all() and (np_int(tok)[~same, 0] == spike[~same]).all()


@pytest.mark.parametrize("V", [36000, 100000, 131072, 140000])
@pytest.mark.parametrize("kind", ["spikes", "p_equals_q"])
def test_degenerate_distributions_large_vocabulary(kind, V):
    """The degenerate rows over many 4096-token chunks: each rejected
    sequence draws exactly the target's spike wherever it lies (any chunk of
    any CTA of the row); with p = q every draft passes and the bonus comes
    from p_K."""
    zp, zq, x, u, V = _degenerate_case(kind, B=6, K=3, V=V, T=1.0, seed=V + len(kind))
    B, K = x.shape
    tok, n = sv.spec_verify_from_logits(zp, zq, x, u, 1.0)
    torch.cuda.synchronize()
    ref = oracle.verify_sampling(np64(zp).reshape(B, K + 1, V), np64(zq).reshape(B, K, V), np_int(x), np64(u), t32(1.0))
    compare_sampling(np_int(tok), np_int(n), ref, K)
    if kind == "p_equals_q":
        assert (np_int(n) == K).all()
    else:
        spike = np.argmax(np64(zp).reshape(B, K + 1, V)[:, 0], axis=1)
        same = np_int(x)[:, 0] == spike
        assert (np_int(n)[~same] == 0).all() and (np_int(tok)[~same, 0] == spike[~same]).all()


def test_tiny_logits_workload():
    w = synth.WORKLOADS["tiny_logits"]
    inp = synth.make_inputs(w, device="cuda")
    B, K, V, T = w.B, w.K, w.V, w.temperature
    dbg = torch.zeros((B, K + 1, sv.SPEC_DEBUG_FIELDS), device="cuda")
    tok, n = sv.spec_verify_from_logits(inp["target_logits"], inp["draft_logits"], inp["draft_tokens"],
                                        inp["uniforms"], T, out_debug=dbg)
    torch.cuda.synchronize()
    ref = oracle.verify_sampling(np64(inp["target_logits"]).reshape(B, K + 1, V),
                                 np64(inp["draft_logits"]).reshape(B, K, V), np_int(inp["draft_tokens"]),
                                 np64(inp["uniforms"]), t32(T))
    compare_sampling(np_int(tok), np_int(n), ref, K)
    compare_debug(np64(dbg), ref, np_int(n), K)


def test_many_draws_over_fixed_logits():
    """Thousands of decisions on one set of logits: every accept count and
    token must agree outside the bands, and band cases stay under 0.1%."""
    B, K, V, T = 256, 4, 32000, 0.8
    zp, zq, x, _ = _from_logits_case(B, K, V, T, seed=77, std=1.0, noise=0.3)
    zp64, zq64, x64 = np64(zp).reshape(B, K + 1, V), np64(zq).reshape(B, K, V), np_int(x)
    totals = dict(draws=0, accept_exempt=0, draw_exempt=0, draw_mismatch_exempt=0, accept_mismatch_exempt=0)
    us = synth.fresh_uniforms(B, K, 8, device="cuda", seed=5)
    for i in range(us.shape[0]):
        u = us[i].contiguous()
        tok, n = sv.spec_verify_from_logits(zp, zq, x, u, T)
        torch.cuda.synchronize()
        ref = oracle.verify_sampling(zp64, zq64, x64, np64(u), t32(T))
        st = compare_sampling(np_int(tok), np_int(n), ref, K)
        for k in totals:
            totals[k] += st[k]
    print(f"\nmany draws: {totals}")
    assert totals["accept_exempt"] + totals["draw_exempt"] <= max(1, 0.001 * totals["draws"])


def test_chi_square_exactness_on_gpu():
    """The GPU path's output at every slot follows p (chi-square, alpha 0.001,
    10^6 rounds at V=16, K=4), the same test the oracle is pinned by."""
    from scipy import stats
    V, K = 16, 4
    rng = np.random.default_rng(21)
    p = np.exp(rng.normal(size=(K + 1, V)))
    p /= p.sum(axis=1, keepdims=True)
    q = np.exp(rng.normal(size=(K, V)))
    q /= q.sum(axis=1, keepdims=True)
    B = 100_000
    zp = torch.tensor(np.log(p), dtype=torch.float32, device="cuda").repeat(B, 1).contiguous()
    zq = torch.tensor(np.log(q), dtype=torch.float32, device="cuda").repeat(B, 1).contiguous()
    g = torch.Generator(device="cuda").manual_seed(3)
    counts = [np.zeros(V) for _ in range(K + 1)]
    for it in range(10):
        x = synth.gumbel_max_tokens(zq, 1.0, g).view(B, K).contiguous()
        u = torch.rand((B, K + 1), generator=g, device="cuda")
        tok, n = sv.spec_verify_from_logits(zp, zq, x, u, 1.0)
        tok, n = np_int(tok), np_int(n)
        for j in range(K + 1):
            sel = n >= j
            counts[j] += np.bincount(tok[sel, j], minlength=V)
    for j in range(K + 1):
        exp = counts[j].sum() * p[j]
        s = ((counts[j] - exp) ** 2 / exp).sum()
        assert s <= stats.chi2.ppf(0.999, V - 1), (j, s)


def test_determinism_bits():
    B, K, V, T = 16, 4, 20000, 0.9
    zp, zq, x, u = _from_logits_case(B, K, V, T, seed=9)
    d1 = torch.zeros((B, K + 1, 6), device="cuda")
    d2 = torch.zeros((B, K + 1, 6), device="cuda")
    t1, n1 = sv.spec_verify_from_logits(zp, zq, x, u, T, out_debug=d1)
    t1, n1 = t1.clone(), n1.clone()
    t2, n2 = sv.spec_verify_from_logits(zp, zq, x, u, T, out_debug=d2)
    torch.cuda.synchronize()
    assert torch.equal(t1, t2) and torch.equal(n1, n2) and torch.equal(d1, d2)


# ---------------------------------------------------------------- whole step, small
@pytest.mark.parametrize("B,K,d,V,T", [(3, 3, 256, 5000, 0.8), (1, 5, 512, 32000, 1.0), (5, 0, 128, 1000, 1.0),
                                       (12, 8, 384, 4099, 1.0),
                                       (9, 4, 384, 2000, 0.7),      # M = 45: 48 columns, last chunk partial
                                       (13, 3, 256, 3001, 1.1),     # M = 52: 64 columns
                                       (8, 7, 512, 7000, 0.9),      # M = 64: every column used
                                       (2, 3, 256, 3000, 1e-6),     # |z / T| in log2 units around 2^22
                                       (2, 3, 256, 3000, 1e-8),     # ... and beyond 2^24
                                       (40, 7, 256, 3001, 0.9),     # M = 320: large-batch head, two chunks of 160
                                       (16, 4, 4096, 32000, 0.9),   # M = 80: large-batch head, draft rows by its side warps
                                       (16, 4, 4096, 32003, 1.0),   # ... V % 4 != 0 (scalar draft loads), last pair tile past V
                                       (20, 12, 128, 1500, 1.3),    # M = 260: two chunks of 160, the second of 100 rows
                                       (100, 10, 128, 2000, 1.0),   # M = 1100: 5 chunks of 224
                                       (80, 0, 128, 1000, 1.0)])    # large-batch head, bonus draws only
def test_spec_verify_small(B, K, d, V, T):
    w = synth.custom("small", B=B, K=K, d=d, V=V, temperature=T, seed=B + K + d + V)
    inp, tok, n, logits, dbg = _run_head_case(w)
    ref = oracle.spec_verify(np64(inp["hidden"]), np64(inp["W"]), np64(inp["draft_logits"]),
                             np_int(inp["draft_tokens"]), np64(inp["uniforms"]), t32(T), B, K)
    err = logits_error(np64(logits), ref["target_logits"])
    assert err["max_abs"] <= LOGIT_ATOL, err
    st = compare_sampling(np_int(tok), np_int(n), ref, K)
    compare_debug(np64(dbg), ref, np_int(n), K, T, err["max_abs"])
    print(f"\nspec_verify small {B},{K},{d},{V},{T}: logits {err} {st}")


@pytest.mark.parametrize("B,K,d,V", [(4, 4, 256, 3000), (40, 3, 512, 1001), (100, 4, 128, 20000),
                                     (16, 4, 256, 4097)])   # M = 80: a 16-column tail in the large-batch epilogue
def test_greedy_small(B, K, d, V):
    w = synth.custom("greedy", B=B, K=K, d=d, V=V, temperature=0.0, noise=0.2, seed=B * K + V)
    inp, tok, n, _, dbg = _run_head_case(w)
    ref = oracle.spec_verify(np64(inp["hidden"]), np64(inp["W"]), None, np_int(inp["draft_tokens"]), None, 0.0, B, K)
    z = sv.spec_lm_head(inp["hidden"], inp["W"])
    torch.cuda.synchronize()
    err = logits_error(np64(z), ref["target_logits"])
    st = compare_greedy(np_int(tok), np_int(n), ref, err["max_abs"])
    assert st["mismatched_near_ties"] == 0, st
    # greedy from the same GPU logits through the other entry point is identical
    tok2, n2 = sv.spec_verify_from_logits(z, None, inp["draft_tokens"], None, 0.0)
    torch.cuda.synchronize()
    assert torch.equal(tok, tok2) and torch.equal(n, n2)
    # debug: the row max equals the max of the GPU logits; argmax ids match the oracle
    dbg = np64(dbg)
    np.testing.assert_array_equal(dbg[:, :, 0].reshape(-1), np64(z).max(axis=1))
    np.testing.assert_array_equal(dbg[:, :, 1].astype(np.int64), ref["argmax"])


# ---------------------------------------------------------------- edge cases
def test_invalid_draft_token_marks_the_sequence():
    B, K, V, T = 4, 3, 1000, 1.0
    zp, zq, x, u = _from_logits_case(B, K, V, T, seed=11)
    x[2, 1] = V + 5
    ws = torch.empty(sv.workspace_bytes(B, K, V, T, False), dtype=torch.uint8, device="cuda")
    tok, n = sv.spec_verify_from_logits(zp, zq, x, u, T, workspace=ws)
    word = sv.read_error(ws)
    assert word & sv.DEVERR_TOKEN_RANGE
    n = np_int(n)
    tok = np_int(tok)
    assert n[2] == -1 and (tok[2] == -1).all()
    ref = oracle.verify_sampling(np64(zp).reshape(B, K + 1, V), np64(zq).reshape(B, K, V),
                                 np.clip(np_int(x), 0, V - 1), np64(u), t32(T))
    keep = [0, 1, 3]
    sub = {k: v[keep] for k, v in ref.items()}
    compare_sampling(tok[keep], n[keep], sub, K)


@pytest.mark.parametrize("M_seq", [1, 16])                 # small-batch and large-batch LM-head schemes
@pytest.mark.parametrize("lo,hi", [(31, 32), (95, 96), (127, 128), (5, 900), (0, 999)])
def test_greedy_exact_ties_pick_the_lowest_id(M_seq, lo, hi):
    """Two identical weight rows that dominate every position's logits give
    exact ties (same bf16 operands, same accumulation order) across a warp
    boundary (31/32), a lane-quadrant boundary (95/96), a vocabulary-tile
    boundary (127/128) and far apart; the greedy target token is the lower
    id, as in the oracle, and drafts equal to it are all accepted."""
    B, K, d, V = M_seq, 4, 128, 1000
    g = torch.Generator(device="cuda").manual_seed(lo * 1000 + hi)
    base = torch.randn(d, generator=g, device="cuda")
    hidden = (base + 0.05 * torch.randn((B * (K + 1), d), generator=g, device="cuda")).to(torch.bfloat16)
    W = 0.01 * torch.randn((V, d), generator=g, device="cuda")
    W[lo] = 3.0 * base / base.norm()
    W[hi] = W[lo]
    W = W.to(torch.bfloat16)
    x = torch.full((B, K), lo, dtype=torch.int32, device="cuda")
    tok, n = sv.spec_verify(hidden, W, None, x, None, 0.0)
    torch.cuda.synchronize()
    ref = oracle.spec_verify(np64(hidden), np64(W), None, np_int(x), None, 0.0, B, K)
    assert (ref["argmax"] == lo).all()
    np.testing.assert_array_equal(np_int(tok), ref["tokens"])
    np.testing.assert_array_equal(np_int(n), ref["num_accepted"])
    assert (np_int(n) == K).all()


def test_nonfinite_logit_marks_the_sequence():
    B, K, V, T = 3, 2, 5000, 1.0
    zp, zq, x, u = _from_logits_case(B, K, V, T, seed=12)
    zp[1 * (K + 1) + 2, 17] = float("nan")
    ws = torch.empty(sv.workspace_bytes(B, K, V, T, False), dtype=torch.uint8, device="cuda")
    tok, n = sv.spec_verify_from_logits(zp, zq, x, u, T, workspace=ws)
    assert sv.read_error(ws) & sv.DEVERR_NONFINITE
    assert np_int(n)[1] == -1 and np_int(n)[0] >= 0 and np_int(n)[2] >= 0
    zp2 = zp.clone()
    zp2[1 * (K + 1) + 2, 17] = float("inf")
    t3, n3 = sv.spec_verify_from_logits(zp2, zq, x, u, 0.0, workspace=torch.empty(
        sv.workspace_bytes(B, K, V, 0.0), dtype=torch.uint8, device="cuda"))
    assert np_int(n3)[1] == -1


@pytest.mark.parametrize("B,K", [(3, 2), (24, 4)])   # the small-batch and the large-batch LM head
def test_nonfinite_hidden_marks_the_sequence(B, K):
    """A NaN or infinite hidden state makes its position's logits non-finite
    (in either head's fused statistics): that sequence is flagged, the others
    are unaffected."""
    w = synth.custom("nf_head", B=B, K=K, d=256, V=3000, temperature=1.0, seed=21 + B)
    inp = synth.make_inputs(w, device="cuda")
    B, K, V, T = w.B, w.K, w.V, w.temperature
    ref = oracle.spec_verify(np64(inp["hidden"]), np64(inp["W"]), np64(inp["draft_logits"]),
                             np_int(inp["draft_tokens"]), np64(inp["uniforms"]), t32(T), B, K)
    for bad in (float("nan"), float("inf"), float("-inf")):
        h = inp["hidden"].clone()
        h[1 * (K + 1) + 2, 5] = bad
        ws = torch.empty(sv.workspace_bytes(B, K, V, T), dtype=torch.uint8, device="cuda")
        tok, n = sv.spec_verify(h, inp["W"], inp["draft_logits"], inp["draft_tokens"], inp["uniforms"], T,
                                workspace=ws)
        assert sv.read_error(ws) & sv.DEVERR_NONFINITE, bad
        n, tok = np_int(n), np_int(tok)
        assert n[1] == -1 and (tok[1] == -1).all(), bad
        keep = [b for b in range(B) if b != 1]
        compare_sampling(tok[keep], n[keep], {k: v[keep] for k, v in ref.items() if k != "target_logits"}, K)


@pytest.mark.parametrize("B,K,d,V", [(3, 2, 256, 3000),      # small-batch head: its side warps
                                     (16, 4, 4096, 32000),  # large-batch head: its side warps
                                     (24, 4, 256, 3000)])   # large-batch head, then the draft-row pass
def test_nonfinite_draft_logit_in_the_whole_step(B, K, d, V):
    """A NaN, +inf or -inf draft logit, wherever the draft rows are reduced
    in the whole step, flags its sequence; the others are unaffected."""
    w = synth.custom("nf_draft", B=B, K=K, d=d, V=V, temperature=1.0, seed=31 + B)
    inp = synth.make_inputs(w, device="cuda")
    ref = oracle.spec_verify(np64(inp["hidden"]), np64(inp["W"]), np64(inp["draft_logits"]),
                             np_int(inp["draft_tokens"]), np64(inp["uniforms"]), t32(w.temperature), B, K)
    for bad in (float("nan"), float("inf"), float("-inf")):
        zq = inp["draft_logits"].clone()
        zq[1 * K + 1, V - 7] = bad   # sequence 1, draft row 1, in the last chunk
        ws = torch.empty(sv.workspace_bytes(B, K, V, w.temperature), dtype=torch.uint8, device="cuda")
        tok, n = sv.spec_verify(inp["hidden"], inp["W"], zq, inp["draft_tokens"], inp["uniforms"], w.temperature,
                                workspace=ws)
        assert sv.read_error(ws) & sv.DEVERR_NONFINITE, bad
        n, tok = np_int(n), np_int(tok)
        assert n[1] == -1 and (tok[1] == -1).all(), bad
        keep = [b for b in range(B) if b != 1]
        compare_sampling(tok[keep], n[keep], {k: v[keep] for k, v in ref.items() if k != "target_logits"}, K)


def test_all_accept_and_first_reject_extremes():
    """u = 0 accepts every draft with p(x) > 0 (then the bonus row is drawn);
    u just below 1 rejects every draft whose a < 1."""
    B, K, V, T = 32, 4, 3000, 1.0
    zp, zq, x, u = _from_logits_case(B, K, V, T, seed=13)
    for fill in (0.0, 0.99999994):
        u2 = torch.full_like(u, fill)
        u2[:, K] = u[:, K]
        tok, n = sv.spec_verify_from_logits(zp, zq, x, u2, T)
        torch.cuda.synchronize()
        ref = oracle.verify_sampling(np64(zp).reshape(B, K + 1, V), np64(zq).reshape(B, K, V), np_int(x),
                                     np64(u2), t32(T))
        compare_sampling(np_int(tok), np_int(n), ref, K)
        if fill == 0.0:
            assert (np_int(n) == K).all()


def test_host_buffer_entry_point_matches_device_entry_point():
    w = synth.custom("host", B=4, K=4, d=512, V=9000, temperature=0.8, seed=4)
    inp = synth.make_inputs(w, device="cuda")
    tok, n = sv.spec_verify(inp["hidden"], inp["W"], inp["draft_logits"], inp["draft_tokens"], inp["uniforms"], 0.8)
    host = {k: v.cpu().pin_memory() for k, v in inp.items() if isinstance(v, torch.Tensor) and k != "W"}
    tok_h, n_h = sv.spec_verify_host(host["hidden"], inp["W"], host["draft_logits"], host["draft_tokens"],
                                     host["uniforms"], 0.8)
    assert torch.equal(tok.cpu(), tok_h) and torch.equal(n.cpu(), n_h)


def test_host_async_steps_in_flight_on_two_streams():
    """spec_verify_host_async: several steps in flight on two streams, each
    with its own workspace and pinned buffers, give the device entry point's
    results step by step."""
    w = synth.custom("host_async", B=6, K=3, d=512, V=7001, temperature=0.9, seed=8)
    inp = synth.make_inputs(w, device="cuda")
    us = synth.fresh_uniforms(w.B, w.K, 6, device="cuda", seed=5)
    ref = []
    for i in range(6):
        t, n = sv.spec_verify(inp["hidden"], inp["W"], inp["draft_logits"], inp["draft_tokens"], us[i], 0.9)
        ref.append((t.cpu(), n.cpu()))
    host = {k: v.cpu().pin_memory() for k, v in inp.items() if isinstance(v, torch.Tensor) and k != "W"}
    slots = [dict(stream=torch.cuda.Stream(), ws=torch.empty(sv.host_workspace_bytes(w.B, w.K, w.d, w.V, 0.9),
                                                             dtype=torch.uint8, device="cuda"))
             for _ in range(2)]
    outs = []
    for i in range(6):
        sl = slots[i % 2]
        u = us[i].cpu().pin_memory()
        ot = torch.empty((w.B, w.K + 1), dtype=torch.int32).pin_memory()
        on = torch.empty((w.B,), dtype=torch.int32).pin_memory()
        sv.spec_verify_host(host["hidden"], inp["W"], host["draft_logits"], host["draft_tokens"], u, 0.9,
                            workspace=sl["ws"], out_tokens=ot, out_num_accepted=on, stream=sl["stream"], wait=False)
        outs.append((ot, on, u))
    torch.cuda.synchronize()
    for (ot, on, _), (rt, rn) in zip(outs, ref):
        assert torch.equal(ot, rt) and torch.equal(on, rn)


# ---------------------------------------------------------------- full-size workloads
@pytest.mark.parametrize("name", ["head_B1_K5_V32000", "head_B8_K4_V128256"])
def test_full_size_sampling_workload(name):
    w = synth.WORKLOADS[name]
    inp, tok, n, logits, dbg = _run_head_case(w)
    ref = oracle.spec_verify(np64(inp["hidden"]), np64(inp["W"]), np64(inp["draft_logits"]),
                             np_int(inp["draft_tokens"]), np64(inp["uniforms"]), t32(w.temperature), w.B, w.K)
    err = logits_error(np64(logits), ref["target_logits"])
    st = compare_sampling(np_int(tok), np_int(n), ref, w.K)
    print(f"\n{name}: logits {err}; decisions {st}; accepted {np_int(n).tolist()}")
    assert err["max_abs"] <= LOGIT_ATOL, err
    compare_debug(np64(dbg), ref, np_int(n), w.K, w.temperature, err["max_abs"])


def _draws_moved_by_logit_error(z32, z64, T, seed, per_row=256):
    """Fraction of inverse-CDF draws (fp64 arithmetic on both sides, fresh
    uniforms per row) whose token changes when the fp64 logits are replaced
    by the LM head's, outside the draw band."""
    rng = np.random.default_rng(seed)
    moved = draws = 0
    for r in range(z64.shape[0]):
        def cdf(z):
            p = np.exp((z - z.max()) / T)
            c = np.cumsum(p)
            return c / c[-1], p / c[-1]
        c64, p64 = cdf(z64[r])
        c32, _ = cdf(z32[r])
        u = rng.random(per_row)
        y64 = np.minimum(np.searchsorted(c64, u, side="right"), len(c64) - 1)
        y32 = np.minimum(np.searchsorted(c32, u, side="right"), len(c32) - 1)
        lo = u - np.where(y64 > 0, c64[np.maximum(y64 - 1, 0)], 0.0)
        hi = c64[y64] - u
        near = np.minimum(lo, hi) < DRAW_BAND * p64[y64]
        moved += int(((y64 != y32) & ~near).sum())
        draws += len(u)
    return moved / draws, draws


def test_head_precision_keeps_draws_headline():
    """The precise LM head's own logit error moves under 0.1 % of inverse-CDF
    draws against the fp64 logits (40 rows of the headline workload)."""
    w = synth.WORKLOADS["head_B8_K4_V128256"]
    inp = synth.make_inputs(w, device="cuda")
    z32 = np64(sv.spec_lm_head(inp["hidden"], inp["W"]))
    z64 = oracle.lm_head(np64(inp["hidden"]), inp["W"].float().cpu().numpy())
    rate, draws = _draws_moved_by_logit_error(z32, z64, t32(w.temperature), seed=5)
    print(f"\nheadline: {rate * 100:.3f} % of {draws} draws moved by the LM head's error")
    assert rate < 1e-3


def test_head_precision_keeps_draws_large_batch():
    """The same measure on 48 rows of the B=64, d=8192 workload, whose LM head
    (576 positions) runs the large-batch kernel's 2048-product groups (an
    accumulator over the whole hidden size moved ~0.24 % of these draws)."""
    w = synth.WORKLOADS["head_B64_K8_V152064"]
    inp = synth.make_inputs(w, device="cuda")
    rows = 48
    z32 = np64(sv.spec_lm_head(inp["hidden"], inp["W"])[:rows])
    z64 = oracle.lm_head(np64(inp["hidden"][:rows]), inp["W"].float().cpu().numpy())
    rate, draws = _draws_moved_by_logit_error(z32, z64, t32(w.temperature), seed=6)
    print(f"\nB64: {rate * 100:.3f} % of {draws} draws moved by the LM head's error")
    assert rate < 1e-3


@pytest.mark.parametrize("B,K,d,V,T", [(1, 4, 4096, 1000, 1.0),     # 8 tiles x 16 groups: 16-way splits
                                       (2, 3, 1024, 5000, 0.9),     # 40 tiles x 4 groups on 152 CTAs
                                       (8, 4, 4096, 20000, 0.8),    # 157 tiles x 16 groups: 2-way splits
                                       (3, 3, 4096, 2000, 0.0)])    # greedy, 16 tiles x 16 groups
def test_streamk_split_tiles(B, K, d, V, T):
    """The precise LM head spreads (tile, group) units evenly over the CTAs; a
    tile split across CTAs is finished by the CTA holding its first group with
    the others' sums from the fixup area.  Logits and results against the
    oracle as everywhere; the logits also agree with the whole-tile schedule
    of the bare LM head to rounding."""
    w = synth.custom("streamk", B=B, K=K, d=d, V=V, temperature=T, noise=0.3, seed=B * 100 + d + V)
    inp, tok, n, logits, dbg = _run_head_case(w)
    z_tile = sv.spec_lm_head(inp["hidden"], inp["W"])
    torch.cuda.synchronize()
    dl = np64(inp["draft_logits"]) if T > 0 else None
    u = np64(inp["uniforms"]) if T > 0 else None
    ref = oracle.spec_verify(np64(inp["hidden"]), np64(inp["W"]), dl, np_int(inp["draft_tokens"]), u, t32(T), B, K)
    if T > 0:
        err = logits_error(np64(logits), ref["target_logits"])
        assert err["max_abs"] <= LOGIT_ATOL and err["rms"] < 1e-5, err
        assert np.abs(np64(logits) - np64(z_tile)).max() < 1e-4
        compare_sampling(np_int(tok), np_int(n), ref, K)
    else:
        err = logits_error(np64(z_tile), ref["target_logits"])
        st = compare_greedy(np_int(tok), np_int(n), ref, err["max_abs"])
        assert st["mismatched_near_ties"] == 0, st
