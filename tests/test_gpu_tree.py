"""Tree-shaped candidate verification on the GPU against the oracle
(oracle/tree_verify.py)."""
import numpy as np
import pytest
import torch

import speculative_decoding_verification_67_gb300 as sv
from oracle import spec_oracle
from oracle import tree_verify as tv
from speculative_decoding_verification_67_gb300 import synth

from _helpers import ACCEPT_BAND, DRAW_BAND, LOGIT_ATOL, t32

pytestmark = pytest.mark.gpu


def compare_tree(tok, path, n, ref, greedy=False, logit_err=0.0):
    """Identical results, except where the oracle's walk made a decision
    within the band (an accept test with |u - a| < ACCEPT_BAND, a draw within
    DRAW_BAND of its CDF step, a greedy row whose top-2 gap is within twice
    the logit error); returns the number of such exempt sequences."""
    tok, path, n = np.asarray(tok), np.asarray(path), np.asarray(n)
    exempt = 0
    for b in range(len(n)):
        info = ref["info"][b]
        if info is None:
            assert n[b] == -1 and (tok[b] == -1).all() and (path[b] == -1).all(), b
            continue
        same = (n[b] == ref["num_accepted"][b] and np.array_equal(tok[b], ref["tokens"][b])
                and np.array_equal(path[b], ref["path"][b]))
        if greedy:
            near = any(g <= 2 * logit_err + 1e-12 for g in info["top2_gap"])
            assert same or near, (b, tok[b], ref["tokens"][b], info["top2_gap"])
            exempt += int(not same)
            continue
        near_acc = any(m < ACCEPT_BAND for m in info["accept"])
        near_draw = min(info["draw_lo"], info["draw_hi"]) < DRAW_BAND * info["draw_mass"]
        if not same:
            path_same = n[b] == ref["num_accepted"][b] and np.array_equal(path[b], ref["path"][b])
            assert (near_draw if path_same else near_acc), (b, tok[b], ref["tokens"][b], path[b], ref["path"][b],
                                                            info)
            exempt += 1
    return exempt


def random_tree(rng, B, N, V, T, noise=0.5, scale=2.0, structured=None):
    """Random parents (or a given parent list), target rows ~ N(0, scale),
    draft rows = target rows + noise, children drawn i.i.d. from their
    parent's draft row."""
    if structured is None:
        par = np.empty((B, N), dtype=np.int64)
        par[:, 0] = -1
        for i in range(1, N):
            par[:, i] = rng.integers(0, i, size=B)
    else:
        par = np.tile(np.asarray(structured), (B, 1))
    zp = rng.normal(0, scale, size=(B, N, V)).astype(np.float32)
    zq = (zp + rng.normal(0, noise, size=(B, N, V))).astype(np.float32)
    tok = np.zeros((B, N), dtype=np.int64)
    Tq = T if T > 0 else 1.0
    for b in range(B):
        for i in range(1, N):
            row = zq[b, par[b, i]].astype(np.float64) / Tq
            gum = -np.log(-np.log(rng.random(V).clip(1e-300)))
            tok[b, i] = int(np.argmax(row + gum))
    u = rng.random((B, N)).astype(np.float32)
    return zp, zq, tok, par, u


def gpu_tree(zp, zq, tok, par, u, T):
    B, N, V = zp.shape
    f = lambda x, dt: torch.as_tensor(np.ascontiguousarray(x), dtype=dt).cuda()
    return sv.spec_tree_verify_from_logits(f(zp.reshape(B * N, V), torch.float32),
                                           f(zq.reshape(B * N, V), torch.float32) if T > 0 else None,
                                           f(tok, torch.int32), f(par, torch.int32),
                                           f(u, torch.float32) if T > 0 else None, T)


def np_(t):
    return t.cpu().numpy()


@pytest.mark.parametrize("N", [1, 2, 9, 33, 256])
@pytest.mark.parametrize("V,T", [(7, 1.0), (1000, 0.6), (5003, 1.5), (32000, 1.0)])
def test_sampling_random_trees(N, V, T):
    rng = np.random.default_rng(N * 1000 + V)
    B = 6 if N < 256 else 2
    zp, zq, tok, par, u = random_tree(rng, B, N, V, T)
    t, p, n = gpu_tree(zp, zq, tok, par, u, T)
    ref = tv.verify_tree(zp, zq, tok, par, u, t32(T))
    compare_tree(np_(t), np_(p), np_(n), ref)


@pytest.mark.parametrize("B,N,V,T", [(12, 9, 32000, 1.0),   # more than 9 trees: 8-CTA clusters
                                     (12, 33, 1000, 0.7),
                                     (9, 17, 131072, 0.9),  # 9 trees of 16 CTAs, slices of 8192
                                     (3, 5, 196608, 1.0)])  # the largest vocabulary, slices of 12288
def test_sampling_random_trees_cluster_sizes(B, N, V, T):
    """A walk runs on 16-CTA clusters while B*16 CTAs fit the SMs and on
    8-CTA clusters otherwise; both against the oracle, at slice sizes up to
    the largest vocabulary."""
    rng = np.random.default_rng(B * 7919 + N * 31 + V)
    zp, zq, tok, par, u = random_tree(rng, B, N, V, T)
    t, p, n = gpu_tree(zp, zq, tok, par, u, T)
    ref = tv.verify_tree(zp, zq, tok, par, u, t32(T))
    compare_tree(np_(t), np_(p), np_(n), ref)


@pytest.mark.parametrize("ctas", ["8", "12", "16"])
@pytest.mark.parametrize("B,N,V,T", [(5, 9, 32000, 1.0), (3, 33, 128256, 0.8), (2, 5, 196608, 1.0), (4, 9, 7, 1.0)])
def test_sampling_every_cluster_size(ctas, B, N, V, T, monkeypatch):
    """Each cluster size of the walk (forced where it fits) against the
    oracle: slices of 4 to 24576 tokens, empty slices at V = 7."""
    monkeypatch.setenv("SPEC_TREE_CLUSTER_CTAS", ctas)
    rng = np.random.default_rng(B * 104729 + N * 13 + V)
    zp, zq, tok, par, u = random_tree(rng, B, N, V, T)
    t, p, n = gpu_tree(zp, zq, tok, par, u, T)
    ref = tv.verify_tree(zp, zq, tok, par, u, t32(T))
    compare_tree(np_(t), np_(p), np_(n), ref)


def test_sampling_deep_and_wide_trees():
    """A chain of depth 40 (high acceptance) and a star of 60 children."""
    rng = np.random.default_rng(17)
    for par_list, noise in ((list(range(-1, 40)), 0.05), ([-1] + [0] * 60, 1.5)):
        N = len(par_list)
        zp, zq, tok, par, u = random_tree(rng, 4, N, 3000, 1.0, noise=noise, structured=par_list)
        t, p, n = gpu_tree(zp, zq, tok, par, u, 1.0)
        ref = tv.verify_tree(zp, zq, tok, par, u, 1.0)
        compare_tree(np_(t), np_(p), np_(n), ref)


def test_chain_tree_equals_the_chain_verify_step():
    """A chain tree on the GPU gives the chain verify step's result (both GPU
    paths), uniforms mapped as in the oracle's chain pin."""
    rng = np.random.default_rng(23)
    B, K, V, T = 16, 6, 4099, 0.8
    N = K + 1
    zp, zq, tok, par, u = random_tree(rng, B, N, V, T, noise=0.3, structured=list(range(-1, K)))
    t, p, n = gpu_tree(zp, zq, tok, par, u, T)
    uc = np.concatenate([u[:, 1:], u[:, :1]], axis=1)
    f = lambda x, dt: torch.as_tensor(np.ascontiguousarray(x), dtype=dt).cuda()
    tc, nc = sv.spec_verify_from_logits(f(zp.reshape(B * N, V), torch.float32),
                                        f(zq[:, :K].reshape(B * K, V), torch.float32), f(tok[:, 1:], torch.int32),
                                        f(uc, torch.float32), T)
    ref = tv.verify_tree(zp, zq, tok, par, u, t32(T))
    ex = compare_tree(np_(t), np_(p), np_(n), ref)
    if ex == 0:
        assert np.array_equal(np_(n), np_(nc)) and np.array_equal(np_(t), np_(tc))


def test_greedy_random_trees():
    rng = np.random.default_rng(5)
    B, N, V = 8, 20, 3000
    zp, zq, tok, par, _ = random_tree(rng, B, N, V, 0.0)
    # make some children carry the argmax so that the walk goes deep
    for b in range(B):
        cur = 0
        for i in range(1, N):
            if par[b, i] == cur and rng.random() < 0.7:
                tok[b, i] = int(np.argmax(zp[b, cur]))
                cur = i
    t, p, n = gpu_tree(zp, None, tok, par, None, 0.0)
    ref = tv.verify_tree(zp, None, tok, par, None, 0.0)
    compare_tree(np_(t), np_(p), np_(n), ref, greedy=True)
    assert (np_(n) > 0).any()


def test_invalid_trees():
    rng = np.random.default_rng(2)
    B, N, V, T = 5, 6, 500, 1.0
    zp, zq, tok, par, u = random_tree(rng, B, N, V, T)
    par[1, 3] = 3                         # a node that is its own parent
    par[2, 0] = 0                         # a root with a parent
    tok[3, 4] = V + 2                     # a token outside the vocabulary
    zp[4, 0, 17] = np.inf                 # a non-finite logit in the root row (always visited)
    t, p, n = gpu_tree(zp, zq, tok, par, u, T)
    assert np_(n).tolist()[1:] == [-1, -1, -1, -1] and np_(n)[0] >= 0
    assert (np_(t)[1:] == -1).all() and (np_(p)[1:] == -1).all()
    for T2 in (0.0,):
        t, p, n = gpu_tree(zp, None, tok, par, None, T2)
        assert np_(n).tolist()[1:4] == [-1, -1, -1]


@pytest.mark.parametrize("name", sorted(synth.TREE_WORKLOADS))
def test_full_size_from_hidden(name):
    """The LM head over every node, then the walk; logits and walk against
    the oracle (fp64 LM head over all B*N rows)."""
    w = synth.TREE_WORKLOADS[name]
    inp = synth.make_tree_inputs(w, device="cuda")
    B, N, V, T = w.B, w.N, w.V, w.temperature
    logits = torch.empty((B * N, V), dtype=torch.float32, device="cuda")
    t, p, n = sv.spec_tree_verify(inp["hidden"], inp["W"], inp["draft_logits"], inp["tokens"], inp["parents"],
                                  inp["uniforms"], T, out_target_logits=logits)
    torch.cuda.synchronize()
    zp = spec_oracle.lm_head(inp["hidden"].double().cpu().numpy(), inp["W"].double().cpu().numpy())
    assert np.abs(logits.double().cpu().numpy() - zp).max() <= LOGIT_ATOL
    ref = tv.verify_tree(zp.reshape(B, N, V), inp["draft_logits"].double().cpu().numpy().reshape(B, N, V),
                         np_(inp["tokens"]), np_(inp["parents"]), inp["uniforms"].double().cpu().numpy(), t32(T))
    compare_tree(np_(t), np_(p), np_(n), ref)
    # greedy on the same tree (drafts = argmax of the draft rows)
    ing = synth.make_tree_inputs(w, device="cuda", greedy_drafts=True)
    t, p, n = sv.spec_tree_verify(ing["hidden"], ing["W"], None, ing["tokens"], ing["parents"], None, 0.0)
    zg = sv.spec_lm_head(ing["hidden"], ing["W"])
    zo = spec_oracle.lm_head(ing["hidden"].double().cpu().numpy(), ing["W"].double().cpu().numpy())
    err = float(np.abs(zg.double().cpu().numpy() - zo).max())
    ref = tv.verify_tree(zo.reshape(B, N, V), None, np_(ing["tokens"]), np_(ing["parents"]), None, 0.0)
    compare_tree(np_(t), np_(p), np_(n), ref, greedy=True, logit_err=err)
