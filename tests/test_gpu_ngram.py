"""Prompt-lookup drafter on the GPU against the oracle
(oracle/ngram_drafter.py): drafts and counts bit-exact."""
import numpy as np
import pytest
import torch

import speculative_decoding_verification_67_gb300 as sv
from oracle import ngram_drafter as ng
from speculative_decoding_verification_67_gb300 import synth

from _helpers import compare_greedy

pytestmark = pytest.mark.gpu


def check(hist, lens, K, n_min, n_max):
    h = torch.as_tensor(np.asarray(hist), dtype=torch.int32).cuda().contiguous()
    L = torch.as_tensor(np.asarray(lens), dtype=torch.int32).cuda()
    ws = sv.ngram_workspace(h.shape[0], h.shape[1], K, n_min, n_max)
    d, c = sv.spec_ngram_propose(h, L, K, n_min, n_max, workspace=ws)
    err = sv.ngram_read_error(ws)
    rd, rc = ng.propose_batch(np.asarray(hist), np.asarray(lens), K, n_min, n_max)
    assert err == 0
    assert np.array_equal(c.cpu().numpy(), rc)
    assert np.array_equal(d.cpu().numpy(), rd)
    return ws


@pytest.mark.parametrize("V", [2, 5, 50, 128256])
@pytest.mark.parametrize("n_min,n_max", [(1, 1), (1, 3), (2, 4), (3, 16)])
def test_random_histories(V, n_min, n_max):
    rng = np.random.default_rng(V * 100 + n_max)
    B, max_len = 37, 20000                      # several chunks of candidate positions per row
    hist = rng.integers(0, V, size=(B, max_len))
    lens = rng.integers(0, max_len + 1, size=B)
    lens[:6] = [0, 1, 2, 3, max_len, max_len - 1]
    for K in (1, 4, 32):
        check(hist, lens, K, n_min, n_max)


def test_matches_across_chunk_boundaries():
    """The only occurrence of the key ends exactly at, or straddles, a chunk
    boundary (chunks of 1024 candidate positions at this batch and length:
    8192 and 16384 are boundaries), so a match reaches into the tokens staged
    before the chunk."""
    B, max_len = 6, 3 * 8192 + 100
    hist = np.arange(B * max_len).reshape(B, max_len) % 1000003 + 10        # no repeats
    lens = np.full(B, max_len)
    key = [1, 2, 3]
    for b, e in enumerate([8191, 8192, 8193, 16383, 16384, 0]):
        L = lens[b]
        hist[b, L - 3:L] = key
        start = e - 2
        if start >= 0:
            hist[b, start:e + 1] = key
        else:
            hist[b, 0] = key[2]                  # a 1-gram occurrence at 0
    check(hist, lens, 8, 1, 3)


def test_periodic_and_copying_histories():
    B, max_len = 4, 5000
    hist = np.zeros((B, max_len), dtype=np.int64)
    hist[0] = np.tile([7, 8, 9], max_len // 3 + 1)[:max_len]
    hist[1] = np.arange(max_len) % 17
    prompt = np.random.default_rng(3).integers(0, 1000, size=2500)
    hist[2, :2500] = prompt
    hist[2, 2500:] = prompt
    hist[3] = 42
    lens = np.array([max_len, 4321, 3100, 999])
    check(hist, lens, 8, 1, 3)


def test_invalid_lengths_and_reuse():
    rng = np.random.default_rng(9)
    B, max_len, K = 5, 300, 4                    # max_len a multiple of 4
    hist = rng.integers(0, 4, size=(B, max_len))
    h = torch.as_tensor(hist, dtype=torch.int32).cuda()
    L = torch.tensor([10, -1, max_len + 1, 0, 300], dtype=torch.int32).cuda()
    ws = sv.ngram_workspace(B, max_len, K)
    d, c = sv.spec_ngram_propose(h, L, K, workspace=ws)
    assert sv.ngram_read_error(ws) == sv.NGRAM_DEVERR_LENGTH
    c = c.cpu().numpy()
    d = d.cpu().numpy()
    assert c[1] == -1 and c[2] == -1 and (d[1] == -1).all() and (d[2] == -1).all()
    for b in (0, 3, 4):
        rd, rc = ng.propose(hist[b, : int(L[b])], K, 1, 3)
        assert c[b] == rc and np.array_equal(d[b], rd)
    # the same workspace again, valid lengths: slots and tickets were reset
    L2 = torch.tensor([10, 20, 30, 0, 300], dtype=torch.int32).cuda()
    d, c = sv.spec_ngram_propose(h, L2, K, workspace=ws)
    assert sv.ngram_read_error(ws) == 0
    rd, rc = ng.propose_batch(hist, L2.cpu().numpy(), K, 1, 3)
    assert np.array_equal(c.cpu().numpy(), rc) and np.array_equal(d.cpu().numpy(), rd)


@pytest.mark.parametrize("name", sorted(synth.NGRAM_WORKLOADS))
def test_full_size_workloads(name):
    w = synth.NGRAM_WORKLOADS[name]
    inp = synth.make_ngram_inputs(w)
    check(inp["history"].numpy(), inp["lengths"].numpy(), w.K, w.n_min, w.n_max)


def test_drafts_feed_greedy_verify():
    """Drafts go straight into the greedy verify step (drafter -> verify):
    the verify result equals the oracle's greedy verify of the same drafts."""
    from oracle import spec_oracle
    rng = np.random.default_rng(4)
    B, K, d_model, V = 6, 4, 256, 3000
    hist = rng.integers(0, V, size=(B, 400))
    hist[:, 200:] = hist[:, :200]                      # outputs copying their prompts
    lens = np.array([400, 350, 260, 300, 399, 211])
    h = torch.as_tensor(hist, dtype=torch.int32).cuda()
    L = torch.as_tensor(lens, dtype=torch.int32).cuda()
    drafts, count = sv.spec_ngram_propose(h, L, K)
    w = synth.custom("ngram_verify", B=B, K=K, d=d_model, V=V, temperature=0.0, seed=5)
    inp = synth.make_inputs(w, device="cuda")
    tok, n = sv.spec_verify(inp["hidden"], inp["W"], None, drafts, None, 0.0)
    ref = spec_oracle.spec_verify(inp["hidden"].double().cpu().numpy(), inp["W"].double().cpu().numpy(), None,
                                  drafts.cpu().numpy(), None, 0.0, B, K)
    logits = sv.spec_lm_head(inp["hidden"], inp["W"])
    err = float(np.abs(logits.double().cpu().numpy() - ref["target_logits"]).max())
    compare_greedy(tok.cpu().numpy(), n.cpu().numpy(), ref, err)
