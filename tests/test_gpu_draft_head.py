"""Draft steps through the target's LM head (spec_draft_step) on the GPU
against the oracle (oracle/draft_head.py), alone and as the drafter of a
full round that the verify step then checks."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_67_gb300 as sv
from oracle import draft_head
from speculative_decoding_verification_67_gb300 import synth

from _helpers import DRAW_BAND, LOGIT_ATOL, compare_sampling, t32

pytestmark = pytest.mark.gpu


def check_step(tok_gpu, ref, logit_err=0.0):
    """Tokens identical except draws within DRAW_BAND of a CDF-step boundary
    (relative to the step's width); returns the number of exempt draws."""
    tok_gpu = np.asarray(tok_gpu)
    exempt = 0
    for b in range(len(tok_gpu)):
        margin = min(ref["draw_lo"][b], ref["draw_hi"][b])
        near = margin < DRAW_BAND * ref["draw_mass"][b]
        exempt += int(near)
        if tok_gpu[b] != ref["tokens"][b]:
            assert near, (b, tok_gpu[b], ref["tokens"][b], margin, ref["draw_mass"][b])
    return exempt


def np64(t):
    return t.double().cpu().numpy()


@pytest.mark.parametrize("B,d,V,T", [(4, 512, 5000, 0.8), (1, 256, 1000, 1.0), (33, 512, 4099, 1.3),
                                     (64, 256, 32000, 0.6), (130, 256, 3001, 0.9)])
def test_single_step_contiguous_logits(B, d, V, T):
    w = synth.custom("draft_case", B=B, K=1, d=d, V=V, temperature=T, seed=B + V)
    inp = synth.make_draft_inputs(w, device="cuda")
    h = inp["draft_hidden"][0]
    u = inp["draft_uniforms"][0]
    logits = torch.empty((B, V), dtype=torch.float32, device="cuda")
    tok, _ = sv.spec_draft_step(h, inp["W"], u, T, out_logits=logits)
    torch.cuda.synchronize()
    ref = draft_head.draft_step(np64(h), np64(inp["W"]), np64(u), t32(T))
    assert np.abs(np64(logits) - ref["logits"]).max() <= LOGIT_ATOL
    check_step(tok.cpu().numpy(), ref)


def test_logits_kept_in_the_workspace():
    w = synth.custom("draft_ws", B=6, K=1, d=512, V=7000, temperature=0.7, seed=3)
    inp = synth.make_draft_inputs(w, device="cuda")
    tok, none = sv.spec_draft_step(inp["draft_hidden"][0], inp["W"], inp["draft_uniforms"][0], 0.7)
    assert none is None
    ref = draft_head.draft_step(np64(inp["draft_hidden"][0]), np64(inp["W"]), np64(inp["draft_uniforms"][0]),
                                t32(0.7))
    check_step(tok.cpu().numpy(), ref)


def test_greedy_step():
    w = synth.custom("draft_greedy", B=40, K=1, d=512, V=9000, temperature=0.0, seed=8)
    inp = synth.make_draft_inputs(w, device="cuda")
    tok, _ = sv.spec_draft_step(inp["draft_hidden"][0], inp["W"], None, 0.0)
    z = sv.spec_lm_head(inp["draft_hidden"][0], inp["W"])
    ref = draft_head.draft_step(np64(inp["draft_hidden"][0]), np64(inp["W"]), None, 0.0)
    err = np.abs(np64(z) - ref["logits"]).max()
    tok = tok.cpu().numpy()
    for b in range(w.B):
        if tok[b] != ref["tokens"][b]:
            assert ref["top2_gap"][b] <= 2 * err + 1e-12, (b, tok[b], ref["tokens"][b], ref["top2_gap"][b])


@pytest.mark.parametrize("name", sorted(synth.DRAFT_WORKLOADS))
def test_round_drafted_through_the_lm_head(name):
    """K draft steps write slots j of one [B][K][V] draft-logits buffer
    (strided rows), then the verify step checks the round; every draft step
    and the verify result agree with the oracle."""
    w = synth.DRAFT_WORKLOADS[name]
    B, K, d, V, T = w.B, w.K, w.d, w.V, w.temperature
    inp = synth.make_draft_inputs(w, device="cuda")
    dl = torch.empty((B, K, V), dtype=torch.float32, device="cuda")
    x = torch.empty((B, K), dtype=torch.int32, device="cuda")
    ws = torch.empty(sv.draft_step_workspace_bytes(B, d, V, T), dtype=torch.uint8, device="cuda")
    for j in range(K):
        tok, _ = sv.spec_draft_step(inp["draft_hidden"][j], inp["W"], inp["draft_uniforms"][j], T,
                                    out_logits=dl[:, j, :], workspace=ws)
        x[:, j] = tok
    torch.cuda.synchronize()
    W64 = np64(inp["W"])
    zq = np.empty((B, K, V))
    for j in range(K):
        ref = draft_head.draft_step(np64(inp["draft_hidden"][j]), W64, np64(inp["draft_uniforms"][j]), t32(T))
        zq[:, j] = ref["logits"]
        check_step(x[:, j].cpu().numpy(), ref)
    assert np.abs(np64(dl) - zq).max() <= LOGIT_ATOL
    # verify the drafted round (draft logits and tokens exactly as the GPU drafted them)
    tokv, n = sv.spec_verify(inp["hidden"], inp["W"], dl.view(B * K, V), x, inp["uniforms"], T)
    ref = oracle.spec_verify(np64(inp["hidden"]), W64, np64(dl.view(B * K, V)), x.cpu().numpy(),
                             np64(inp["uniforms"]), t32(T), B, K)
    compare_sampling(tokv.cpu().numpy(), n.cpu().numpy(), ref, K)


def test_repeated_draws_full_size():
    """Many draws from fixed draft logits of the B=8, V=128256 step: the
    inverse-CDF draw agrees with the oracle's on every draw outside the band."""
    w = synth.DRAFT_WORKLOADS["draft_B8_K4_V128256"]
    inp = synth.make_draft_inputs(w, device="cuda")
    h, W = inp["draft_hidden"][0], inp["W"]
    B, V, T = w.B, w.V, w.temperature
    logits = torch.empty((B, V), dtype=torch.float32, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(11)
    z = draft_head.draft_step(np64(h), np64(W), np.zeros(B), t32(T))["logits"]
    exempt = 0
    for r in range(64):
        u = torch.rand((B,), generator=g, device="cuda")
        tok, _ = sv.spec_draft_step(h, W, u, T, out_logits=logits)
        ref = draft_head.draft_step_from_logits(z, np64(u), t32(T))
        exempt += check_step(tok.cpu().numpy(), ref)
    assert exempt <= 1


def test_strided_slot_above_the_fused_statistics_batch():
    """More rows than the small-batch LM head takes (the large-batch head,
    its statistics in the epilogue), writing slot 1 of a [B][3][V] buffer."""
    B, d, V, T = 100, 256, 5003, 0.9
    w = synth.custom("draft_strided", B=B, K=1, d=d, V=V, temperature=T, seed=21)
    inp = synth.make_draft_inputs(w, device="cuda")
    buf = torch.full((B, 3, V), float("nan"), dtype=torch.float32, device="cuda")
    tok, _ = sv.spec_draft_step(inp["draft_hidden"][0], inp["W"], inp["draft_uniforms"][0], T,
                                out_logits=buf[:, 1, :])
    torch.cuda.synchronize()
    ref = draft_head.draft_step(np64(inp["draft_hidden"][0]), np64(inp["W"]), np64(inp["draft_uniforms"][0]),
                                t32(T))
    assert np.abs(np64(buf[:, 1, :]) - ref["logits"]).max() <= LOGIT_ATOL
    assert torch.isnan(buf[:, 0, :]).all() and torch.isnan(buf[:, 2, :]).all()   # other slots untouched
    check_step(tok.cpu().numpy(), ref)
