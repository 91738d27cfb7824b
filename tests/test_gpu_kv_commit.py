"""KV-cache commit on the GPU against the oracle (oracle/kv_commit.py):
pool bytes and lengths bit-exact, on seeded synthetic caches."""
import numpy as np
import pytest
import torch

import speculative_decoding_verification_67_gb300 as sv
from oracle import kv_commit
from speculative_decoding_verification_67_gb300 import synth

pytestmark = pytest.mark.gpu


def run_both(inp, page_size, in_place=False, S=None):
    """Commit on the GPU and in the oracle from identical inputs; returns
    (gpu pool, gpu lengths, gpu error word, oracle pool, oracle lengths, oracle bad)."""
    host = {k: v.cpu().numpy() for k, v in inp.items()}
    pool = inp["pool"].clone()
    seq_len = inp["seq_len"].clone()
    if in_place:
        ws = sv.spec_kv_commit(inp["num_accepted"], seq_len, inp["block_table"], pool, None, S=S)
        ref_len, ref_bad = kv_commit.commit_in_place(host["num_accepted"], host["seq_len"], host["block_table"],
                                                     host["pool"].shape[1], page_size, S)
        ref_pool = host["pool"]
    else:
        ws = sv.spec_kv_commit(inp["num_accepted"], seq_len, inp["block_table"], pool, inp["staged"])
        ref_pool = host["pool"].copy()
        ref_len, ref_bad = kv_commit.commit(host["num_accepted"], host["seq_len"], host["block_table"], ref_pool,
                                            host["staged"], page_size)
    err = sv.kv_commit_read_error(ws)
    return pool.cpu().numpy(), seq_len.cpu().numpy(), err, ref_pool, ref_len, ref_bad


def small(B, K, layers, E, page_size, draft=False, seed=1, max_len=40, bad_rows=0):
    w = synth.KvWorkload("kv_case", B=B, K=K, layers=layers, entry_bytes=E, page_size=page_size, min_len=0,
                         max_len=max_len, accept_rate=0.6, draft_cache=draft, seed=seed)
    return w, synth.make_kv_inputs(w, device="cuda", bad_rows=bad_rows)


@pytest.mark.parametrize("page_size", [1, 3, 16])
@pytest.mark.parametrize("E", [16, 48, 4096, 4096 * 2 + 16 * 5])
@pytest.mark.parametrize("draft", [False, True])
def test_staged_commit_matches_oracle(page_size, E, draft):
    w, inp = small(B=7, K=4, layers=3, E=E, page_size=page_size, draft=draft, seed=E + page_size, bad_rows=1)
    n = inp["num_accepted"]
    n[0] = w.K                      # an all-accepted sequence
    n[1] = 0
    pool, lens, err, ref_pool, ref_len, ref_bad = run_both(inp, page_size)
    assert not ref_bad.any()
    assert err == 0
    assert np.array_equal(lens, ref_len)
    assert np.array_equal(pool, ref_pool)


def test_in_place_commit_only_moves_lengths():
    w, inp = small(B=9, K=6, layers=2, E=64, page_size=4, bad_rows=2)
    pool, lens, err, ref_pool, ref_len, ref_bad = run_both(inp, 4, in_place=True, S=w.S)
    assert err == 0 and not ref_bad.any()
    assert np.array_equal(lens, ref_len)
    assert np.array_equal(pool, ref_pool)


def test_invalid_sequences_untouched_and_reported():
    w, inp = small(B=6, K=4, layers=2, E=32, page_size=4, seed=9)
    bt = inp["block_table"]
    L = inp["seq_len"]
    n = inp["num_accepted"]
    n[:] = 3
    L[1] = w.max_pages * 4 - 2          # committed range runs past the block table
    col = int(L[2]) // 4
    bt[2, col] = inp["pool"].shape[1] + 5   # a page outside the pool
    L[3] = -4                            # negative length
    pool, lens, err, ref_pool, ref_len, ref_bad = run_both(inp, 4)
    assert ref_bad.tolist() == [False, True, True, True, False, False]
    assert err == sv.KV_DEVERR_CAPACITY | sv.KV_DEVERR_PAGE | sv.KV_DEVERR_LENGTH
    assert np.array_equal(lens, ref_len)
    assert np.array_equal(pool, ref_pool)
    # the error word belongs to the latest call: a clean commit clears it
    n[:] = 0
    L[1:4] = 0
    bt[2, col] = 0
    ws = sv.spec_kv_commit(n, L.clone(), bt, inp["pool"].clone(), inp["staged"])
    assert sv.kv_commit_read_error(ws) == 0


def test_repeated_calls_reuse_the_workspace():
    """Four rounds through one workspace; lengths grow until some sequences
    run past their block table."""
    B, S, layers, E, ps, max_pages = 5, 4, 2, 80, 2, 8
    g = torch.Generator().manual_seed(3)
    bt = torch.randperm(B * max_pages, generator=g).to(torch.int32).view(B, max_pages)
    pool = torch.randint(0, 256, (layers, B * max_pages, ps, E), generator=g, dtype=torch.uint8)
    seq_len = torch.randint(0, 6, (B,), generator=g, dtype=torch.int32)
    ref_pool, ref_len = pool.numpy().copy(), seq_len.numpy().astype(np.int64)
    pool, seq_len, bt_d = pool.cuda(), seq_len.cuda(), bt.cuda()
    ws = sv.kv_workspace(pool, B, S, max_pages)
    for r in range(4):
        n = torch.randint(-1, S, (B,), generator=g, dtype=torch.int32)
        staged = torch.randint(0, 256, (layers, B, S, E), generator=g, dtype=torch.uint8)
        sv.spec_kv_commit(n.cuda(), seq_len, bt_d, pool, staged.cuda(), workspace=ws)
        ref_len, bad = kv_commit.commit(n.numpy(), ref_len, bt.numpy(), ref_pool, staged.numpy(), ps)
        assert (sv.kv_commit_read_error(ws) != 0) == bool(bad.any())
    assert np.array_equal(seq_len.cpu().numpy(), ref_len)
    assert np.array_equal(pool.cpu().numpy(), ref_pool)


@pytest.mark.parametrize("name", sorted(synth.KV_WORKLOADS))
def test_full_size_workloads(name):
    w = synth.KV_WORKLOADS[name]
    inp = synth.make_kv_inputs(w, device="cuda")
    pool, lens, err, ref_pool, ref_len, ref_bad = run_both(inp, w.page_size)
    assert err == 0 and not ref_bad.any()
    assert np.array_equal(lens, ref_len)
    assert np.array_equal(pool, ref_pool)


def test_commit_after_gpu_verify():
    """The verify step's own num_accepted (including its -1 rows) drives the
    commit of both caches."""
    vw = synth.custom("kv_verify", B=6, K=4, d=0, V=700, temperature=1.0)
    vin = synth.make_inputs(vw, device="cuda")
    x = vin["draft_tokens"].clone()
    x[2, 1] = vw.V + 3                   # a device-input error: sequence 2 comes back as -1
    tok, n = sv.spec_verify_from_logits(vin["target_logits"], vin["draft_logits"], x, vin["uniforms"], 1.0)
    assert int(n[2]) == -1
    for draft in (False, True):
        w, inp = small(B=6, K=4, layers=2, E=48, page_size=4, draft=draft, seed=21)
        inp["num_accepted"] = n.clone()
        pool, lens, err, ref_pool, ref_len, ref_bad = run_both(inp, 4)
        assert err == 0
        assert np.array_equal(lens, ref_len)
        assert np.array_equal(pool, ref_pool)


def test_large_batch_takes_the_plan_and_copy_path():
    """More sequences than the fused kernel's shared-memory scan holds: the
    one-CTA plan kernel and its dependent copy kernel."""
    w, inp = small(B=5000, K=2, layers=2, E=32, page_size=4, seed=77, max_len=30, bad_rows=7)
    pool, lens, err, ref_pool, ref_len, ref_bad = run_both(inp, 4)
    assert err == 0 and not ref_bad.any()
    assert np.array_equal(lens, ref_len)
    assert np.array_equal(pool, ref_pool)


def test_fused_ticket_returns_to_zero():
    w, inp = small(B=33, K=3, layers=4, E=64, page_size=8, seed=12)
    ws = sv.spec_kv_commit(inp["num_accepted"], inp["seq_len"].clone(), inp["block_table"], inp["pool"].clone(),
                           inp["staged"])
    torch.cuda.synchronize()
    ctrl = ws[:12].view(torch.int32).cpu().tolist()
    assert ctrl[0] == 0 and ctrl[2] == 0
    assert ctrl[1] == int((inp["num_accepted"].cpu().clamp_min(-1) + 1).clamp(max=w.S).sum())
