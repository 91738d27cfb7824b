"""The no-allocation entry point (spec_verify_from_logits_noalloc).

It serves callers that cannot allocate device memory while they decode --
for instance a serving process that reserved the whole GPU for weights and
key-value cache at start-up -- by using a fixed scratch array inside the
library instead of a caller workspace.  These tests call it through the C ABI
and check that it returns exactly what the workspace-taking entry point
returns on the same inputs, on two calls in a row (the shared scratch keeps
the previous call's contents, which must not leak into the next result).

The file is named to be collected last, so that a run stopping at the first
failure has already run every other test.
"""
import pytest
import torch

import speculative_decoding_verification_67_gb300 as sv
from speculative_decoding_verification_67_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from speculative_decoding_verification_67_gb300 import _build
    _build.build()
    sv.library()


def _case(B, K, V, T, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    zp = torch.randn((B * (K + 1), V), generator=g, device="cuda") * 2.0
    zq = (zp.view(B, K + 1, V)[:, :K] + 0.5 * torch.randn((B, K, V), generator=g, device="cuda")).reshape(B * K, V)
    x = synth.gumbel_max_tokens(zq, T if T > 0 else 1.0, g).view(B, K).contiguous()
    u = torch.rand((B, K + 1), generator=g, device="cuda")
    return zp.contiguous(), zq.contiguous(), x, u


def _outputs(B, K):
    return (torch.full((B, K + 1), -7, dtype=torch.int32, device="cuda"),
            torch.full((B,), -7, dtype=torch.int32, device="cuda"),
            torch.zeros((B, K + 1, sv.SPEC_DEBUG_FIELDS), device="cuda"))


@pytest.mark.parametrize("B,K,V,T", [(1, 4, 1000, 1.0), (8, 4, 32000, 0.8), (16, 3, 5001, 0.0)])
def test_noalloc_matches_workspace_entry_point_twice(B, K, V, T):
    ref_tok, ref_n, ref_dbg = _outputs(B, K)
    for call, seed in enumerate((B * 7 + V, B * 7 + V + 1)):  # two calls in a row, different inputs
        zp, zq, x, u = _case(B, K, V, T, seed)
        sv.spec_verify_from_logits(zp, zq if T > 0 else None, x, u if T > 0 else None, T,
                                   out_tokens=ref_tok, out_num_accepted=ref_n, out_debug=ref_dbg)
        tok, n, dbg = _outputs(B, K)
        sv.spec_verify_from_logits_noalloc(zp, zq if T > 0 else None, x, u if T > 0 else None, T,
                                           out_tokens=tok, out_num_accepted=n, out_debug=dbg)
        torch.cuda.synchronize()
        assert torch.equal(tok, ref_tok), (call, tok, ref_tok)
        assert torch.equal(n, ref_n), (call, n, ref_n)
        # same kernels on the same inputs: the diagnostics agree to f32 rounding
        torch.testing.assert_close(dbg, ref_dbg, rtol=1e-5, atol=1e-6)
        assert sv.noalloc_read_error() == 0


def test_noalloc_refuses_requests_beyond_its_scratch():
    # B*(2K+1) rows x ceil(V/4096) partials of 16 bytes: 256*17*38*16 bytes = 2.6 MB > 1 MiB
    B, K, V = 256, 8, 152064
    assert B * (2 * K + 1) * ((V + 4095) // 4096) * 16 > sv.NOALLOC_SCRATCH_BYTES
    d = sv.SpecDims(B, K, 0, V)
    status = sv.library().spec_verify_from_logits_noalloc(None, None, None, None, 1.0, None, None, d, None, None)
    assert status == 8  # SPEC_ERR_SCRATCH_LIMIT, before any argument is touched
    assert "scratch" in sv.library().spec_status_string(8).decode()


def test_noalloc_at_the_largest_request_that_fits():
    """The largest batch whose from-logits workspace fits the fixed scratch
    (K = 4, V = 128256, T = 0.8), twice in a row: identical to the
    workspace entry point."""
    K, V, T = 4, 128256, 0.8
    lib = sv.library()
    size = lambda b: lib.spec_verify_from_logits_workspace_bytes(sv.SpecDims(b, K, 0, V), T)
    B = 1
    while size(B + 1) <= sv.NOALLOC_SCRATCH_BYTES:
        B += 1
    for seed in (11, 12):
        zp, zq, x, u = _case(B, K, V, T, seed)
        ref_tok, ref_n, _ = _outputs(B, K)
        sv.spec_verify_from_logits(zp, zq, x, u, T, out_tokens=ref_tok, out_num_accepted=ref_n)
        tok, n, _ = _outputs(B, K)
        sv.spec_verify_from_logits_noalloc(zp, zq, x, u, T, out_tokens=tok, out_num_accepted=n)
        torch.cuda.synchronize()
        assert torch.equal(tok, ref_tok) and torch.equal(n, ref_n), (B, seed)
        assert sv.noalloc_read_error() == 0
