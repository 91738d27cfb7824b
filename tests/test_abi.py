"""The C-ABI library: it builds for sm_103a, loads without a GPU, exports every
symbol the headers under include/ declare, and rejects bad host-side arguments
before touching CUDA."""
import ctypes
import os
import re

import pytest

import speculative_decoding_verification_67_gb300 as sv
from speculative_decoding_verification_67_gb300 import _build

INCLUDE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return sv.library()


def declared_functions():
    names = set()
    for header in sorted(os.listdir(INCLUDE)):
        if header.endswith(".h"):
            text = open(os.path.join(INCLUDE, header)).read()
            names |= set(re.findall(r"SPEC_API\s+[\w\s\*]*?\b(spec_\w+)\s*\(", text))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 9, names
    for name in names:
        assert hasattr(lib, name), name


def test_version_and_status_strings(lib):
    assert lib.spec_abi_version() == 1
    for s in range(8):
        assert lib.spec_status_string(s).decode().startswith("SPEC_")
    assert lib.spec_status_string(99).decode() == "SPEC_ERR_UNKNOWN"


def test_workspace_sizes(lib):
    small = sv.workspace_bytes(1, 4, 1000, 1.0, logits_in_workspace=False)
    with_logits = sv.workspace_bytes(1, 4, 1000, 1.0, logits_in_workspace=True)
    assert with_logits - small >= 5 * 1000 * 4
    greedy = sv.workspace_bytes(256, 4, 128256, 0.0)
    assert greedy >= 1280 * ((128256 + 127) // 128) * 8
    assert lib.spec_verify_workspace_bytes(sv.SpecDims(0, 4, 0, 1000), 1.0, 1) == 0
    assert lib.spec_verify_workspace_bytes(sv.SpecDims(1, 33, 0, 1000), 1.0, 1) == 0
    assert lib.spec_verify_workspace_bytes(sv.SpecDims(1, 4, 0, 1000), -1.0, 1) == 0


def _fake(addr):
    return ctypes.c_void_p(addr)


def test_host_side_argument_errors(lib):
    """Errors that are returned before any CUDA call (safe without a GPU)."""
    good = _fake(0x10000)
    d = sv.SpecDims(2, 3, 64, 1000)
    ws = sv.workspace_bytes(2, 3, 1000, 0.8)
    args = lambda **kw: dict(dict(h=good, W=good, dl=good, x=good, u=good, T=0.8, ot=good, on=good, dims=d,
                                  ws=good, nws=ws, otl=_fake(None), dbg=_fake(None), s=_fake(None)), **kw)

    def call(**kw):
        a = args(**kw)
        return lib.spec_verify(a["h"], a["W"], a["dl"], a["x"], a["u"], a["T"], a["ot"], a["on"], a["dims"],
                               a["ws"], a["nws"], a["otl"], a["dbg"], a["s"])

    assert call(dims=sv.SpecDims(0, 3, 64, 1000)) == 2          # B < 1
    assert call(dims=sv.SpecDims(2, 40, 64, 1000)) == 2         # K > 32
    assert call(dims=sv.SpecDims(2, 3, 60, 1000)) == 2          # d % 8
    assert call(h=_fake(None)) == 1                              # null hidden
    assert call(h=_fake(0x10008)) == 3                           # misaligned
    assert call(T=float("nan")) == 1
    assert call(T=-1.0) == 1
    assert call(dl=_fake(None)) == 1                             # sampling needs draft logits
    assert call(u=_fake(None)) == 1
    assert call(ws=_fake(None)) == 4
    assert call(nws=ws - 1) == 4
    assert call(T=0.0, otl=good) == 1                            # greedy never writes logits
    assert lib.spec_lm_head(good, good, good, 0, 64, 1000, _fake(None)) == 2
    assert lib.spec_lm_head(good, good, _fake(None), 4, 64, 1000, _fake(None)) == 1
    assert lib.spec_verify_from_logits(_fake(None), good, good, good, 1.0, good, good, d, good, ws,
                                       _fake(None), _fake(None)) == 1


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    monkeypatch.setattr(sv, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(sv, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        sv.library()


def test_kv_commit_host_side_errors(lib):
    good = _fake(0x10000)
    d = sv.SpecKvDims(4, 5, 2, 16, 100, 10, 4096)

    nws = lib.spec_kv_commit_workspace_bytes(d)
    assert nws >= 256 + 8 * 4 * 5
    assert lib.spec_kv_commit_workspace_bytes(sv.SpecKvDims(0, 5, 2, 16, 100, 10, 4096)) == 0

    def call(n=good, L=good, bt=good, st=good, pool=good, dims=d, ws=good, size=nws):
        return lib.spec_kv_commit(n, L, bt, st, pool, dims, ws, size, _fake(None))

    assert call(n=_fake(None)) == 1
    assert call(ws=_fake(None)) == 1
    assert call(pool=_fake(None)) == 1                          # staged mode needs the pool
    assert call(dims=sv.SpecKvDims(0, 5, 2, 16, 100, 10, 4096)) == 2
    assert call(dims=sv.SpecKvDims(4, 257, 2, 16, 100, 10, 4096)) == 2
    assert call(dims=sv.SpecKvDims(4, 5, 2, 16, 100, 10, 24)) == 2   # entry_bytes % 16
    assert call(dims=sv.SpecKvDims(4, 5, 2, 0, 100, 10, 4096)) == 2
    assert call(st=_fake(0x10008)) == 3
    assert call(ws=_fake(0x10004)) == 3
    assert call(L=_fake(0x10002)) == 3
    assert call(size=nws - 1) == 4


def test_ngram_host_side_errors(lib):
    good = _fake(0x10000)
    d = sv.SpecNgramDims(4, 1024, 4, 1, 3)
    nws = lib.spec_ngram_workspace_bytes(d)
    assert nws >= 256 + 4 * 12
    for bad in (sv.SpecNgramDims(0, 1024, 4, 1, 3), sv.SpecNgramDims(4, 1022, 4, 1, 3),
                sv.SpecNgramDims(4, 1024, 33, 1, 3), sv.SpecNgramDims(4, 1024, 4, 3, 2),
                sv.SpecNgramDims(4, 1024, 4, 1, 17), sv.SpecNgramDims(4, 1024, 4, 0, 3)):
        assert lib.spec_ngram_workspace_bytes(bad) == 0

    def call(h=good, L=good, od=good, oc=good, dims=d, ws=good, size=nws):
        return lib.spec_ngram_propose(h, L, od, oc, dims, ws, size, _fake(None))

    assert call(h=_fake(None)) == 1
    assert call(dims=sv.SpecNgramDims(4, 1022, 4, 1, 3)) == 2
    assert call(h=_fake(0x10004)) == 3
    assert call(oc=_fake(0x10002)) == 3
    assert call(size=nws - 1) == 4


def test_draft_step_host_side_errors(lib):
    good = _fake(0x10000)
    d = sv.SpecDims(4, 0, 512, 5000)
    nws = lib.spec_draft_step_workspace_bytes(d, 0.8)
    assert nws > 0 and lib.spec_draft_step_workspace_bytes(d, -1.0) == 0
    assert lib.spec_draft_step_workspace_bytes(sv.SpecDims(4, 0, 500, 5000), 0.8) == 0   # d % 8

    def call(h=good, W=good, u=good, T=0.8, ot=good, ol=good, ld=5000, dims=d, ws=good, size=nws):
        return lib.spec_draft_step(h, W, u, T, ot, ol, ld, dims, ws, size, _fake(None))

    assert call(h=_fake(None)) == 1
    assert call(u=_fake(None)) == 1                 # sampling needs uniforms
    assert call(T=0.0) == 1                         # greedy never writes logits
    assert call(ld=4999) == 1
    assert call(T=float("nan")) == 1
    assert call(dims=sv.SpecDims(0, 0, 512, 5000)) == 2
    assert call(h=_fake(0x10008)) == 3
    assert call(ol=_fake(None), size=nws - 1) == 4   # logits kept in the workspace


def test_tree_host_side_errors(lib):
    good = _fake(0x10000)
    d = sv.SpecTreeDims(2, 16, 512, 5000)
    nws = lib.spec_tree_workspace_bytes(d, 0.8, 1)
    assert nws >= 256 + 4 * 32 * 5000
    assert lib.spec_tree_workspace_bytes(sv.SpecTreeDims(2, 257, 512, 5000), 0.8, 1) == 0     # N > 256
    assert lib.spec_tree_workspace_bytes(sv.SpecTreeDims(2, 16, 512, 200000), 0.8, 1) == 0    # V too large

    def call(h=good, W=good, dl=good, tok=good, par=good, u=good, T=0.8, ot=good, op=good, on=good, dims=d, ws=good,
             size=nws, otl=_fake(None)):
        return lib.spec_tree_verify(h, W, dl, tok, par, u, T, ot, op, on, dims, ws, size, otl, _fake(None))

    assert call(h=_fake(None)) == 1
    assert call(par=_fake(None)) == 1
    assert call(u=_fake(None)) == 1
    assert call(T=0.0, otl=good) == 1
    assert call(dims=sv.SpecTreeDims(2, 0, 512, 5000)) == 2
    assert call(dims=sv.SpecTreeDims(2, 16, 500, 5000)) == 2
    assert call(dl=_fake(0x10004)) == 3
    assert call(size=nws - 1) == 4


def _noalloc_boundary(lib, K, V, T):
    """The largest B whose from-logits workspace fits the no-allocation scratch."""
    size = lambda B: lib.spec_verify_from_logits_workspace_bytes(sv.SpecDims(B, K, 0, V), T)
    B = 1
    while size(B + 1) <= sv.NOALLOC_SCRATCH_BYTES:
        B += 1
    return B, size(B), size(B + 1)


def test_from_logits_workspace_query(lib):
    T = 0.8
    for B, K, V in [(1, 4, 1000), (8, 4, 128256), (64, 8, 152064), (3, 0, 5000)]:
        for t in (T, 0.0):
            exact = lib.spec_verify_from_logits_workspace_bytes(sv.SpecDims(B, K, 0, V), t)
            upper = lib.spec_verify_workspace_bytes(sv.SpecDims(B, K, 0, V), t, 0)
            assert 0 < exact <= upper, (B, K, V, t, exact, upper)
    assert lib.spec_verify_from_logits_workspace_bytes(sv.SpecDims(0, 4, 0, 1000), T) == 0
    assert lib.spec_verify_from_logits_workspace_bytes(sv.SpecDims(1, 4, 0, 1000), -1.0) == 0
    assert lib.spec_verify_from_logits_workspace_bytes(sv.SpecDims(1, 4, 0, 1000), float("inf")) == 0


@pytest.mark.parametrize("K,V,T", [(4, 128256, 0.8), (8, 152064, 1.0), (4, 128256, 0.0)])
def test_noalloc_limit_follows_the_documented_query(lib, K, V, T):
    """The no-allocation entry point refuses exactly the requests whose
    spec_verify_from_logits_workspace_bytes exceeds its scratch: one sequence
    more than the largest that fits is refused before any pointer is looked
    at; the largest that fits passes the size rule (and then fails on the
    null logits pointer, or without a GPU on the device query)."""
    B, fits, over = _noalloc_boundary(lib, K, V, T)
    assert fits <= sv.NOALLOC_SCRATCH_BYTES < over
    call = lambda b: lib.spec_verify_from_logits_noalloc(None, None, None, None, T, None, None,
                                                         sv.SpecDims(b, K, 0, V), None, None)
    assert call(B + 1) == 8   # SPEC_ERR_SCRATCH_LIMIT
    assert call(B) in (1, 5)  # SPEC_ERR_ARG on a GPU machine, SPEC_ERR_CUDA without one
