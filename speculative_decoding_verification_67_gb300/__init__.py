"""Target-side verify-and-accept step of speculative decoding on one GB300.

Python binding of the C-ABI library ``libspec_verify.so`` (declared in
``include/spec_verify.h``).  The functions here only check and marshal
arguments (torch tensors -> device pointers, the current CUDA stream); every
step of the computation runs in the library's sm_103a kernels.  There is no
fallback: if the library has not been built, every call raises.

Names follow the C ABI:

* :func:`spec_verify` -- LM head + verify-and-accept from hidden states;
* :func:`spec_verify_from_logits` -- verify-and-accept on given logits;
* :func:`spec_lm_head` -- the LM-head contraction alone;
* :func:`spec_verify_host` -- :func:`spec_verify` with host (CPU) tensors;
* :func:`read_error` -- the device error word of a workspace;
* :func:`spec_kv_commit` -- commit the kept cache entries of a round
  (``include/spec_kv_commit.h``);
* :func:`spec_ngram_propose` -- prompt-lookup drafts (``include/spec_ngram.h``);
* :func:`spec_draft_step` -- one draft step through the target's LM head
  (``include/spec_draft.h``);
* :func:`spec_tree_verify` / :func:`spec_tree_verify_from_logits` -- tree-shaped
  candidates (``include/spec_tree.h``).
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "SPEC_DEBUG_FIELDS", "SpecError", "library", "workspace_bytes", "host_workspace_bytes",
    "spec_verify", "spec_verify_from_logits", "spec_lm_head", "spec_verify_host", "read_error",
    "spec_verify_from_logits_noalloc", "noalloc_read_error", "Verifier",
    "kv_workspace", "spec_kv_commit", "kv_commit_read_error",
    "ngram_workspace", "spec_ngram_propose", "ngram_read_error",
    "draft_step_workspace_bytes", "spec_draft_step",
    "tree_workspace_bytes", "spec_tree_verify", "spec_tree_verify_from_logits",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libspec_verify.so")
SPEC_DEBUG_FIELDS = 6
DEVERR_TOKEN_RANGE, DEVERR_NONFINITE, DEVERR_TIMEOUT = 0x1, 0x2, 0x4


class SpecDims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("K", ctypes.c_int32), ("d", ctypes.c_int32), ("V", ctypes.c_int32)]


class SpecKvDims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("S", ctypes.c_int32), ("layers", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("num_pages", ctypes.c_int32), ("max_pages", ctypes.c_int32),
                ("entry_bytes", ctypes.c_int64)]


class SpecNgramDims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("max_len", ctypes.c_int32), ("K", ctypes.c_int32),
                ("n_min", ctypes.c_int32), ("n_max", ctypes.c_int32)]


class SpecTreeDims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("N", ctypes.c_int32), ("d", ctypes.c_int32), ("V", ctypes.c_int32)]


class SpecError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


_lib = None

_VP, _I32, _F32, _SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
_SIGS = {
    "spec_abi_version": (_I32, []),
    "spec_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "spec_verify_workspace_bytes": (_SZ, [SpecDims, _F32, _I32]),
    "spec_verify_from_logits_workspace_bytes": (_SZ, [SpecDims, _F32]),
    "spec_verify": (ctypes.c_int, [_VP, _VP, _VP, _VP, _VP, _F32, _VP, _VP, SpecDims, _VP, _SZ, _VP, _VP, _VP]),
    "spec_verify_timed": (ctypes.c_int, [_VP, _VP, _VP, _VP, _VP, _F32, _VP, _VP, SpecDims, _VP, _SZ, _VP, _VP, _VP,
                                         ctypes.POINTER(_VP)]),
    "spec_verify_from_logits": (ctypes.c_int, [_VP, _VP, _VP, _VP, _F32, _VP, _VP, SpecDims, _VP, _SZ, _VP, _VP]),
    "spec_lm_head": (ctypes.c_int, [_VP, _VP, _VP, _I32, _I32, _I32, _VP]),
    "spec_verify_host_workspace_bytes": (_SZ, [SpecDims, _F32]),
    "spec_verify_host": (ctypes.c_int, [_VP, _VP, _VP, _VP, _VP, _F32, _VP, _VP, SpecDims, _VP, _SZ, _VP]),
    "spec_verify_host_async": (ctypes.c_int, [_VP, _VP, _VP, _VP, _VP, _F32, _VP, _VP, SpecDims, _VP, _SZ, _VP]),
    "spec_verify_read_error": (ctypes.c_int, [_VP, ctypes.POINTER(_I32), _VP]),
    "spec_verify_from_logits_noalloc": (ctypes.c_int, [_VP, _VP, _VP, _VP, _F32, _VP, _VP, SpecDims, _VP, _VP]),
    "spec_verify_noalloc_read_error": (ctypes.c_int, [ctypes.POINTER(_I32), _VP]),
    "spec_kv_commit_workspace_bytes": (_SZ, [SpecKvDims]),
    "spec_kv_commit": (ctypes.c_int, [_VP, _VP, _VP, _VP, _VP, SpecKvDims, _VP, _SZ, _VP]),
    "spec_kv_commit_read_error": (ctypes.c_int, [_VP, ctypes.POINTER(_I32), _VP]),
    "spec_ngram_workspace_bytes": (_SZ, [SpecNgramDims]),
    "spec_draft_step_workspace_bytes": (_SZ, [SpecDims, _F32]),
    "spec_tree_workspace_bytes": (_SZ, [SpecTreeDims, _F32, _I32]),
    "spec_tree_verify": (ctypes.c_int, [_VP, _VP, _VP, _VP, _VP, _VP, _F32, _VP, _VP, _VP, SpecTreeDims, _VP, _SZ,
                                        _VP, _VP]),
    "spec_tree_verify_from_logits": (ctypes.c_int, [_VP, _VP, _VP, _VP, _VP, _F32, _VP, _VP, _VP, SpecTreeDims, _VP,
                                                    _SZ, _VP]),
    "spec_draft_step": (ctypes.c_int, [_VP, _VP, _VP, _F32, _VP, _VP, ctypes.c_int64, SpecDims, _VP, _SZ, _VP]),
    "spec_ngram_propose": (ctypes.c_int, [_VP, _VP, _VP, _VP, SpecNgramDims, _VP, _SZ, _VP]),
    "spec_ngram_read_error": (ctypes.c_int, [_VP, ctypes.POINTER(_I32), _VP]),
}
NOALLOC_SCRATCH_BYTES = 1 << 20


def library() -> ctypes.CDLL:
    """The loaded C-ABI library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()' "
                "or python -m speculative_decoding_verification_67_gb300._build)")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _check(status: int) -> None:
    if status != 0:
        msg = library().spec_status_string(status).decode()
        raise SpecError(status, msg)


def _ptr(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(None if t is None else t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t, name, dtype, shape, device=None):
    if t is None:
        raise ValueError(f"{name} is required")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device == "cuda" and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device == "cpu" and t.is_cuda:
        raise ValueError(f"{name} must be a host tensor")
    return t


def workspace_bytes(B: int, K: int, V: int, temperature: float, logits_in_workspace: bool = True) -> int:
    n = library().spec_verify_workspace_bytes(SpecDims(B, K, 0, V), float(temperature), int(logits_in_workspace))
    if n == 0:
        raise ValueError("invalid sizes")
    return int(n)


def from_logits_workspace_bytes(B: int, K: int, V: int, temperature: float) -> int:
    """Workspace of spec_verify_from_logits (and the no-allocation limit's measure)."""
    n = library().spec_verify_from_logits_workspace_bytes(SpecDims(B, K, 0, V), float(temperature))
    if n == 0:
        raise ValueError("invalid sizes")
    return int(n)


def host_workspace_bytes(B: int, K: int, d: int, V: int, temperature: float) -> int:
    n = library().spec_verify_host_workspace_bytes(SpecDims(B, K, d, V), float(temperature))
    if n == 0:
        raise ValueError("invalid sizes")
    return int(n)


def _outputs(B, K, device, out_tokens, out_num_accepted):
    if out_tokens is None:
        out_tokens = torch.empty((B, K + 1), dtype=torch.int32, device=device)
    if out_num_accepted is None:
        out_num_accepted = torch.empty((B,), dtype=torch.int32, device=device)
    _need(out_tokens, "out_tokens", torch.int32, (B, K + 1), "cuda")
    _need(out_num_accepted, "out_num_accepted", torch.int32, (B,), "cuda")
    return out_tokens, out_num_accepted


def spec_verify(hidden, W_lm, draft_logits, draft_tokens, uniforms, temperature: float, *,
                out_tokens=None, out_num_accepted=None, workspace=None, out_target_logits=None,
                out_debug=None, stream=None, stage_events=None):
    """LM head + verify-and-accept.  hidden bf16 [B*(K+1), d], W_lm bf16 [V, d],
    draft_logits f32 [B*K, V] (None when temperature == 0), draft_tokens int32
    [B, K], uniforms f32 [B, K+1] (None when temperature == 0).
    Returns (out_tokens int32 [B, K+1], out_num_accepted int32 [B])."""
    B, K = draft_tokens.shape
    V, d = W_lm.shape
    T = float(temperature)
    _need(draft_tokens, "draft_tokens", torch.int32, (B, K), "cuda")
    _need(hidden, "hidden", torch.bfloat16, (B * (K + 1), d), "cuda")
    _need(W_lm, "W_lm", torch.bfloat16, (V, d), "cuda")
    if T > 0:
        _need(draft_logits, "draft_logits", torch.float32, (B * K, V), "cuda")
        _need(uniforms, "uniforms", torch.float32, (B, K + 1), "cuda")
    if out_target_logits is not None:
        _need(out_target_logits, "out_target_logits", torch.float32, (B * (K + 1), V), "cuda")
    if out_debug is not None:
        _need(out_debug, "out_debug", torch.float32, (B, K + 1, SPEC_DEBUG_FIELDS), "cuda")
    out_tokens, out_num_accepted = _outputs(B, K, hidden.device, out_tokens, out_num_accepted)
    need = library().spec_verify_workspace_bytes(SpecDims(B, K, d, V), T, int(out_target_logits is None))
    if workspace is None:
        workspace = torch.empty(max(int(need), 16), dtype=torch.uint8, device=hidden.device)
    args = (_ptr(hidden), _ptr(W_lm), _ptr(draft_logits if T > 0 else None), _ptr(draft_tokens if K > 0 else None),
            _ptr(uniforms if T > 0 else None), T, _ptr(out_tokens), _ptr(out_num_accepted), SpecDims(B, K, d, V),
            _ptr(workspace), workspace.numel(), _ptr(out_target_logits), _ptr(out_debug), _stream(stream))
    if stage_events is None:
        _check(library().spec_verify(*args))
    else:
        # three torch.cuda.Event(enable_timing=True): before the LM head,
        # between the head and the finishing kernel, after it
        handles = (_VP * 3)(*[ctypes.c_void_p(ev.cuda_event) for ev in stage_events])
        _check(library().spec_verify_timed(*args, handles))
    return out_tokens, out_num_accepted


def spec_verify_from_logits(target_logits, draft_logits, draft_tokens, uniforms, temperature: float, *,
                            out_tokens=None, out_num_accepted=None, workspace=None, out_debug=None,
                            stream=None):
    """Verify-and-accept on given target logits f32 [B*(K+1), V]."""
    B, K = draft_tokens.shape
    V = target_logits.shape[1]
    T = float(temperature)
    _need(draft_tokens, "draft_tokens", torch.int32, (B, K), "cuda")
    _need(target_logits, "target_logits", torch.float32, (B * (K + 1), V), "cuda")
    if T > 0:
        _need(draft_logits, "draft_logits", torch.float32, (B * K, V), "cuda")
        _need(uniforms, "uniforms", torch.float32, (B, K + 1), "cuda")
    if out_debug is not None:
        _need(out_debug, "out_debug", torch.float32, (B, K + 1, SPEC_DEBUG_FIELDS), "cuda")
    out_tokens, out_num_accepted = _outputs(B, K, target_logits.device, out_tokens, out_num_accepted)
    need = library().spec_verify_from_logits_workspace_bytes(SpecDims(B, K, 0, V), T)
    if workspace is None:
        workspace = torch.empty(max(int(need), 16), dtype=torch.uint8, device=target_logits.device)
    _check(library().spec_verify_from_logits(
        _ptr(target_logits), _ptr(draft_logits if T > 0 else None), _ptr(draft_tokens if K > 0 else None),
        _ptr(uniforms if T > 0 else None), T, _ptr(out_tokens), _ptr(out_num_accepted), SpecDims(B, K, 0, V),
        _ptr(workspace), workspace.numel(), _ptr(out_debug), _stream(stream)))
    return out_tokens, out_num_accepted


def spec_verify_from_logits_noalloc(target_logits, draft_logits, draft_tokens, uniforms, temperature: float, *,
                                    out_tokens, out_num_accepted, out_debug=None, stream=None):
    """spec_verify_from_logits without a workspace, for callers that cannot
    allocate device memory while they decode (the library's fixed
    NOALLOC_SCRATCH_BYTES array serves as scratch; calls on one device must
    not overlap).  The outputs must be given: nothing is allocated here."""
    B, K = draft_tokens.shape
    V = target_logits.shape[1]
    T = float(temperature)
    _need(draft_tokens, "draft_tokens", torch.int32, (B, K), "cuda")
    _need(target_logits, "target_logits", torch.float32, (B * (K + 1), V), "cuda")
    if T > 0:
        _need(draft_logits, "draft_logits", torch.float32, (B * K, V), "cuda")
        _need(uniforms, "uniforms", torch.float32, (B, K + 1), "cuda")
    _need(out_tokens, "out_tokens", torch.int32, (B, K + 1), "cuda")
    _need(out_num_accepted, "out_num_accepted", torch.int32, (B,), "cuda")
    if out_debug is not None:
        _need(out_debug, "out_debug", torch.float32, (B, K + 1, SPEC_DEBUG_FIELDS), "cuda")
    _check(library().spec_verify_from_logits_noalloc(
        _ptr(target_logits), _ptr(draft_logits if T > 0 else None), _ptr(draft_tokens if K > 0 else None),
        _ptr(uniforms if T > 0 else None), T, _ptr(out_tokens), _ptr(out_num_accepted), SpecDims(B, K, 0, V),
        _ptr(out_debug), _stream(stream)))
    return out_tokens, out_num_accepted


def noalloc_read_error(stream=None) -> int:
    """Device error word of the no-allocation entry point's last call."""
    word = ctypes.c_int32(0)
    st = library().spec_verify_noalloc_read_error(ctypes.byref(word), _stream(stream))
    if st not in (0, 7):
        _check(st)
    return int(word.value)


def spec_lm_head(hidden, W_lm, logits=None, stream=None):
    """logits f32 [M, V] = hidden bf16 [M, d] @ W_lm bf16 [V, d]^T."""
    M, d = hidden.shape
    V = W_lm.shape[0]
    _need(hidden, "hidden", torch.bfloat16, (M, d), "cuda")
    _need(W_lm, "W_lm", torch.bfloat16, (V, d), "cuda")
    if logits is None:
        logits = torch.empty((M, V), dtype=torch.float32, device=hidden.device)
    _need(logits, "logits", torch.float32, (M, V), "cuda")
    _check(library().spec_lm_head(_ptr(hidden), _ptr(W_lm), _ptr(logits), M, d, V, _stream(stream)))
    return logits


def spec_verify_host(hidden, W_lm, draft_logits, draft_tokens, uniforms, temperature: float, *,
                     workspace=None, out_tokens=None, out_num_accepted=None, stream=None, wait: bool = True):
    """spec_verify with the per-step tensors (hidden, draft_logits, draft_tokens,
    uniforms) and the outputs in host memory (pin them for asynchronous
    copies); W_lm stays on the device.  Returns host tensors once they are
    ready; with ``wait=False`` (spec_verify_host_async) it returns at once and
    the outputs are valid after the stream's work completes -- the inputs must
    stay unmodified until then."""
    B, K = draft_tokens.shape
    V, d = W_lm.shape
    T = float(temperature)
    _need(draft_tokens, "draft_tokens", torch.int32, (B, K), "cpu")
    _need(hidden, "hidden", torch.bfloat16, (B * (K + 1), d), "cpu")
    _need(W_lm, "W_lm", torch.bfloat16, (V, d), "cuda")
    if T > 0:
        _need(draft_logits, "draft_logits", torch.float32, (B * K, V), "cpu")
        _need(uniforms, "uniforms", torch.float32, (B, K + 1), "cpu")
    if out_tokens is None:
        out_tokens = torch.empty((B, K + 1), dtype=torch.int32).pin_memory()
    if out_num_accepted is None:
        out_num_accepted = torch.empty((B,), dtype=torch.int32).pin_memory()
    _need(out_tokens, "out_tokens", torch.int32, (B, K + 1), "cpu")
    _need(out_num_accepted, "out_num_accepted", torch.int32, (B,), "cpu")
    if workspace is None:
        workspace = torch.empty(host_workspace_bytes(B, K, d, V, T), dtype=torch.uint8, device=W_lm.device)
    fn = library().spec_verify_host if wait else library().spec_verify_host_async
    _check(fn(
        _ptr(hidden), _ptr(W_lm), _ptr(draft_logits if T > 0 else None), _ptr(draft_tokens if K > 0 else None),
        _ptr(uniforms if T > 0 else None), T, _ptr(out_tokens), _ptr(out_num_accepted), SpecDims(B, K, d, V),
        _ptr(workspace), workspace.numel(), _stream(stream)))
    return out_tokens, out_num_accepted


def read_error(workspace, stream=None) -> int:
    """Synchronises the stream and returns the workspace's device error word."""
    word = ctypes.c_int32(0)
    st = library().spec_verify_read_error(_ptr(workspace), ctypes.byref(word), _stream(stream))
    if st not in (0, 7):
        _check(st)
    return int(word.value)


class Verifier:
    """Holds a workspace (and output buffers) sized for one shape, for
    repeated calls of :func:`spec_verify` without per-call allocation."""

    def __init__(self, B: int, K: int, d: int, V: int, temperature: float, device="cuda",
                 keep_logits: bool = False):
        self.B, self.K, self.d, self.V, self.T = B, K, d, V, float(temperature)
        self.target_logits = (torch.empty((B * (K + 1), V), dtype=torch.float32, device=device)
                              if keep_logits and self.T > 0 else None)
        n = library().spec_verify_workspace_bytes(SpecDims(B, K, d, V), self.T, int(self.target_logits is None))
        self.workspace = torch.empty(max(int(n), 16), dtype=torch.uint8, device=device)
        self.out_tokens = torch.empty((B, K + 1), dtype=torch.int32, device=device)
        self.out_num_accepted = torch.empty((B,), dtype=torch.int32, device=device)

    def __call__(self, hidden, W_lm, draft_logits, draft_tokens, uniforms, out_debug=None, stream=None,
                 stage_events=None):
        return spec_verify(hidden, W_lm, draft_logits, draft_tokens, uniforms, self.T,
                           out_tokens=self.out_tokens, out_num_accepted=self.out_num_accepted,
                           workspace=self.workspace, out_target_logits=self.target_logits,
                           out_debug=out_debug, stream=stream, stage_events=stage_events)


# ---------------------------------------------------------------- KV commit
KV_DEVERR_CAPACITY, KV_DEVERR_PAGE, KV_DEVERR_LENGTH = 1, 2, 4


def _kv_dims(num_accepted, block_table, pool, staged, S):
    if pool is None or pool.dim() != 4 or not pool.is_cuda or not pool.is_contiguous():
        raise ValueError("pool must be a contiguous CUDA tensor [layers][num_pages][page_size][E]")
    layers, num_pages, page_size, E = pool.shape
    B = num_accepted.shape[0]
    if staged is not None:
        if staged.dtype != pool.dtype:
            raise ValueError("staged and pool must share a dtype")
        S = staged.shape[2]
        _need(staged, "staged", pool.dtype, (layers, B, S, E), "cuda")
    elif S is None:
        raise ValueError("S is required in in-place mode")
    if block_table.dim() != 2:
        raise ValueError("block_table must be [B][max_pages]")
    return SpecKvDims(B, int(S), layers, page_size, num_pages, block_table.shape[1], E * pool.element_size())


def kv_workspace(pool, B: int, S: int, max_pages: int = 1, device=None) -> torch.Tensor:
    """A zeroed workspace for :func:`spec_kv_commit` on caches shaped like
    ``pool`` with ``B`` sequences of ``S`` staged entries (reusable across
    calls; each call leaves it ready for the next)."""
    layers, num_pages, page_size, E = pool.shape
    dims = SpecKvDims(B, S, layers, page_size, num_pages, max_pages, E * pool.element_size())
    n = library().spec_kv_commit_workspace_bytes(dims)
    if n == 0:
        raise ValueError("invalid sizes")
    return torch.zeros(int(n), dtype=torch.uint8, device=pool.device if device is None else device)


def spec_kv_commit(num_accepted, seq_len, block_table, pool, staged=None, *, S: int = None, workspace=None,
                   stream=None):
    """Commit one round's kept cache entries.

    ``pool`` [layers][num_pages][page_size][E] and ``staged``
    [layers][B][S][E] (same dtype; E elements make one entry) or None for
    in-place mode, where ``S`` must be given.  ``num_accepted`` and
    ``seq_len`` int32 [B] (``seq_len`` is advanced in place), ``block_table``
    int32 [B][max_pages].  Returns the workspace (its error word is read by
    :func:`kv_commit_read_error`)."""
    dims = _kv_dims(num_accepted, block_table, pool, staged, S)
    _need(num_accepted, "num_accepted", torch.int32, (dims.B,), "cuda")
    _need(seq_len, "seq_len", torch.int32, (dims.B,), "cuda")
    _need(block_table, "block_table", torch.int32, (dims.B, dims.max_pages), "cuda")
    if workspace is None:
        workspace = kv_workspace(pool, dims.B, dims.S, dims.max_pages)
    if workspace.dtype != torch.uint8 or not workspace.is_cuda:
        raise ValueError("workspace must be a CUDA uint8 tensor")
    _check(library().spec_kv_commit(_ptr(num_accepted), _ptr(seq_len), _ptr(block_table), _ptr(staged),
                                    _ptr(pool), dims, _ptr(workspace), workspace.numel(), _stream(stream)))
    return workspace


def kv_commit_read_error(workspace, stream=None) -> int:
    """Synchronises the stream and returns the error word of the latest commit
    on ``workspace`` (KV_DEVERR_* bits)."""
    word = ctypes.c_int32(0)
    _check(library().spec_kv_commit_read_error(_ptr(workspace), ctypes.byref(word), _stream(stream)))
    return int(word.value)


# ---------------------------------------------------------- prompt lookup
NGRAM_DEVERR_LENGTH, NGRAM_DEVERR_TIMEOUT = 1, 2


def ngram_workspace(B: int, max_len: int, K: int, n_min: int = 1, n_max: int = 3, device="cuda") -> torch.Tensor:
    """A zeroed workspace for :func:`spec_ngram_propose` (reusable across calls)."""
    n = library().spec_ngram_workspace_bytes(SpecNgramDims(B, max_len, K, n_min, n_max))
    if n == 0:
        raise ValueError("invalid sizes")
    return torch.zeros(int(n), dtype=torch.uint8, device=device)


def spec_ngram_propose(history, lengths, K: int, n_min: int = 1, n_max: int = 3, *, out_drafts=None,
                       out_count=None, workspace=None, stream=None):
    """Prompt-lookup drafts: ``history`` int32 [B][max_len] (max_len a
    multiple of 4), ``lengths`` int32 [B] -> (drafts int32 [B][K], count
    int32 [B])."""
    if history is None or history.dim() != 2:
        raise ValueError("history must be [B][max_len]")
    B, max_len = history.shape
    _need(history, "history", torch.int32, (B, max_len), "cuda")
    _need(lengths, "lengths", torch.int32, (B,), "cuda")
    if out_drafts is None:
        out_drafts = torch.empty((B, K), dtype=torch.int32, device=history.device)
    if out_count is None:
        out_count = torch.empty((B,), dtype=torch.int32, device=history.device)
    _need(out_drafts, "out_drafts", torch.int32, (B, K), "cuda")
    _need(out_count, "out_count", torch.int32, (B,), "cuda")
    if workspace is None:
        workspace = ngram_workspace(B, max_len, K, n_min, n_max, device=history.device)
    dims = SpecNgramDims(B, max_len, K, n_min, n_max)
    _check(library().spec_ngram_propose(_ptr(history), _ptr(lengths), _ptr(out_drafts), _ptr(out_count), dims,
                                        _ptr(workspace), workspace.numel(), _stream(stream)))
    return out_drafts, out_count


def ngram_read_error(workspace, stream=None) -> int:
    """Synchronises the stream; the error word of the latest proposal call."""
    word = ctypes.c_int32(0)
    _check(library().spec_ngram_read_error(_ptr(workspace), ctypes.byref(word), _stream(stream)))
    return int(word.value)


# --------------------------------------------------------------- draft step
def draft_step_workspace_bytes(B: int, d: int, V: int, temperature: float) -> int:
    n = library().spec_draft_step_workspace_bytes(SpecDims(B, 0, d, V), float(temperature))
    if n == 0:
        raise ValueError("invalid sizes")
    return int(n)


def spec_draft_step(hidden, W_lm, uniforms, temperature: float, *, out_tokens=None, out_logits=None,
                    workspace=None, stream=None):
    """One draft step through the target's LM head: ``hidden`` bf16 [B, d]
    (the draft model's estimate of the target's hidden state), ``W_lm`` bf16
    [V, d], ``uniforms`` f32 [B] (None at T = 0).  ``out_logits`` (T > 0
    only) is an f32 [B, V] view whose rows may be strided, e.g. slot j of a
    [B, K, V] draft-logits buffer.  Returns (tokens int32 [B], out_logits)."""
    B, d = hidden.shape
    V = W_lm.shape[0]
    T = float(temperature)
    _need(hidden, "hidden", torch.bfloat16, (B, d), "cuda")
    _need(W_lm, "W_lm", torch.bfloat16, (V, d), "cuda")
    if T > 0:
        _need(uniforms, "uniforms", torch.float32, (B,), "cuda")
    ld = 0
    if out_logits is not None:
        if out_logits.dtype != torch.float32 or tuple(out_logits.shape) != (B, V) or out_logits.stride(1) != 1 \
                or not out_logits.is_cuda:
            raise ValueError("out_logits must be a CUDA f32 [B, V] view with unit column stride")
        ld = out_logits.stride(0)
    if out_tokens is None:
        out_tokens = torch.empty((B,), dtype=torch.int32, device=hidden.device)
    _need(out_tokens, "out_tokens", torch.int32, (B,), "cuda")
    if workspace is None:
        workspace = torch.empty(draft_step_workspace_bytes(B, d, V, T), dtype=torch.uint8, device=hidden.device)
    _check(library().spec_draft_step(_ptr(hidden), _ptr(W_lm), _ptr(uniforms if T > 0 else None), T,
                                     _ptr(out_tokens), _ptr(out_logits), ld, SpecDims(B, 0, d, V),
                                     _ptr(workspace), workspace.numel(), _stream(stream)))
    return out_tokens, out_logits


# --------------------------------------------------------------- tree verify
def tree_workspace_bytes(B: int, N: int, V: int, temperature: float, logits_in_workspace: bool = True) -> int:
    n = library().spec_tree_workspace_bytes(SpecTreeDims(B, N, 0, V), float(temperature), int(logits_in_workspace))
    if n == 0:
        raise ValueError("invalid sizes")
    return int(n)


def _tree_outputs(B, N, device, out_tokens, out_path, out_num_accepted):
    if out_tokens is None:
        out_tokens = torch.empty((B, N), dtype=torch.int32, device=device)
    if out_path is None:
        out_path = torch.empty((B, N), dtype=torch.int32, device=device)
    if out_num_accepted is None:
        out_num_accepted = torch.empty((B,), dtype=torch.int32, device=device)
    _need(out_tokens, "out_tokens", torch.int32, (B, N), "cuda")
    _need(out_path, "out_path", torch.int32, (B, N), "cuda")
    _need(out_num_accepted, "out_num_accepted", torch.int32, (B,), "cuda")
    return out_tokens, out_path, out_num_accepted


def _tree_inputs(tokens, parents, uniforms, draft_logits, B, N, V, T):
    _need(tokens, "tokens", torch.int32, (B, N), "cuda")
    _need(parents, "parents", torch.int32, (B, N), "cuda")
    if T > 0:
        _need(uniforms, "uniforms", torch.float32, (B, N), "cuda")
        _need(draft_logits, "draft_logits", torch.float32, (B * N, V), "cuda")


def spec_tree_verify(hidden, W_lm, draft_logits, tokens, parents, uniforms, temperature: float, *, out_tokens=None,
                     out_path=None, out_num_accepted=None, workspace=None, out_target_logits=None, stream=None):
    """Tree verification from every node's hidden state: ``hidden`` bf16
    [B*N, d], ``W_lm`` bf16 [V, d], ``draft_logits`` f32 [B*N, V] (T > 0),
    ``tokens`` / ``parents`` int32 [B, N], ``uniforms`` f32 [B, N] (T > 0).
    Returns (tokens, path, num_accepted)."""
    B, N = tokens.shape
    M, d = hidden.shape
    V = W_lm.shape[0]
    T = float(temperature)
    _need(hidden, "hidden", torch.bfloat16, (B * N, d), "cuda")
    _need(W_lm, "W_lm", torch.bfloat16, (V, d), "cuda")
    _tree_inputs(tokens, parents, uniforms, draft_logits, B, N, V, T)
    outs = _tree_outputs(B, N, hidden.device, out_tokens, out_path, out_num_accepted)
    if out_target_logits is not None:
        _need(out_target_logits, "out_target_logits", torch.float32, (B * N, V), "cuda")
    if workspace is None:
        workspace = torch.empty(tree_workspace_bytes(B, N, V, T, out_target_logits is None), dtype=torch.uint8,
                                device=hidden.device)
    _check(library().spec_tree_verify(
        _ptr(hidden), _ptr(W_lm), _ptr(draft_logits if T > 0 else None), _ptr(tokens), _ptr(parents),
        _ptr(uniforms if T > 0 else None), T, _ptr(outs[0]), _ptr(outs[1]), _ptr(outs[2]),
        SpecTreeDims(B, N, d, V), _ptr(workspace), workspace.numel(), _ptr(out_target_logits), _stream(stream)))
    return outs


def spec_tree_verify_from_logits(target_logits, draft_logits, tokens, parents, uniforms, temperature: float, *,
                                 out_tokens=None, out_path=None, out_num_accepted=None, workspace=None, stream=None):
    """Tree verification on given target logits f32 [B*N, V]."""
    B, N = tokens.shape
    V = target_logits.shape[1]
    T = float(temperature)
    _need(target_logits, "target_logits", torch.float32, (B * N, V), "cuda")
    _tree_inputs(tokens, parents, uniforms, draft_logits, B, N, V, T)
    outs = _tree_outputs(B, N, target_logits.device, out_tokens, out_path, out_num_accepted)
    if workspace is None:
        # (sized for the LM-head path, which holds more partials than this one)
        workspace = torch.empty(tree_workspace_bytes(B, N, V, T, False), dtype=torch.uint8,
                                device=target_logits.device)
    _check(library().spec_tree_verify_from_logits(
        _ptr(target_logits), _ptr(draft_logits if T > 0 else None), _ptr(tokens), _ptr(parents),
        _ptr(uniforms if T > 0 else None), T, _ptr(outs[0]), _ptr(outs[1]), _ptr(outs[2]), SpecTreeDims(B, N, 0, V),
        _ptr(workspace), workspace.numel(), _stream(stream)))
    return outs
