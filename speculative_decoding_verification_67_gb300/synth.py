"""Seeded synthetic inputs for the verify-and-accept step.

This module is the one piece that the CUDA path and the CPU oracle both
consume.  It holds no arithmetic of the verify step itself: only random
draws and the stand-in for the draft model (a noisy copy of the target's
hidden state pushed through the same LM-head weight, whose tokens are drawn
with the Gumbel-max trick rather than with the inverse-CDF rule the verify
step uses).

Workloads (the five synthetic configurations the step is measured on):

=====================  ==============================================================
name                   recipe
=====================  ==============================================================
tiny_logits            B=1, K=4, V=1000, no LM head: target logits z_p ~ N(0, std 2)
                       for K+1 rows; draft logits z_q = z_p[:K] + N(0, std 0.5);
                       T = 1
head_B1_K5_V32000      B=1, K=5, d=4096, V=32000; h ~ N(0,1) bf16, W ~ N(0, 1/sqrt d)
                       bf16; z_q = (h[:K] + 0.3 eps) W^T in fp32; T = 1
head_B8_K4_V128256     B=8, K=4, d=4096, V=128256 (Llama-3-8B-shaped head);
                       noise 0.3; T = 0.8
head_B64_K8_V152064    B=64, K=8, d=8192, V=152064 (70B-class head); noise 1.0; T = 1
greedy_B256_K4_V128256 B=256, K=4, d=4096, V=128256; T = 0; drafts are the argmax of
                       (h + 0.2 eps) W^T; no draft logits, no uniforms
=====================  ==============================================================

"N(0, s)" names the standard deviation.  Draft tokens at T > 0 are sampled
from softmax(z_q / T) (Gumbel-max); uniforms are U[0, 1) fp32, K accept
uniforms and one draw uniform per sequence.  The seed of workload i (in the
table order, from 1) is 6700 + i.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    K: int
    d: int            # 0 = no LM head (logits are given)
    V: int
    temperature: float
    noise: float      # draft-side noise on the hidden state (std)
    logit_std: float = 2.0      # tiny_logits only: std of z_p
    draft_logit_noise: float = 0.5  # tiny_logits only: std of z_q - z_p
    seed: int = 0

    @property
    def M(self) -> int:
        return self.B * (self.K + 1)

    @property
    def greedy(self) -> bool:
        return self.temperature == 0.0


WORKLOADS = {
    w.name: w
    for w in (
        Workload("tiny_logits", B=1, K=4, d=0, V=1000, temperature=1.0, noise=0.0, seed=6701),
        Workload("head_B1_K5_V32000", B=1, K=5, d=4096, V=32000, temperature=1.0, noise=0.3, seed=6702),
        Workload("head_B8_K4_V128256", B=8, K=4, d=4096, V=128256, temperature=0.8, noise=0.3, seed=6703),
        Workload("head_B64_K8_V152064", B=64, K=8, d=8192, V=152064, temperature=1.0, noise=1.0, seed=6704),
        Workload("greedy_B256_K4_V128256", B=256, K=4, d=4096, V=128256, temperature=0.0, noise=0.2, seed=6705),
    )
}


def custom(name: str, B: int, K: int, d: int, V: int, temperature: float, noise: float = 0.3,
           seed: int = 1) -> Workload:
    """A workload of the same recipe at other sizes (parity cases, edge cases)."""
    return Workload(name, B=B, K=K, d=d, V=V, temperature=temperature, noise=noise, seed=seed)


def _gen(device: torch.device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(shape, g, device, chunk_rows: int = 16384) -> torch.Tensor:
    """Standard normal fp32 drawn in row chunks (bounded scratch for big W)."""
    out = torch.empty(shape, dtype=torch.float32, device=device)
    rows = shape[0]
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        out[r0:r1] = torch.randn((r1 - r0,) + tuple(shape[1:]), generator=g, device=device)
    return out


def _randn_bf16(shape, scale: float, g, device, chunk_rows: int = 16384) -> torch.Tensor:
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    rows = shape[0]
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        x = torch.randn((r1 - r0,) + tuple(shape[1:]), generator=g, device=device)
        out[r0:r1] = (x * scale).to(torch.bfloat16)
    return out


def _project(x: torch.Tensor, W: torch.Tensor, chunk_rows: int = 16384) -> torch.Tensor:
    """Draft-model stand-in: fp32 x times the bf16 weight (upcast), fp32 result.

    Plain fp32 matmul with TF32 disabled; the result is an input of the verify
    step, read byte-for-byte the same by the CUDA path and the oracle."""
    prev = torch.get_float32_matmul_precision()
    torch.set_float32_matmul_precision("highest")
    try:
        out = torch.empty((x.shape[0], W.shape[0]), dtype=torch.float32, device=x.device)
        for v0 in range(0, W.shape[0], chunk_rows):
            v1 = min(W.shape[0], v0 + chunk_rows)
            out[:, v0:v1] = x @ W[v0:v1].float().t()
        return out
    finally:
        torch.set_float32_matmul_precision(prev)


def gumbel_max_tokens(logits: torch.Tensor, temperature: float, g: torch.Generator) -> torch.Tensor:
    """Draw one token per row from softmax(logits / T) with the Gumbel-max trick."""
    u = torch.rand(logits.shape, generator=g, device=logits.device, dtype=torch.float64)
    u = u.clamp_min(1e-300)
    gumbel = -torch.log(-torch.log(u))
    return torch.argmax(logits.double() / temperature + gumbel, dim=-1).to(torch.int32)


def make_inputs(w: Workload, device="cpu", seed: int | None = None) -> dict:
    """All inputs of one verify call for workload ``w`` on ``device``.

    Returns a dict with (absent keys are None):
      hidden        bf16 [B*(K+1), d]   (row b*(K+1)+j is position j of sequence b)
      W             bf16 [V, d]         (LM-head weight, nn.Linear layout)
      target_logits fp32 [B*(K+1), V]   (tiny_logits only: the given z_p)
      draft_logits  fp32 [B*K, V]       (T > 0)
      draft_tokens  int32 [B, K]
      uniforms      fp32 [B, K+1]       (T > 0)
    """
    device = torch.device(device)
    g = _gen(device, w.seed if seed is None else seed)
    B, K, d, V = w.B, w.K, w.d, w.V
    out = dict(hidden=None, W=None, target_logits=None, draft_logits=None,
               draft_tokens=None, uniforms=None)
    if d == 0:
        zp = _randn((B * (K + 1), V), g, device) * w.logit_std
        zp3 = zp.view(B, K + 1, V)
        eps = _randn((B * K, V), g, device).view(B, K, V)
        zq = (zp3[:, :K, :] + w.draft_logit_noise * eps).reshape(B * K, V).contiguous()
        out["target_logits"] = zp.contiguous()
        draft_logits = zq
    else:
        h = _randn_bf16((B * (K + 1), d), 1.0, g, device)
        W = _randn_bf16((V, d), 1.0 / math.sqrt(d), g, device)
        out["hidden"], out["W"] = h, W
        hk = h.view(B, K + 1, d)[:, :K, :].reshape(B * K, d).float()
        eps = _randn((B * K, d), g, device) if B * K > 0 else torch.zeros((0, d), device=device)
        draft_logits = _project(hk + w.noise * eps, W) if B * K > 0 else \
            torch.zeros((0, V), dtype=torch.float32, device=device)
    if w.greedy:
        out["draft_tokens"] = torch.argmax(draft_logits, dim=-1).to(torch.int32).view(B, K).contiguous()
    else:
        out["draft_logits"] = draft_logits.contiguous()
        if B * K > 0:
            out["draft_tokens"] = gumbel_max_tokens(draft_logits, w.temperature, g).view(B, K).contiguous()
        else:
            out["draft_tokens"] = torch.zeros((B, 0), dtype=torch.int32, device=device)
        out["uniforms"] = torch.rand((B, K + 1), generator=g, device=device, dtype=torch.float32)
    return out


def target_logits(hidden: torch.Tensor, W: torch.Tensor) -> torch.Tensor:
    """fp32 target logits of the given hidden states, computed the way the draft
    logits are (plain fp32 matmul, TF32 off): an input for the steps that take
    logits directly, at the shape of a head workload.  Not the LM head under
    test -- only the generator's own stand-in for a target model's output."""
    return _project(hidden.float(), W)


def fresh_uniforms(B: int, K: int, count: int, device="cpu", seed: int = 99) -> torch.Tensor:
    """``count`` independent sets of uniforms [count, B, K+1] (repeat draws over fixed logits)."""
    g = _gen(torch.device(device), seed)
    return torch.rand((count, B, K + 1), generator=g, device=device, dtype=torch.float32)


# ---------------------------------------------------------------------------
# KV-cache commit inputs.  Paged caches shaped like the models whose heads the
# verify workloads use: an entry is one layer's key and value for one position
# (8 KV heads x 128 dims x 2 (K and V) x bf16 = 4096 bytes).  Committed lengths
# are uniform in [min_len, max_len); the number of accepted drafts is the run
# length of Bernoulli(accept_rate) successes, capped at K (the shape the
# verify step produces for i.i.d. acceptance).  Only the pages the commit can
# touch (the columns covering positions L .. L+S-1) are distinct pool pages,
# in shuffled order; every other block-table column names page 0, which a
# commit of these lengths never writes.
# ---------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class KvWorkload:
    name: str
    B: int
    K: int
    layers: int
    entry_bytes: int
    page_size: int
    min_len: int
    max_len: int
    accept_rate: float
    draft_cache: bool = False   # S = K (a separate draft model's cache) instead of K+1
    seed: int = 0

    @property
    def S(self) -> int:
        return self.K if self.draft_cache else self.K + 1

    @property
    def max_pages(self) -> int:
        return (self.max_len + self.S + self.page_size - 1) // self.page_size


KV_WORKLOADS = {
    w.name: w
    for w in (
        KvWorkload("kv_B8_K4_L32_E4096", B=8, K=4, layers=32, entry_bytes=4096, page_size=16,
                   min_len=512, max_len=4096, accept_rate=0.75, seed=6711),
        KvWorkload("kv_B64_K8_L80_E4096", B=64, K=8, layers=80, entry_bytes=4096, page_size=16,
                   min_len=512, max_len=8192, accept_rate=0.3, seed=6712),
    )
}


def make_kv_inputs(w: KvWorkload, device="cpu", seed: int | None = None, bad_rows: int = 0) -> dict:
    """num_accepted, seq_len, block_table (int32), pool uint8
    [layers][num_pages][page_size][E], staged uint8 [layers][B][S][E].
    ``bad_rows`` sequences get num_accepted = -1 (a row the verify step
    flagged)."""
    g = torch.Generator().manual_seed(w.seed if seed is None else seed)
    B, S, ps = w.B, w.S, w.page_size
    seq_len = torch.randint(w.min_len, w.max_len, (B,), generator=g, dtype=torch.int64)
    succ = torch.rand((B, w.K), generator=g) < w.accept_rate
    n = torch.cumprod(succ.to(torch.int64), dim=1).sum(dim=1)
    if bad_rows:
        n[torch.randperm(B, generator=g)[:bad_rows]] = -1
    cols = [list(range(int(L) // ps, (int(L) + S - 1) // ps + 1)) for L in seq_len]
    num_pages = 1 + sum(len(c) for c in cols)
    perm = (torch.randperm(num_pages - 1, generator=g) + 1).tolist()
    bt = torch.zeros((B, w.max_pages), dtype=torch.int32)
    k = 0
    for b in range(B):
        for c in cols[b]:
            bt[b, c] = perm[k]
            k += 1
    E = w.entry_bytes
    gd = _gen(torch.device(device), (w.seed if seed is None else seed) + 1)
    pool = torch.randint(0, 256, (w.layers, num_pages, ps, E), generator=gd, dtype=torch.uint8,
                         device=device)
    staged = torch.randint(0, 256, (w.layers, B, S, E), generator=gd, dtype=torch.uint8, device=device)
    return dict(num_accepted=n.to(torch.int32).to(device), seq_len=seq_len.to(torch.int32).to(device),
                block_table=bt.to(device), pool=pool, staged=staged)


# ---------------------------------------------------------------------------
# Prompt-lookup drafter inputs: histories shaped like an output rewriting its
# prompt (the case the drafter is meant for).  Each history is a prompt of
# tokens drawn from a Zipf(1.2) law over the vocabulary (common tokens recur,
# as in text and code), followed by an output built from copies of prompt
# spans (start uniform, length geometric with mean 32) with probability 0.85
# and otherwise 1-4 fresh Zipf tokens (the edits).  The prompt is 60% of the
# history; history lengths are uniform in [max_len/2, max_len].
# ---------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class NgramWorkload:
    name: str
    B: int
    max_len: int
    K: int
    n_min: int
    n_max: int
    V: int = 128256
    seed: int = 0


NGRAM_WORKLOADS = {
    w.name: w
    for w in (
        NgramWorkload("ngram_B8_L8192_K4", B=8, max_len=8192, K=4, n_min=1, n_max=3, seed=6721),
        NgramWorkload("ngram_B256_L32768_K8", B=256, max_len=32768, K=8, n_min=1, n_max=3, seed=6722),
    )
}


def _zipf_tokens(n: int, V: int, g: torch.Generator) -> torch.Tensor:
    """n token ids with P(rank r) proportional to r^-1.2, ranks shuffled onto ids."""
    u = torch.rand(n, generator=g, dtype=torch.float64)
    # inverse CDF of the continuous power law on [1, V+1), floored to a rank
    a = 1.2
    lo, hi = 1.0, float(V + 1) ** (1 - a)
    r = ((lo + u * (hi - lo)) ** (1.0 / (1 - a))).floor().clamp(1, V).to(torch.int64) - 1
    return r


def make_ngram_inputs(w: NgramWorkload, device="cpu", seed: int | None = None) -> dict:
    """history int32 [B][max_len] (zero past each length), lengths int32 [B]."""
    g = torch.Generator().manual_seed(w.seed if seed is None else seed)
    perm = torch.randperm(w.V, generator=g)
    hist = torch.zeros((w.B, w.max_len), dtype=torch.int64)
    lens = torch.randint(w.max_len // 2, w.max_len + 1, (w.B,), generator=g)
    for b in range(w.B):
        L = int(lens[b])
        P = max(1, int(0.6 * L))
        prompt = _zipf_tokens(P, w.V, g)
        out = [prompt]
        n = P
        while n < L:
            if float(torch.rand(1, generator=g)) < 0.85:
                # geometric span length, mean 32, by inverse CDF
                span = int(math.floor(math.log(1 - float(torch.rand(1, generator=g))) / math.log(1 - 1 / 32))) + 1
                s = int(torch.randint(0, P, (1,), generator=g))
                piece = prompt[s:s + span]
            else:
                piece = _zipf_tokens(int(torch.randint(1, 5, (1,), generator=g)), w.V, g)
            out.append(piece)
            n += len(piece)
        row = torch.cat(out)[:L]
        hist[b, :L] = perm[row]
    return dict(history=hist.to(torch.int32).to(device), lengths=lens.to(torch.int32).to(device))


# ---------------------------------------------------------------------------
# Drafter that reuses the target's LM head (EAGLE-style): the draft model's
# estimate h-hat of the target's hidden state at slot j is a noisy copy of
# it, h_hat[j][b] = bf16(h[b, j] + noise * eps); the draft logits of slot j
# are h_hat[j] through the same bf16 LM-head weight.  Uniforms: one per
# (draft step, sequence) for the draft draws, and the verify step's [B][K+1].
# ---------------------------------------------------------------------------
DRAFT_WORKLOADS = {
    w.name: w
    for w in (
        Workload("draft_B8_K4_V128256", B=8, K=4, d=4096, V=128256, temperature=0.8, noise=0.3, seed=6731),
        Workload("draft_B64_K4_V128256", B=64, K=4, d=4096, V=128256, temperature=0.8, noise=0.3, seed=6732),
    )
}


def make_draft_inputs(w: Workload, device="cpu", seed: int | None = None) -> dict:
    """hidden bf16 [B*(K+1), d] (target), W bf16 [V, d], draft_hidden bf16
    [K, B, d], draft_uniforms f32 [K, B], uniforms f32 [B, K+1]."""
    device = torch.device(device)
    g = _gen(device, w.seed if seed is None else seed)
    B, K, d, V = w.B, w.K, w.d, w.V
    h = _randn_bf16((B * (K + 1), d), 1.0, g, device)
    W = _randn_bf16((V, d), 1.0 / math.sqrt(d), g, device)
    hk = h.view(B, K + 1, d)[:, :K, :].float().permute(1, 0, 2)          # [K, B, d]
    eps = _randn((K * B, d), g, device).view(K, B, d)
    draft_hidden = (hk + w.noise * eps).to(torch.bfloat16).contiguous()
    draft_uniforms = torch.rand((K, B), generator=g, device=device, dtype=torch.float32)
    uniforms = torch.rand((B, K + 1), generator=g, device=device, dtype=torch.float32)
    return dict(hidden=h, W=W, draft_hidden=draft_hidden, draft_uniforms=draft_uniforms, uniforms=uniforms)


# ---------------------------------------------------------------------------
# Tree-shaped candidates.  A tree of fixed shape per workload: the root has
# branching[0] children, each of those branching[1], and so on; nodes are
# numbered level by level (parents before children).  Every node has a
# target hidden state h ~ N(0, 1) bf16 (one tree-attention target pass) and
# a draft row z_q = (h + noise * eps) W^T in fp32 (the draft model at that
# node); the children of a node are independent draws from softmax(z_q / T)
# (Gumbel-max), the condition of the tree rule's exactness.  Uniforms
# [B][N]: u[b][i] tests node i, u[b][0] is the final draw.
# ---------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class TreeWorkload:
    name: str
    B: int
    branching: tuple
    d: int
    V: int
    temperature: float
    noise: float
    seed: int = 0

    @property
    def N(self) -> int:
        n, width = 1, 1
        for k in self.branching:
            width *= k
            n += width
        return n


TREE_WORKLOADS = {
    w.name: w
    for w in (
        TreeWorkload("tree_B8_N16_V128256", B=8, branching=(3, 2, 1), d=4096, V=128256, temperature=0.8,
                     noise=0.3, seed=6741),
        TreeWorkload("tree_B4_N40_V128256", B=4, branching=(3, 3, 3), d=4096, V=128256, temperature=1.0,
                     noise=0.5, seed=6742),
    )
}


def tree_parents(branching) -> list:
    parents = [-1]
    level = [0]
    for k in branching:
        nxt = []
        for p in level:
            for _ in range(k):
                parents.append(p)
                nxt.append(len(parents) - 1)
        level = nxt
    return parents


def make_tree_inputs(w: TreeWorkload, device="cpu", seed: int | None = None, greedy_drafts: bool = False) -> dict:
    """hidden bf16 [B*N, d], W bf16 [V, d], draft_logits f32 [B*N, V],
    tokens / parents int32 [B, N], uniforms f32 [B, N]."""
    device = torch.device(device)
    g = _gen(device, w.seed if seed is None else seed)
    B, N, d, V = w.B, w.N, w.d, w.V
    h = _randn_bf16((B * N, d), 1.0, g, device)
    W = _randn_bf16((V, d), 1.0 / math.sqrt(d), g, device)
    eps = _randn((B * N, d), g, device)
    zq = _project(h.float() + w.noise * eps, W)
    par = torch.tensor(tree_parents(w.branching), dtype=torch.int32, device=device).repeat(B, 1)
    tok = torch.zeros((B, N), dtype=torch.int32, device=device)
    T = w.temperature if w.temperature > 0 else 1.0
    zq3 = zq.view(B, N, V)
    for i in range(1, N):
        pi = int(par[0, i])
        if greedy_drafts:
            tok[:, i] = torch.argmax(zq3[:, pi, :], dim=-1).to(torch.int32)
        else:
            tok[:, i] = gumbel_max_tokens(zq3[:, pi, :], T, g)
    u = torch.rand((B, N), generator=g, device=device, dtype=torch.float32)
    return dict(hidden=h, W=W, draft_logits=zq.contiguous(), tokens=tok, parents=par, uniforms=u)
