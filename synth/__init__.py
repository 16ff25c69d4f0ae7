"""Seeded synthetic inputs for the Medusa verify round.

This module is the only code shared by the fp64 oracle and the CUDA path.  It
draws random tensors and holds the five workload shapes; it contains none of
the method's arithmetic (no heads, tree compilation, attention, acceptance or
compaction).  Random numbers that the method would consume are drawn here and
passed in as plain inputs.

Every tensor is drawn from its own ``torch.Generator`` seeded from the workload
seed and a fixed per-tensor tag, so any subset can be regenerated on any device
without drawing the others.  Values are drawn in fp32 and then rounded to the
workload dtype; both consumers see the rounded values.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

# --------------------------------------------------------------------------- #
# Workload shapes
# --------------------------------------------------------------------------- #


@dataclass(frozen=True)
class Workload:
    """Shapes of one synthetic verify round.

    template: ("regular", widths) or ("greedy", budget, ranks).
    """

    name: str
    seed: int
    batch: int
    template: tuple
    topk: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    prefix_len: Optional[int]          # fixed L, or None for a drawn range
    prefix_range: Optional[tuple]      # (lo, hi) inclusive, drawn per sequence
    n_heads: int                       # Medusa heads K
    hidden: int                        # d
    vocab: int                         # V
    dtype: str                         # "f32" or "bf16"
    accept: tuple                      # acceptance policies exercised
    page_size: int = 0                 # 0 = contiguous cache
    plant: bool = True                 # plant target argmax on candidates
    rope_base: float = 10000.0
    epsilon: float = 0.09
    delta: float = 0.3

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


WORKLOADS = {
    "tiny-fp32": Workload(
        name="tiny-fp32", seed=1001, batch=1, template=("regular", (2, 3)), topk=3,
        n_q_heads=4, n_kv_heads=4, head_dim=64, prefix_len=64, prefix_range=None,
        n_heads=2, hidden=256, vocab=1000, dtype="f32", accept=("greedy",), plant=False),
    "vicuna7b-64": Workload(
        name="vicuna7b-64", seed=1002, batch=1, template=("greedy", 63, 10), topk=10,
        n_q_heads=32, n_kv_heads=32, head_dim=128, prefix_len=2048, prefix_range=None,
        n_heads=4, hidden=4096, vocab=32000, dtype="bf16", accept=("greedy", "typical")),
    "llama3-8b-256": Workload(
        name="llama3-8b-256", seed=1003, batch=1, template=("greedy", 255, 10), topk=10,
        n_q_heads=32, n_kv_heads=8, head_dim=128, prefix_len=4096, prefix_range=None,
        n_heads=4, hidden=4096, vocab=128256, dtype="bf16", accept=("greedy", "typical")),
    "serving-b16-paged": Workload(
        name="serving-b16-paged", seed=1004, batch=16, template=("greedy", 63, 10), topk=10,
        n_q_heads=32, n_kv_heads=8, head_dim=128, prefix_len=None, prefix_range=(512, 8192),
        n_heads=4, hidden=4096, vocab=32000, dtype="bf16", accept=("greedy",), page_size=16),
    "longctx-341": Workload(
        name="longctx-341", seed=1005, batch=1, template=("regular", (4, 4, 4, 4)), topk=4,
        n_q_heads=64, n_kv_heads=8, head_dim=128, prefix_len=32768, prefix_range=None,
        n_heads=4, hidden=8192, vocab=128256, dtype="bf16", accept=("typical",)),
}
WORKLOAD_ORDER = ["tiny-fp32", "vicuna7b-64", "llama3-8b-256", "serving-b16-paged", "longctx-341"]


def rank_accuracy(n_heads: int, n_ranks: int) -> np.ndarray:
    """Synthetic exact-rank accuracies a_k^(i) = 0.7 * 0.6^(k-1) * 0.45^(i-1).

    Returned 0-based as acc[k, i] (head k, rank i) in float64.  Each entry is
    built by repeated multiplication so that every consumer sees the same doubles.
    """
    acc = np.empty((n_heads, n_ranks), dtype=np.float64)
    head_factor = 0.7
    for k in range(n_heads):
        rank_factor = head_factor
        for i in range(n_ranks):
            acc[k, i] = rank_factor
            rank_factor = rank_factor * 0.45
        head_factor = head_factor * 0.6
    return acc


# --------------------------------------------------------------------------- #
# Random tensors
# --------------------------------------------------------------------------- #

_TAGS = {
    "h": 1, "w1": 2, "w2": 3, "w_lm": 4, "q": 5, "k_new": 6, "v_new": 7,
    "cache_k": 8, "cache_v": 9, "logits": 10, "lengths": 11, "pages": 12,
    "plant": 13, "b1": 14, "misc": 15,
}


def generator(seed: int, tag: str, device="cpu", sub: int = 0) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000003 + _TAGS[tag] * 1009 + sub)
    return g


def normal(shape, std: float, seed: int, tag: str, device="cpu", dtype=torch.float32,
           sub: int = 0) -> torch.Tensor:
    """N(0, std^2) drawn in fp32 on `device`, then rounded to `dtype`."""
    g = generator(seed, tag, device, sub)
    x = torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def uniform(shape, seed: int, tag: str, device="cpu", sub: int = 0) -> torch.Tensor:
    g = generator(seed, tag, device, sub)
    return torch.rand(tuple(shape), generator=g, device=device, dtype=torch.float64)


def prefix_lengths(w: Workload) -> np.ndarray:
    """Committed prefix length per sequence (int64, host)."""
    if w.prefix_len is not None:
        return np.full(w.batch, w.prefix_len, dtype=np.int64)
    lo, hi = w.prefix_range
    g = generator(w.seed, "lengths")
    return torch.randint(lo, hi + 1, (w.batch,), generator=g).numpy().astype(np.int64)


@dataclass
class PagedLayout:
    """Page table for a paged cache: block_table[b, j] = physical page of rows [16j, 16j+16)."""

    page_size: int
    n_pages: int
    block_table: np.ndarray   # int64 [B, max_blocks], -1 where unused


def paged_layout(w: Workload, lengths: np.ndarray, n_rows: int, guard: int = 16) -> PagedLayout:
    """Shuffled page assignment: each sequence owns ceil((L_b + N + guard)/ps) pages."""
    ps = w.page_size
    need = [int(math.ceil((int(L) + n_rows + guard) / ps)) for L in lengths]
    total = sum(need)
    g = generator(w.seed, "pages")
    perm = torch.randperm(total, generator=g).numpy().astype(np.int64)
    maxb = max(need)
    table = np.full((w.batch, maxb), -1, dtype=np.int64)
    off = 0
    for b, nb in enumerate(need):
        table[b, :nb] = perm[off:off + nb]
        off += nb
    return PagedLayout(page_size=ps, n_pages=total, block_table=table)


def head_weights(w: Workload, device="cpu", dtype=None):
    """h [B, d], W1 [K, d, d] ~ N(0, 0.02^2), W2 [K, V, d] ~ N(0, 1/d), W_LM [V, d] ~ N(0, 1/d)."""
    dt = dtype or w.torch_dtype
    d, V, K = w.hidden, w.vocab, w.n_heads
    h = normal((w.batch, d), 1.0, w.seed, "h", device, dt)
    w1 = normal((K, d, d), 0.02, w.seed, "w1", device, dt)
    w2 = torch.empty((K, V, d), device=device, dtype=dt)
    for k in range(K):
        w2[k] = normal((V, d), 1.0 / math.sqrt(d), w.seed, "w2", device, dt, sub=k)
    w_lm = normal((V, d), 1.0 / math.sqrt(d), w.seed, "w_lm", device, dt)
    return h, w1, w2, w_lm


def tree_qkv(w: Workload, n_rows: int, device="cpu", dtype=None):
    """Tree-row queries/keys/values before RoPE: q [B,N,Hq,dh], k/v [B,N,Hkv,dh] ~ N(0,1)."""
    dt = dtype or w.torch_dtype
    B, dh = w.batch, w.head_dim
    q = normal((B, n_rows, w.n_q_heads, dh), 1.0, w.seed, "q", device, dt)
    k = normal((B, n_rows, w.n_kv_heads, dh), 1.0, w.seed, "k_new", device, dt)
    v = normal((B, n_rows, w.n_kv_heads, dh), 1.0, w.seed, "v_new", device, dt)
    return q, k, v


def prefix_kv(w: Workload, lengths: np.ndarray, device="cpu", dtype=None):
    """Committed prefix K (already rotated) and V per sequence: list of [Hkv, L_b, dh] ~ N(0,1)."""
    dt = dtype or w.torch_dtype
    ks, vs = [], []
    for b, L in enumerate(lengths):
        ks.append(normal((w.n_kv_heads, int(L), w.head_dim), 1.0, w.seed, "cache_k", device, dt, sub=b))
        vs.append(normal((w.n_kv_heads, int(L), w.head_dim), 1.0, w.seed, "cache_v", device, dt, sub=b))
    return ks, vs


def target_logits(w: Workload, n_rows: int, device="cpu", dtype=None, sub: int = 0):
    """Target verification logits [B, N, V] ~ N(0,1) before any planting."""
    dt = dtype or w.torch_dtype
    return normal((w.batch, n_rows, w.vocab), 1.0, w.seed, "logits", device, dt, sub=sub)


def plant_uniforms(w: Workload, n_rows: int, sub: int = 0) -> np.ndarray:
    """U(0,1) per (sequence, tree row) used to pick the planted rank."""
    return uniform((w.batch, n_rows), w.seed, "plant", sub=sub).numpy()


def plant_argmax(logits: torch.Tensor, pool: np.ndarray, row_depth: np.ndarray,
                 acc: np.ndarray, u01: np.ndarray) -> torch.Tensor:
    """Plant the argmax of target row u on a head candidate.

    For row u at depth t (t < K) the candidate for depth t+1 comes from head t.
    Rank i (0-based) is chosen as the first i whose running sum of acc[t, :i+1]
    exceeds u01[b, u]; the logit of pool[b, t, i] is then set to rowmax + 1.
    Rows whose draw exceeds every running sum are left unplanted.

    logits: [B, N, V] tensor (modified in place and returned), pool: [B, K, R] ids,
    row_depth: [N] depths, acc: [K, R'] accuracies, u01: [B, N].
    """
    B, N, V = logits.shape
    K, R = pool.shape[1], pool.shape[2]
    host = logits.detach().to("cpu", torch.float32)
    rowmax = host.max(dim=-1).values
    for b in range(B):
        for u in range(N):
            t = int(row_depth[u])
            if t >= K:
                continue
            run = 0.0
            for i in range(min(R, acc.shape[1])):
                run = run + float(acc[t, i])
                if u01[b, u] < run:
                    tok = int(pool[b, t, i])
                    val = float(rowmax[b, u]) + 1.0
                    logits[b, u, tok] = torch.tensor(val, dtype=logits.dtype)
                    break
    return logits


def random_pool(w: Workload, seed_sub: int = 0):
    """Seeded stand-in for the heads' output: root [B] and per-head candidate pools
    [B, K, topk] of distinct token ids (int64, host)."""
    g = generator(w.seed, "misc", sub=100 + seed_sub)
    root = torch.randint(0, w.vocab, (w.batch,), generator=g).numpy().astype(np.int64)
    pool = np.zeros((w.batch, w.n_heads, w.topk), dtype=np.int64)
    for b in range(w.batch):
        for k in range(w.n_heads):
            pool[b, k] = torch.randperm(w.vocab, generator=g)[:w.topk].numpy()
    return root, pool


def small_variant(w: Workload, **kw) -> Workload:
    """A copy of a workload with some fields replaced (for scaled-down parity cases)."""
    from dataclasses import replace
    return replace(w, **kw)
