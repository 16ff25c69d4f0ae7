"""Medusa heads, root selection and per-head top-k pools (oracle).

Test infrastructure only (see ``oracle/__init__.py``).

Head k reads the frontier hidden state h and computes
    z_k = h + SiLU(W1_k h [+ b1_k]),   logits_k = W2_k z_k
([CN] "Medusa 的核心思路与系统位置"; [Math] "The Medusa head: math and shapes";
[M7.2] §0x02A with one residual block).  The root is the argmax of the ordinary
LM head W_LM h ([M7.2] §0x04D).  Each head contributes the TOPK highest-scoring
token ids as its candidate pool ([PartII] Part 4).  All arithmetic in float64.
"""
from __future__ import annotations

import numpy as np


def silu(x: np.ndarray) -> np.ndarray:
    """SiLU(x) = x * sigmoid(x) = x / (1 + e^-x)."""
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-x))


def ranked_ids(values: np.ndarray, k: int) -> np.ndarray:
    """Ids of the k largest entries of a 1-D vector, by value descending, ties to the lower id."""
    v = np.asarray(values, dtype=np.float64)
    ids = np.arange(v.shape[0])
    order = np.lexsort((ids, -v))   # primary key -v, secondary key id
    return order[:k]


def residual(h: np.ndarray, w1: np.ndarray, b1: np.ndarray | None = None) -> np.ndarray:
    """z[t, k, :] = h[t] + SiLU(W1[k] h[t] + b1[k]) for every row t and head k."""
    h = np.asarray(h, dtype=np.float64)
    w1 = np.asarray(w1, dtype=np.float64)
    pre = np.einsum("kij,tj->tki", w1, h)
    if b1 is not None:
        pre = pre + np.asarray(b1, dtype=np.float64)[None, :, :]
    return h[:, None, :] + silu(pre)


def head_logits(z: np.ndarray, w2: np.ndarray) -> np.ndarray:
    """logits[t, k, :] = W2[k] z[t, k].  A 2-D w2 is one matrix shared by every head."""
    z = np.asarray(z, dtype=np.float64)
    w2 = np.asarray(w2, dtype=np.float64)
    if w2.ndim == 2:
        return np.einsum("vj,tkj->tkv", w2, z)
    return np.einsum("kvj,tkj->tkv", w2, z)


def medusa_heads(h, w1, w2, w_lm, topk: int, b1=None):
    """One proposal step on T frontier rows.

    h [T, d]; w1 [K, d, d]; w2 [K, V, d] or shared [V, d]; w_lm [V, d].
    Returns (root [T], pool [T, K, topk], logits [T, K+1, V]) where logits[:, 0]
    are the LM-head logits and logits[:, 1+k] head k's logits.
    """
    h = np.asarray(h, dtype=np.float64)
    lm = h @ np.asarray(w_lm, dtype=np.float64).T
    z = residual(h, w1, b1)
    hl = head_logits(z, w2)
    T, K, V = hl.shape
    root = np.array([ranked_ids(lm[t], 1)[0] for t in range(T)], dtype=np.int64)
    pool = np.zeros((T, K, topk), dtype=np.int64)
    for t in range(T):
        for k in range(K):
            pool[t, k] = ranked_ids(hl[t, k], topk)
    logits = np.concatenate([lm[:, None, :], hl], axis=1)
    return root, pool, logits


def head_logit_rows(h_t, w1_head, w2_row, lm_row, rows, b1_head=None):
    """Selected logits of one frontier row, for sampled checks at full size.

    rows: list of (m, v) with m = 0 for the LM head or 1 + k for Medusa head k.
    Weights are fetched through accessors so that only the touched ones are read:
    w1_head(k) -> [d, d], w2_row(k, v) -> [d], lm_row(v) -> [d], b1_head(k) -> [d].
    """
    h_t = np.asarray(h_t, dtype=np.float64)
    out = np.zeros(len(rows), dtype=np.float64)
    z_cache = {}
    for i, (m, v) in enumerate(rows):
        if m == 0:
            out[i] = float(np.asarray(lm_row(v), dtype=np.float64) @ h_t)
            continue
        k = m - 1
        if k not in z_cache:
            pre = np.asarray(w1_head(k), dtype=np.float64) @ h_t
            if b1_head is not None:
                pre = pre + np.asarray(b1_head(k), dtype=np.float64)
            z_cache[k] = h_t + silu(pre)
        out[i] = float(np.asarray(w2_row(k, v), dtype=np.float64) @ z_cache[k])
    return out
