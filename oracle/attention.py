"""Tree verification attention (oracle).

Test infrastructure only (see ``oracle/__init__.py``).

N packed tree rows attend to P committed prefix keys plus the tree block
under the ancestor-or-self mask, with RoPE applied at logical positions
P + depth(u) ([M7.2] §0x03, §0x03A, §0x03C; [CN] "Tree Attention";
[Math] "Tree attention: the mask math").  Scores are scaled by 1/sqrt(dh).

RoPE convention (the pages name RoPE but not its layout): rotate-half pairs
(i, i + dh/2) with angle pos * base^(-2i/dh).  The committed prefix K in the
cache is already rotated; tree queries and keys arrive unrotated.
"""
from __future__ import annotations

import math

import numpy as np


def rope(x: np.ndarray, pos, base: float = 10000.0) -> np.ndarray:
    """Rotate-half RoPE of x[..., dh] at integer positions `pos` (broadcast over x[..., 0])."""
    x = np.asarray(x, dtype=np.float64)
    dh = x.shape[-1]
    half = dh // 2
    inv_freq = np.array([base ** (-2.0 * i / dh) for i in range(half)], dtype=np.float64)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * inv_freq
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def _softmax_attend(qv: np.ndarray, keys: np.ndarray, values: np.ndarray, scale: float):
    """softmax(q . K^T * scale) V for one query vector; also returns the log-sum-exp."""
    s = keys @ qv * scale
    m = s.max()
    e = np.exp(s - m)
    z = e.sum()
    return (e @ values) / z, m + math.log(z)


def visibility(L: int, mask) -> np.ndarray:
    """Rectangular visibility A[u, j] of N tree queries over P + N keys ([M7.2] §0x03C):
    every committed prefix key is visible, the tree block is the ancestor mask."""
    mask = np.asarray(mask, dtype=bool)
    return np.concatenate([np.ones((mask.shape[0], L), dtype=bool), mask], axis=1)


def tree_attention(q, k_new, v_new, prefix_k, prefix_v, L: int, depth, mask,
                   base: float = 10000.0, scale: float | None = None):
    """Dense rectangular masked attention for one sequence ([M7.2] §0x03C).

    q [N, Hq, dh]; k_new, v_new [N, Hkv, dh] (unrotated tree rows);
    prefix_k, prefix_v [Hkv, L, dh] (prefix K already rotated); depth [N]; mask [N, N].
    Returns (out [N, Hq, dh], lse [N, Hq], staged_k [N, Hkv, dh]) where staged_k
    is the rotated tree K written at cache rows L + u.
    """
    q = np.asarray(q, dtype=np.float64)
    k_new = np.asarray(k_new, dtype=np.float64)
    v_new = np.asarray(v_new, dtype=np.float64)
    pk = np.asarray(prefix_k, dtype=np.float64)[:, :L]
    pv = np.asarray(prefix_v, dtype=np.float64)[:, :L]
    N, Hq, dh = q.shape
    Hkv = k_new.shape[1]
    g = Hq // Hkv
    scale = 1.0 / math.sqrt(dh) if scale is None else scale
    pos = L + np.asarray(depth, dtype=np.int64)
    qr = rope(q, pos[:, None], base)
    kr = rope(k_new, pos[:, None], base)

    vis = visibility(L, mask)
    out = np.zeros((N, Hq, dh))
    lse = np.zeros((N, Hq))
    for h in range(Hq):
        kv = h // g
        keys = np.concatenate([pk[kv], kr[:, kv]], axis=0)      # [L+N, dh]
        vals = np.concatenate([pv[kv], v_new[:, kv]], axis=0)
        s = (qr[:, h] @ keys.T) * scale                        # [N, L+N]
        s = np.where(vis, s, -np.inf)
        m = s.max(axis=1, keepdims=True)
        e = np.exp(s - m)
        z = e.sum(axis=1, keepdims=True)
        out[:, h] = (e @ vals) / z
        lse[:, h] = (m + np.log(z))[:, 0]
    return out, lse, kr


def path_attention(q, k_new, v_new, prefix_k, prefix_v, L: int, parent, u: int, h: int,
                   base: float = 10000.0, scale: float | None = None):
    """Brute force for node u and query head h: plain causal attention of u over
    the prefix followed by u's own root-to-node path, as if that path were the
    only continuation ([CN] "Tree Attention"; [CN] "Mask、位置和 KV 必须一起验证").

    Uses only the parent chain, not the mask or the depth array; positions are
    the path's own sequence positions L, L+1, ...
    """
    q = np.asarray(q, dtype=np.float64)
    k_new = np.asarray(k_new, dtype=np.float64)
    v_new = np.asarray(v_new, dtype=np.float64)
    Hq, dh = q.shape[1], q.shape[2]
    g = Hq // k_new.shape[1]
    kv = h // g
    scale = 1.0 / math.sqrt(dh) if scale is None else scale
    chain = []
    node = u
    while node >= 0:
        chain.append(node)
        node = int(parent[node])
    chain.reverse()                       # root ... u
    keys = [np.asarray(prefix_k, dtype=np.float64)[kv, :L]]
    vals = [np.asarray(prefix_v, dtype=np.float64)[kv, :L]]
    for t, node in enumerate(chain):
        keys.append(rope(k_new[node, kv][None, :], np.array([L + t]), base))
        vals.append(v_new[node, kv][None, :])
    keys = np.concatenate(keys, axis=0)
    vals = np.concatenate(vals, axis=0)
    qv = rope(q[u, h][None, :], np.array([L + len(chain) - 1]), base)[0]
    out, _ = _softmax_attend(qv, keys, vals, scale)
    return out


def single_query_attention(qv, keys, values, scale):
    """Textbook attention of one (already rotated) query over explicit keys/values."""
    return _softmax_attend(np.asarray(qv, np.float64), np.asarray(keys, np.float64),
                           np.asarray(values, np.float64), scale)[0]


def node_attention_rows(q_uh, k_tree, v_tree, prefix_k_h, prefix_v_h, L: int, depth, mask_row,
                        u: int, base: float = 10000.0, scale: float | None = None):
    """Output and log-sum-exp of node u for one query head.

    q_uh [dh] unrotated query of (u, h); k_tree, v_tree [N, dh] unrotated tree keys
    and values of that head's KV group; prefix_k_h, prefix_v_h [L, dh];
    depth [N]; mask_row [N] bool (mask[u, :]).
    """
    q_uh = np.asarray(q_uh, dtype=np.float64)
    dh = q_uh.shape[0]
    scale = 1.0 / math.sqrt(dh) if scale is None else scale
    depth = np.asarray(depth, dtype=np.int64)
    vis = np.nonzero(np.asarray(mask_row, dtype=bool))[0]
    qr = rope(q_uh[None, :], np.array([L + depth[u]]), base)[0]
    kt = rope(np.asarray(k_tree, np.float64)[vis], L + depth[vis], base)
    keys = np.concatenate([np.asarray(prefix_k_h, np.float64)[:L], kt], axis=0)
    vals = np.concatenate([np.asarray(prefix_v_h, np.float64)[:L],
                           np.asarray(v_tree, np.float64)[vis]], axis=0)
    return _softmax_attend(qr, keys, vals, scale)
