"""One whole verify round, composed from the five oracle steps.

Test infrastructure only (see ``oracle/__init__.py``).

Round order ([M7.2] §0x07A; [CN] "一次完整解码迭代"; [PartII] Part 1):
heads + top-k  ->  tree fill  ->  tree attention (stages K/V at rows L + u)
->  acceptance  ->  winning-path K/V compaction.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import accept as acc_mod
from . import attention, compact, heads, tree


def template_for(spec, topk: int, n_heads: int, acc=None) -> tree.Template:
    """Compile a workload's template spec: ("regular", widths) or ("greedy", budget, ranks)."""
    kind = spec[0]
    if kind == "regular":
        return tree.compile_template(tree.regular_paths(spec[1]), topk, n_heads)
    if kind == "greedy":
        budget, ranks = spec[1], spec[2]
        if acc is None:
            raise ValueError("greedy template needs rank accuracies")
        return tree.compile_template(tree.greedy_tree(acc[:, :ranks], budget), topk, n_heads)
    raise ValueError(kind)


def tree_fill(tmpl: tree.Template, root: int, pool: np.ndarray, L: int):
    """tokens[u] = cand[slot[u]] with cand = [root, pool[0, :], pool[1, :], ...];
    pos[u] = L + depth[u] ([M7.2] §0x01B, §0x04A "Candidate gather", "Visibility and position")."""
    cand = np.concatenate([[int(root)], np.asarray(pool, dtype=np.int64).reshape(-1)])
    tokens = cand[tmpl.slot]
    pos = int(L) + tmpl.depth
    return tokens.astype(np.int64), pos.astype(np.int64)


@dataclass
class RoundResult:
    root: int
    pool: np.ndarray
    head_logits: np.ndarray
    tokens: np.ndarray
    pos: np.ndarray
    attn_out: np.ndarray
    attn_lse: np.ndarray
    staged_k: np.ndarray
    accept: acc_mod.AcceptResult
    new_len: int


def run_sequence(tmpl, h_t, w1, w2, w_lm, q, k_new, v_new, cache_k, cache_v, L, logits,
                 mode="greedy", base=10000.0, temperature=1.0, epsilon=0.09, delta=0.3,
                 entropy_guard=False, b1=None) -> RoundResult:
    """Full round for one sequence.  cache_k/cache_v [Hkv, cap, dh] float64 are mutated
    (staged tree rows, then compaction)."""
    root, pool, hl = heads.medusa_heads(np.asarray(h_t)[None, :], w1, w2, w_lm, tmpl.topk, b1)
    root, pool = int(root[0]), pool[0]
    tokens, pos = tree_fill(tmpl, root, pool, L)
    out, lse, kr = attention.tree_attention(q, k_new, v_new, cache_k, cache_v, L,
                                            tmpl.depth, tmpl.mask, base)
    N = tmpl.n_rows
    cache_k[:, L:L + N, :] = np.transpose(kr, (1, 0, 2))
    cache_v[:, L:L + N, :] = np.transpose(np.asarray(v_new, np.float64), (1, 0, 2))
    res = acc_mod.accept(logits, tokens, tmpl.retrieve, mode, temperature, epsilon, delta,
                         entropy_guard)
    new_len = compact.kv_compact(cache_k, cache_v, L, res.out_rows)
    return RoundResult(root=root, pool=pool, head_logits=hl[0], tokens=tokens, pos=pos,
                       attn_out=out, attn_lse=lse, staged_k=kr, accept=res, new_len=new_len)
