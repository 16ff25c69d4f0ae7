"""Greedy and fast-typical acceptance over the packed tree (oracle).

Test infrastructure only (see ``oracle/__init__.py``).

Target logits of packed row u score the successor of u's token: along a
retrieval path [u_0, u_1, ...] the candidate token of u_{j+1} is judged by
row u_j ([M7.2] §0x03D; [PartII] Part 7).

  greedy   edge j passes iff tok(u_{j+1}) == argmax of row u_j
           ([M7.2] §0x04D; ties in the argmax go to the lowest token id)
  typical  edge j passes iff p_{u_j}(tok(u_{j+1})) > min(eps, delta * exp(-H(p_{u_j})))
           with p = softmax(logits / T) and H the entropy
           ([M7.2] §0x04E; [CN] "接受机制"; [Math] "Typical acceptance, not exact match")

A path's accepted length a_p counts the edges before its first failing edge.
The winner is the path of largest a_p; greedy keeps the first such path in
retrieval order (path 0 when nothing passes); typical breaks length ties by
the largest accepted log-likelihood sum_{j<a} log p, then by the lowest path
index.  G = a + 1 tokens (root included) are published ([M7.2] §0x06A).

Everything is evaluated once per unique packed row, not per gathered path
position ([M7.2] §0x07B notes both give the same decisions).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np


@dataclass
class RowStats:
    argmax: int
    m: float        # max of logits / T
    log_z: float    # log sum exp(logits / T - m)
    entropy: float  # H of softmax(logits / T)


def row_stats(logits_row, temperature: float = 1.0, entropy_guard: bool = False) -> RowStats:
    """Argmax, log-partition and entropy of one target row in float64.

    With entropy_guard the entropy is -sum p log(p + 1e-5), the guarded form the
    pinned implementation uses ([M7.2] §0x04E); otherwise the exact entropy.
    """
    x = np.asarray(logits_row, dtype=np.float64) / float(temperature)
    am = int(np.flatnonzero(x == x.max())[0])        # lowest id among maxima
    m = float(x.max())
    e = np.exp(x - m)
    z = float(e.sum())
    p = e / z
    if entropy_guard:
        h = float(-(p * np.log(p + 1e-5)).sum())
    else:
        nz = p > 0
        h = float(-(p[nz] * np.log(p[nz])).sum())
    return RowStats(argmax=am, m=m, log_z=math.log(z), entropy=h)


def log_prob(logits_row, tok: int, st: RowStats, temperature: float = 1.0) -> float:
    return float(np.float64(logits_row[tok]) / temperature - st.m - st.log_z)


def edge_score(lp: float) -> float:
    """Contribution of one accepted edge to the typical tie-break: its log-probability,
    so that comparing sums compares products of probabilities ([M7.2] §0x04E)."""
    return lp


@dataclass
class AcceptResult:
    best_path: int
    accept_len: int                 # a: accepted suffix edges
    out_rows: np.ndarray            # [G] packed rows u_0..u_a
    out_tokens: np.ndarray          # [G] tokens on those rows
    frontier_row: int               # u_a: row whose logits start the next round
    per_path_len: np.ndarray        # a_p for every path
    per_path_score: np.ndarray      # sum of accepted log p (typical), 0 for greedy
    margins: list                   # (|p - tau| / tau) of every typical decision taken


def accept(logits, tokens, retrieve, mode: str = "greedy", temperature: float = 1.0,
           epsilon: float = 0.09, delta: float = 0.3, entropy_guard: bool = False) -> AcceptResult:
    """Acceptance for one sequence.

    logits [N, V]; tokens [N] (token fed into each packed row); retrieve [n_paths, D+1]
    with -1 padding.  mode is "greedy" or "typical".
    """
    logits = np.asarray(logits)
    tokens = np.asarray(tokens, dtype=np.int64)
    retrieve = np.asarray(retrieve, dtype=np.int64)
    stats = {}

    def stat(u):
        if u not in stats:
            stats[u] = row_stats(logits[u], temperature, entropy_guard)
        return stats[u]

    n_paths = retrieve.shape[0]
    lens = np.zeros(n_paths, dtype=np.int64)
    scores = np.zeros(n_paths, dtype=np.float64)
    margins = []
    for pi in range(n_paths):
        nodes = [int(u) for u in retrieve[pi] if u >= 0]
        a, score = 0, 0.0
        for j in range(len(nodes) - 1):
            u, child = nodes[j], nodes[j + 1]
            tok = int(tokens[child])
            st = stat(u)
            if mode == "greedy":
                ok = tok == st.argmax
            elif mode == "typical":
                lp = log_prob(logits[u], tok, st, temperature)
                p = math.exp(lp)
                tau = min(epsilon, delta * math.exp(-st.entropy))
                margins.append(abs(p - tau) / tau)
                ok = p > tau
                if ok:
                    score += edge_score(lp)
            else:
                raise ValueError(mode)
            if not ok:
                break
            a += 1
        lens[pi] = a
        scores[pi] = score

    best_len = int(lens.max())
    if mode == "greedy":
        best = int(np.flatnonzero(lens == best_len)[0])
    else:
        best = None
        for pi in range(n_paths):
            if lens[pi] != best_len:
                continue
            if best is None or scores[pi] > scores[best]:
                best = pi
    rows = np.array([int(u) for u in retrieve[best][:best_len + 1]], dtype=np.int64)
    return AcceptResult(best_path=best, accept_len=best_len, out_rows=rows,
                        out_tokens=tokens[rows], frontier_row=int(rows[-1]),
                        per_path_len=lens, per_path_score=scores, margins=margins)


def target_logits(hidden, w_lm, rows=None) -> np.ndarray:
    """The target's vocabulary projection of the tree rows, logits[u] = W_LM hidden[u],
    in float64 ([M7.2] §0x07B: C_LMproj(N) with F_LMproj = 2 N d V; §0x07C: dense
    target logits hold N V elements).  Only `rows` are computed (default: every row);
    the others are NaN, since acceptance reads internal rows only.

    hidden [N, d]; w_lm [V, d].
    """
    h = np.asarray(hidden, dtype=np.float64)
    w = np.asarray(w_lm, dtype=np.float64)
    out = np.full((h.shape[0], w.shape[0]), np.nan)
    for u in (range(h.shape[0]) if rows is None else rows):
        out[int(u)] = w @ h[int(u)]
    return out


def accept_hidden(hidden, w_lm, tokens, retrieve, internal, mode: str = "greedy", temperature: float = 1.0,
                  epsilon: float = 0.09, delta: float = 0.3) -> AcceptResult:
    """Acceptance with the target's vocabulary projection folded in: the projection of
    every internal row (`internal`: rows with children), then `accept` on those rows.
    Leaves are never projected; no other row is read by acceptance ([M7.2] §0x07B:
    a unique-row posterior instead of gathered path logits)."""
    logits = target_logits(hidden, w_lm, internal)
    return accept(logits, tokens, retrieve, mode, temperature, epsilon, delta)
