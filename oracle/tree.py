"""Rank-path tree templates (oracle).

Test infrastructure only (see ``oracle/__init__.py``).

A template is a prefix-closed set of rank paths.  Path (r_1, ..., r_t) means
"rank r_1 of head 0 at depth 1, ..., rank r_t of head t-1 at depth t"
([M7.2] §0x00D, §0x04A; [PartII] Part 5).  The empty path is the LM-head root.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


class TemplateError(ValueError):
    pass


@dataclass
class Template:
    """The four coupled buffers of [M7.2] §0x04A plus the derived structure.

    rows are numbered in canonical order: row(()) = 0, row(p) = 1 + index of p
    in the non-root paths sorted by (len(p), p).
    """

    paths: list            # all paths by row, paths[0] == ()
    topk: int              # pool width TOPK used by the slot formula
    depth: np.ndarray      # [N] int64, len(path)
    parent: np.ndarray     # [N] int64, row of path[:-1]; -1 for the root
    slot: np.ndarray       # [N] int64, tree_indices: 0 for the root, 1 + (t-1)*TOPK + r_t
    mask: np.ndarray       # [N, N] bool, mask[u, v] = path(v) is a prefix of path(u)
    retrieve: np.ndarray   # [n_paths, D+1] int64, maximal paths as row chains, -1 padded

    @property
    def n_rows(self) -> int:
        return len(self.paths)

    @property
    def max_depth(self) -> int:
        return int(self.depth.max())

    @property
    def n_paths(self) -> int:
        return int(self.retrieve.shape[0])

    def row_of(self, path) -> int:
        return self.paths.index(tuple(path))


def _is_prefix(a: tuple, b: tuple) -> bool:
    """True when a is a prefix of b (a == b counts)."""
    return len(a) <= len(b) and b[:len(a)] == a


def compile_template(paths, topk: int, n_heads: int | None = None) -> Template:
    """Compile a rank-path family into the tree buffers ([M7.2] §0x04A).

    Rejects duplicates, ranks outside [0, topk), paths deeper than n_heads and
    families that are not prefix-closed.
    """
    given = [tuple(int(r) for r in p) for p in paths]
    if len(set(given)) != len(given):
        raise TemplateError("duplicate path")
    for p in given:
        if len(p) == 0:
            raise TemplateError("the empty path is the implicit root")
        if any(r < 0 or r >= topk for r in p):
            raise TemplateError(f"rank outside [0, {topk}) in {p}")
        if n_heads is not None and len(p) > n_heads:
            raise TemplateError(f"path {p} deeper than {n_heads} heads")
    present = set(given)
    for p in given:
        if len(p) > 1 and p[:-1] not in present:
            raise TemplateError(f"not prefix-closed: {p} without {p[:-1]}")

    # Canonical order: by length, then lexicographically ([M7.2] §0x04A "Canonical row map").
    ordered = [()] + sorted(given, key=lambda p: (len(p), p))
    row = {p: i for i, p in enumerate(ordered)}
    n = len(ordered)

    depth = np.array([len(p) for p in ordered], dtype=np.int64)
    parent = np.array([-1] + [row[p[:-1]] for p in ordered[1:]], dtype=np.int64)
    # tree_indices: head t-1 rank r_t lands in slot 1 + (t-1)*TOPK + r_t; slot 0 is the root.
    slot = np.array([0] + [1 + (len(p) - 1) * topk + p[-1] for p in ordered[1:]], dtype=np.int64)

    # Visibility by the literal prefix test M[u, v] = 1[p_v is a prefix of p_u].
    mask = np.zeros((n, n), dtype=bool)
    for u in range(n):
        for v in range(n):
            mask[u, v] = _is_prefix(ordered[v], ordered[u])

    # Retrieval rows: one per maximal path, in canonical order, padded with -1
    # ([M7.2] §0x04A "Retrieval paths and sentinels").
    maximal = [p for p in ordered
               if not any(len(q) > len(p) and _is_prefix(p, q) for q in ordered)]
    width = int(depth.max()) + 1
    retrieve = np.full((len(maximal), width), -1, dtype=np.int64)
    for i, p in enumerate(maximal):
        for t in range(len(p) + 1):
            retrieve[i, t] = row[p[:t]]

    return Template(paths=ordered, topk=topk, depth=depth, parent=parent, slot=slot,
                    mask=mask, retrieve=retrieve)


def regular_paths(widths) -> list:
    """All rank paths of a regular Cartesian tree with per-depth widths s_1..s_K ([CN], [Math])."""
    out = []
    frontier = [()]
    for s in widths:
        frontier = [p + (r,) for p in frontier for r in range(int(s))]
        out.extend(frontier)
    return out


def path_weight(path, acc: np.ndarray) -> float:
    """w(r_1..r_t) = prod_j a_j^(r_j) under the independence model ([M7.2] §0x04B)."""
    w = 1.0
    for j, r in enumerate(path):
        w = w * float(acc[j, r])
    return w


def _before(wa: float, pa: tuple, wb: float, pb: tuple, rel: float = 1e-12) -> bool:
    """Selection order: larger weight first; weights within `rel` tie, then shorter, then lexicographic."""
    big = max(wa, wb)
    if abs(wa - wb) <= rel * big:
        return (len(pa), pa) < (len(pb), pb)
    return wa > wb


def greedy_tree(acc: np.ndarray, budget: int, max_depth: int | None = None) -> list:
    """Greedy frontier search of [M7.2] §0x04C / [PartII] Part 3.

    acc[k, i] is the exact-rank accuracy of head k at rank i.  Starting from the
    root, repeatedly admit the frontier path of largest weight (ties as in
    `_before`, frontier scanned in (len, path) order) and open its children,
    until `budget` non-root paths are chosen.  Returns the paths in the order
    they were admitted.
    """
    acc = np.asarray(acc, dtype=np.float64)
    K, R = acc.shape
    depth_cap = K if max_depth is None else min(K, max_depth)
    if np.any(acc < 0) or np.any(acc > 1):
        raise TemplateError("accuracies must lie in [0, 1]")
    frontier = {(r,): path_weight((r,), acc) for r in range(R)}
    chosen = []
    while len(chosen) < budget and frontier:
        best = None
        for p in sorted(frontier, key=lambda q: (len(q), q)):
            if best is None or _before(frontier[p], p, frontier[best], best):
                best = p
        chosen.append(best)
        del frontier[best]
        if len(best) < depth_cap:
            for r in range(R):
                child = best + (r,)
                frontier[child] = path_weight(child, acc)
    return chosen


def expected_accept_length(paths, acc: np.ndarray) -> float:
    """E_hat[A(T)] = sum over non-root nodes of w(u) ([M7.2] §0x04B)."""
    return float(sum(path_weight(p, acc) for p in paths if len(p) > 0))


def regular_node_count(widths) -> int:
    """N_tree = sum_k prod_{i<=k} s_i ([M7.2] §0x02B; [CN] "多个 Medusa Head 如何产生候选树")."""
    total, prod = 0, 1
    for s in widths:
        prod *= int(s)
        total += prod
    return total
