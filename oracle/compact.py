"""Winning-path K/V compaction (oracle).

Test infrastructure only (see ``oracle/__init__.py``).

With G = a + 1 published tokens and winning rows u_0..u_a, staged source
rows s_j = P + u_j are gathered into a snapshot first and then written to the
compact destinations d_j = P + j; the committed length becomes P + G
([M7.2] §0x06A, §0x06B; [CN] "一次完整解码迭代" step 5).
"""
from __future__ import annotations

import numpy as np


def kv_compact(cache_k: np.ndarray, cache_v: np.ndarray, L: int, rows) -> int:
    """Compact in place.  cache_k/cache_v [Hkv, capacity, dh] of one sequence and one layer.

    Returns the new committed length L + G.
    """
    rows = np.asarray(rows, dtype=np.int64)
    G = rows.shape[0]
    src = L + rows
    snap_k = cache_k[:, src, :].copy()     # snapshot before any write
    snap_v = cache_v[:, src, :].copy()
    cache_k[:, L:L + G, :] = snap_k
    cache_v[:, L:L + G, :] = snap_v
    return L + G


def compaction_map(L: int, rows):
    """(sources, destinations) of the gather-and-compact step."""
    rows = np.asarray(rows, dtype=np.int64)
    return L + rows, L + np.arange(rows.shape[0], dtype=np.int64)
