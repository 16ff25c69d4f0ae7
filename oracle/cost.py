"""Parameter, FLOP and byte ledgers of one round (oracle).

Test infrastructure only (see ``oracle/__init__.py``).  Formulas of
[M7.2] §0x02E (heads), §0x06 and §0x07C (K/V payload), §0x07B (attention pairs).
"""
from __future__ import annotations

import numpy as np


def residual_block_params(d: int) -> int:
    """P_res = d^2 + d."""
    return d * d + d


def head_params_independent(K: int, R_h: int, d: int, V: int) -> int:
    """K [R_h (d^2 + d) + V d]."""
    return K * (R_h * residual_block_params(d) + V * d)


def head_params_shared(K: int, R_h: int, d: int) -> int:
    """K R_h (d^2 + d)."""
    return K * R_h * residual_block_params(d)


def head_flops(K: int, T_h: int, R_h: int, d: int, V: int) -> int:
    """F_heads = 2 K T_h (R_h d^2 + V d)."""
    return 2 * K * T_h * (R_h * d * d + V * d)


def kv_bytes_per_node(layers: int, H_kv: int, d_h: int, bytes_per: int) -> int:
    """B_KV/node = L_layers * 2 H_kv d_h b."""
    return layers * 2 * H_kv * d_h * bytes_per


def attention_pairs(P: int, mask: np.ndarray):
    """(E_dense, E_allowed) = (N (P + N), N P + sum M)."""
    N = mask.shape[0]
    return N * (P + N), N * P + int(np.asarray(mask, dtype=bool).sum())
