"""ctypes declarations of the C ABI in include/medusa_gb300.h.

Loading fails loudly when libmedusa_gb300.so has not been built: there is no
fallback implementation of any step.
"""
from __future__ import annotations

import ctypes as C
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmedusa_gb300.so")

OK, EINVAL, ECAPACITY, EUNSUPPORTED, ETEMPLATE, ECUDA, EWORKSPACE, EPATH, ETIMEOUT = 0, -1, -2, -3, -4, -5, -6, -7, -8
ERANGE = -9
F32, BF16 = 0, 1
GREEDY, TYPICAL = 0, 1
MAX_ROWS, MAX_DEPTH, MAX_TOPK = 4096, 16, 32
MAX_LAYERS = 4096
ATTN_STATIC_SCRATCH_BYTES = 32 * 1024 * 1024

EXPORTED = [
    "medusa_tree_regular", "medusa_tree_greedy", "medusa_tree_bytes", "medusa_tree_compile",
    "medusa_tree_upload", "medusa_tree_batch", "medusa_tree_greedy_device_bytes", "medusa_tree_greedy_device",
    "medusa_heads_topk_workspace", "medusa_heads_topk", "medusa_tree_fill",
    "medusa_tree_attn_workspace", "medusa_tree_attn_verify", "medusa_tree_attn_verify_static",
    "medusa_tree_accept_workspace",
    "medusa_tree_accept", "medusa_tree_accept_commit", "medusa_tree_accept_hidden_workspace", "medusa_tree_accept_hidden", "medusa_kv_compact", "medusa_kv_compact_layers", "medusa_kv_mirror_sync", "medusa_round_workspace", "medusa_round_create",
    "medusa_round_launch", "medusa_round_destroy", "medusa_status_string", "medusa_abi_version",
    "medusa_test_set_stall_ns",
]


class MedusaTree(C.Structure):
    _fields_ = [
        ("n_rows", C.c_int32), ("n_words", C.c_int32), ("max_depth", C.c_int32),
        ("n_paths", C.c_int32), ("topk", C.c_int32), ("n_internal", C.c_int32),
        ("slot", C.c_void_p), ("depth", C.c_void_p), ("parent", C.c_void_p),
        ("retrieve", C.c_void_p), ("internal", C.c_void_p), ("internal_index", C.c_void_p),
        ("anc", C.c_void_p), ("per_seq", C.c_void_p),
    ]


class MedusaKV(C.Structure):
    _fields_ = [
        ("k", C.c_void_p), ("v", C.c_void_p), ("dtype", C.c_int32), ("n_kv_heads", C.c_int32),
        ("head_dim", C.c_int32), ("capacity", C.c_int32), ("page_size", C.c_int32),
        ("block_table", C.c_void_p), ("max_blocks", C.c_int32), ("n_pages", C.c_int32),
        ("k_f16", C.c_void_p), ("v_f16", C.c_void_p),
    ]


class MedusaRoundDesc(C.Structure):
    """medusa_round_desc: every argument of the five calls of one round."""
    _fields_ = [
        ("tree", MedusaTree), ("B", C.c_int32), ("dtype", C.c_int32),
        ("h", C.c_void_p), ("d", C.c_int32), ("V", C.c_int32), ("K", C.c_int32), ("topk", C.c_int32),
        ("w1", C.c_void_p), ("b1", C.c_void_p), ("w2", C.c_void_p), ("w2_head_stride", C.c_int64),
        ("w_lm", C.c_void_p), ("root", C.c_void_p), ("pool", C.c_void_p),
        ("L", C.c_void_p), ("tokens", C.c_void_p), ("pos", C.c_void_p),
        ("n_q_heads", C.c_int32), ("q", C.c_void_p), ("k_new", C.c_void_p), ("v_new", C.c_void_p),
        ("cache", MedusaKV), ("max_prefix", C.c_int32), ("rope_base", C.c_float), ("scale", C.c_float),
        ("out", C.c_void_p), ("lse", C.c_void_p), ("attn_status", C.c_void_p),
        ("logits", C.c_void_p), ("mode", C.c_int32), ("temperature", C.c_float), ("epsilon", C.c_float),
        ("delta", C.c_float), ("entropy_guard", C.c_int32),
        ("best_path", C.c_void_p), ("accept_len", C.c_void_p), ("out_tokens", C.c_void_p),
        ("out_rows", C.c_void_p), ("frontier_row", C.c_void_p),
        ("L_out", C.c_void_p), ("compact_status", C.c_void_p), ("hidden_target", C.c_void_p),
        ("fuse_commit", C.c_int32),
    ]


class MedusaError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} failed: {msg} (status {status})")
        self.status = status


_lib = None


def lib() -> C.CDLL:
    """The loaded library; raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it with medusa_speculative_tree_gb300.build.build()")
    L = C.CDLL(LIB_PATH)
    P, I32, I64, SZ, F, VP = C.POINTER, C.c_int32, C.c_int64, C.c_size_t, C.c_float, C.c_void_p
    sig = {
        "medusa_tree_regular": (I32, [VP, I32, VP, I32, P(I32)]),
        "medusa_tree_greedy": (I32, [VP, I32, I32, I32, VP, P(I32)]),
        "medusa_tree_bytes": (SZ, [I32, I32]),
        "medusa_tree_compile": (I32, [VP, I32, I32, I32, I32, VP, SZ, P(MedusaTree)]),
        "medusa_tree_upload": (I32, [P(MedusaTree), VP, VP, SZ, P(MedusaTree), VP]),
        "medusa_tree_batch": (I32, [P(MedusaTree), I32, VP, SZ, P(MedusaTree), VP]),
        "medusa_tree_greedy_device_bytes": (SZ, [I32, I32, I32, I32]),
        "medusa_tree_greedy_device": (I32, [VP, I32, I32, I32, I32, I32, VP, SZ, VP, VP, P(MedusaTree), VP]),
        "medusa_heads_topk_workspace": (SZ, [I32, I32, I32, I32, I32]),
        "medusa_heads_topk": (I32, [VP, I32, I32, I32, I32, VP, VP, VP, I64, VP, I32, I32, VP, VP,
                                    VP, VP, SZ, VP]),
        "medusa_tree_fill": (I32, [P(MedusaTree), I32, I32, VP, VP, VP, VP, VP, VP]),
        "medusa_tree_attn_workspace": (SZ, [P(MedusaTree), I32, I32, P(MedusaKV), I32]),
        "medusa_tree_attn_verify": (I32, [P(MedusaTree), I32, I32, VP, VP, VP, P(MedusaKV), VP, I32,
                                          F, F, VP, VP, VP, VP, SZ, VP]),
        "medusa_tree_attn_verify_static": (I32, [P(MedusaTree), I32, I32, VP, VP, VP, P(MedusaKV), VP,
                                                 I32, F, F, VP, VP, VP, VP]),
        "medusa_tree_accept_workspace": (SZ, [P(MedusaTree), I32, I32]),
        "medusa_tree_accept": (I32, [P(MedusaTree), I32, I32, VP, I32, VP, I32, F, F, F, I32, VP, VP,
                                     VP, VP, VP, VP, SZ, VP]),
        "medusa_tree_accept_commit": (I32, [P(MedusaTree), I32, I32, VP, I32, VP, I32, F, F, F, I32, P(MedusaKV), VP,
                                            VP, VP, VP, VP, VP, VP, VP, VP, SZ, VP]),
        "medusa_tree_accept_hidden_workspace": (SZ, [P(MedusaTree), I32, I32, I32]),
        "medusa_tree_accept_hidden": (I32, [P(MedusaTree), I32, I32, I32, VP, VP, VP, I32, F, F, F, VP, VP, VP, VP,
                                            VP, VP, SZ, VP]),
        "medusa_kv_compact": (I32, [P(MedusaKV), P(MedusaTree), I32, VP, VP, VP, VP, VP, VP]),
        "medusa_kv_compact_layers": (I32, [P(MedusaKV), I32, P(MedusaTree), I32, VP, VP, VP, VP, VP, VP]),
        "medusa_kv_mirror_sync": (I32, [P(MedusaKV), I32, VP]),
        "medusa_round_workspace": (SZ, [P(MedusaRoundDesc)]),
        "medusa_round_create": (I32, [P(MedusaRoundDesc), VP, SZ, VP, P(VP)]),
        "medusa_round_launch": (I32, [VP, VP]),
        "medusa_round_destroy": (I32, [VP]),
        "medusa_status_string": (C.c_char_p, [I32]),
        "medusa_abi_version": (I32, []),
        "medusa_test_set_stall_ns": (None, [C.c_uint64]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def check(fn: str, status: int) -> None:
    if status != OK:
        raise MedusaError(fn, status, lib().medusa_status_string(status).decode())
