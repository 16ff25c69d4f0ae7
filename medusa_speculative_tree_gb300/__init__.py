"""GB300-native Medusa verify round: heads + top-k, tree fill, tree attention,
acceptance and K/V compaction as CUDA kernels for sm_103a behind a C ABI
(include/medusa_gb300.h).  This package holds the in-tree build and a thin
ctypes binding; importing it does not load the library until a call is made.
"""
from . import api  # noqa: F401
from .api import (KVCache, MedusaRound, Template, TemplateBatch, batch_template_arrays, medusa_heads_topk,
                  medusa_kv_compact, medusa_tree_greedy_device,
                  medusa_kv_compact_layers, medusa_tree_accept, medusa_tree_accept_commit,
                  medusa_tree_accept_hidden, medusa_tree_attn_verify,
                  medusa_tree_attn_workspace, medusa_tree_fill, medusa_tree_greedy, medusa_tree_regular)

__all__ = [
    "KVCache", "MedusaRound", "Template", "TemplateBatch", "batch_template_arrays", "medusa_tree_greedy_device",
    "medusa_heads_topk", "medusa_tree_fill",
    "medusa_tree_attn_verify", "medusa_tree_attn_workspace", "medusa_tree_accept", "medusa_tree_accept_commit", "medusa_tree_accept_hidden",
    "medusa_kv_compact",
    "medusa_kv_compact_layers", "medusa_tree_greedy", "medusa_tree_regular",
]
