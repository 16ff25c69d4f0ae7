"""Python binding of the C ABI, same names as the C entry points.

Argument marshalling only: tensors are passed as device pointers with the
current CUDA stream; every step of the round runs in libmedusa_gb300.so.
PyTorch supplies device memory (outputs and workspaces) and streams.
"""
from __future__ import annotations

import ctypes as C
from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np
import torch

from . import _native as nat
from ._native import check, lib


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(device=None):
    return C.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float32:
        return nat.F32
    if dt == torch.bfloat16:
        return nat.BF16
    raise TypeError(f"unsupported dtype {dt}")


def _need_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("expected contiguous CUDA tensors")


class _Workspace:
    """Zero-initialised device scratch, grown on demand and reused between calls.

    Kernels that keep ticket counters in their workspace return those counters to
    zero, so a reused buffer needs no clearing."""

    def __init__(self):
        self.buf = {}

    def get(self, key, nbytes: int, device) -> torch.Tensor:
        cur = self.buf.get((key, device))
        if cur is None or cur.numel() < nbytes:
            cur = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)
            self.buf[(key, device)] = cur
        return cur


_WS = _Workspace()


# ----------------------------------------------------------------------------- templates

def medusa_tree_regular(widths: Sequence[int]) -> list:
    """Rank paths of a regular Cartesian tree (host, C++)."""
    K = len(widths)
    n = C.c_int32(0)
    w = np.ascontiguousarray(widths, dtype=np.int32)
    check("medusa_tree_regular", lib().medusa_tree_regular(w.ctypes.data, K, None, 0, C.byref(n)))
    cap = max(n.value, 1)
    out = np.full((cap, max(K, 1)), -1, dtype=np.int32)
    check("medusa_tree_regular", lib().medusa_tree_regular(w.ctypes.data, K, out.ctypes.data, cap,
                                                           C.byref(n)))
    return [tuple(int(x) for x in row if x >= 0) for row in out[:n.value]]


def medusa_tree_greedy(acc: np.ndarray, budget: int) -> list:
    """Greedy frontier tree search (host, C++); paths in admission order."""
    acc = np.ascontiguousarray(acc, dtype=np.float64)
    K, R = acc.shape
    out = np.full((max(budget, 1), K), -1, dtype=np.int32)
    n = C.c_int32(0)
    check("medusa_tree_greedy", lib().medusa_tree_greedy(acc.ctypes.data, K, R, budget,
                                                         out.ctypes.data, C.byref(n)))
    return [tuple(int(x) for x in row if x >= 0) for row in out[:n.value]]


class Template:
    """A compiled tree template: host blob (for inspection) and its device copy."""

    def __init__(self, paths, topk: int, n_heads: int = 0, device=None):
        paths = [tuple(int(r) for r in p) for p in paths]
        max_len = max([len(p) for p in paths], default=0)
        arr = np.full((max(len(paths), 1), max(max_len, 1)), -1, dtype=np.int32)
        for i, p in enumerate(paths):
            arr[i, :len(p)] = p
        nbytes = lib().medusa_tree_bytes(len(paths), max_len)
        self._host = np.zeros(nbytes // 8 + 2, dtype=np.uint64)     # 8-byte aligned blob
        self.host = nat.MedusaTree()
        check("medusa_tree_compile",
              lib().medusa_tree_compile(arr.ctypes.data, len(paths), max_len, topk, n_heads,
                                        self._host.ctypes.data, self._host.nbytes, C.byref(self.host)))
        self.n_rows = self.host.n_rows
        self.n_words = self.host.n_words
        self.max_depth = self.host.max_depth
        self.n_paths = self.host.n_paths
        self.topk = self.host.topk
        self.n_internal = self.host.n_internal
        self.dev = None
        self.device = None
        if device is not None:
            self.to(device)

    def _arr(self, field, count, dtype=np.int32):
        addr = getattr(self.host, field)
        buf = (C.c_char * (count * np.dtype(dtype).itemsize)).from_address(addr)
        return np.frombuffer(buf, dtype=dtype).copy()

    @property
    def slot(self):
        return self._arr("slot", self.n_rows)

    @property
    def depth(self):
        return self._arr("depth", self.n_rows)

    @property
    def parent(self):
        return self._arr("parent", self.n_rows)

    @property
    def retrieve(self):
        return self._arr("retrieve", self.n_paths * (self.max_depth + 1)).reshape(
            self.n_paths, self.max_depth + 1)

    @property
    def internal(self):
        return self._arr("internal", self.n_internal)

    @property
    def anc(self):
        return self._arr("anc", self.n_rows * self.n_words, np.uint64).reshape(self.n_rows, self.n_words)

    def to(self, device):
        device = torch.device(device)
        self._dev_buf = torch.empty(self._host.nbytes, dtype=torch.uint8, device=device)
        self.dev = nat.MedusaTree()
        check("medusa_tree_upload",
              lib().medusa_tree_upload(C.byref(self.host), self._host.ctypes.data,
                                       C.c_void_p(self._dev_buf.data_ptr()), self._dev_buf.numel(),
                                       C.byref(self.dev), _stream(device)))
        torch.cuda.current_stream(device).synchronize()     # host blob copied before it may change
        self.device = device
        return self


class TemplateBatch:
    """Per-sequence templates of one batch (medusa_tree_batch): sequence b verifies
    templates[index[b]].  Usable wherever a Template is: per-row tensors are laid out
    with the batch's bound n_rows (and max_depth + 1 for published rows)."""

    def __init__(self, templates: Sequence[Template], index: Sequence[int], device=None):
        device = torch.device(device) if device is not None else templates[0].device
        B = len(index)
        self._templates = list(templates)
        self._descs = (nat.MedusaTree * B)(*[templates[int(i)].dev for i in index])
        nbytes = B * C.sizeof(nat.MedusaTree)
        self._dev_descs = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self.dev = nat.MedusaTree()
        check("medusa_tree_batch",
              lib().medusa_tree_batch(self._descs, B, C.c_void_p(self._dev_descs.data_ptr()), nbytes,
                                      C.byref(self.dev), _stream(device)))
        torch.cuda.current_stream(device).synchronize()     # host descriptors copied
        self.index = [int(i) for i in index]
        self.device = device
        self.n_rows = self.dev.n_rows
        self.n_words = self.dev.n_words
        self.max_depth = self.dev.max_depth
        self.n_paths = self.dev.n_paths
        self.topk = self.dev.topk
        self.n_internal = self.dev.n_internal

    @classmethod
    def from_device(cls, dev: "nat.MedusaTree", keep=(), device=None):
        """A batch descriptor built on the device (medusa_tree_greedy_device)."""
        self = cls.__new__(cls)
        self._templates = []
        self._keep = keep
        self.dev = dev
        self.index = None
        self.device = torch.device(device) if device is not None else None
        self.n_rows = dev.n_rows
        self.n_words = dev.n_words
        self.max_depth = dev.max_depth
        self.n_paths = dev.n_paths
        self.topk = dev.topk
        self.n_internal = dev.n_internal
        return self


def medusa_tree_greedy_device(acc, budget: int, topk: int):
    """Greedy trees built on the GPU, one per sequence (medusa_tree_greedy_device):
    acc [B, K, R] float64 CUDA tensor of rank accuracies.  Returns (TemplateBatch, status [B])."""
    _need_cuda(acc)
    if acc.dtype != torch.float64 or acc.dim() != 3:
        raise ValueError("acc must be a [B, K, R] float64 CUDA tensor")
    B, K, R = acc.shape
    dev = acc.device
    nb = lib().medusa_tree_greedy_device_bytes(B, K, R, budget)
    if nb == 0:
        raise ValueError("invalid greedy tree shape")
    buf = torch.empty(nb, dtype=torch.uint8, device=dev)
    descs = torch.empty(B * C.sizeof(nat.MedusaTree), dtype=torch.uint8, device=dev)
    status = torch.empty(B, dtype=torch.int32, device=dev)
    out = nat.MedusaTree()
    check("medusa_tree_greedy_device",
          lib().medusa_tree_greedy_device(_ptr(acc), B, K, R, budget, topk, _ptr(buf), nb, _ptr(descs), _ptr(status),
                                          C.byref(out), _stream(dev)))
    return TemplateBatch.from_device(out, keep=(buf, descs, acc), device=dev), status


def batch_template_arrays(batch, b: int) -> dict:
    """Host copies of sequence b's template arrays of a batch built by
    medusa_tree_greedy_device (read from the blob buffer that holds them)."""
    buf, descs = batch._keep[0], batch._keep[1]
    sz = C.sizeof(nat.MedusaTree)
    raw = descs[b * sz:(b + 1) * sz].cpu().numpy().tobytes()
    t = nat.MedusaTree.from_buffer_copy(raw)
    host = buf.cpu().numpy()
    base = buf.data_ptr()

    def arr(addr, count, dtype):
        off = int(addr) - base
        nbytes = count * np.dtype(dtype).itemsize
        return host[off:off + nbytes].view(dtype).copy()
    N, W = t.n_rows, t.max_depth + 1
    return {"n_rows": N, "n_words": t.n_words, "max_depth": t.max_depth, "n_paths": t.n_paths,
            "topk": t.topk, "n_internal": t.n_internal,
            "slot": arr(t.slot, N, np.int32), "depth": arr(t.depth, N, np.int32),
            "parent": arr(t.parent, N, np.int32),
            "retrieve": arr(t.retrieve, t.n_paths * W, np.int32).reshape(t.n_paths, W),
            "internal": arr(t.internal, t.n_internal, np.int32),
            "internal_index": arr(t.internal_index, N, np.int32),
            "anc": arr(t.anc, N * t.n_words, np.uint64).reshape(N, t.n_words)}


# ----------------------------------------------------------------------------- KV cache

@dataclass
class KVCache:
    """One layer's cache: contiguous [B, Hkv, cap, dh] or paged [pages, Hkv, 16, dh].

    k_f16 / v_f16: an optional fp16 mirror of a bf16 cache (same shapes), which the
    tensor-core attention reads instead of converting the prefix on every call; the
    library's own cache writes keep it in step once filled (add_mirror, sync_mirror)."""

    k: torch.Tensor
    v: torch.Tensor
    block_table: Optional[torch.Tensor] = None    # int32 [B, max_blocks] for paged caches
    capacity: Optional[int] = None
    k_f16: Optional[torch.Tensor] = None
    v_f16: Optional[torch.Tensor] = None

    def add_mirror(self) -> "KVCache":
        """Allocate the fp16 mirror and fill it from the cache (medusa_kv_mirror_sync)."""
        self.k_f16 = torch.empty(self.k.shape, dtype=torch.float16, device=self.k.device)
        self.v_f16 = torch.empty(self.v.shape, dtype=torch.float16, device=self.v.device)
        self.sync_mirror()
        return self

    def sync_mirror(self):
        """Refill the mirror from the cache, stream-ordered (after writes made outside
        this library)."""
        B = self.k.shape[0] if self.block_table is None else 1
        check("medusa_kv_mirror_sync", lib().medusa_kv_mirror_sync(C.byref(self.desc()), B, _stream(self.k.device)))

    def desc(self) -> nat.MedusaKV:
        _need_cuda(self.k, self.v, self.block_table, self.k_f16, self.v_f16)
        d = nat.MedusaKV()
        d.k, d.v = self.k.data_ptr(), self.v.data_ptr()
        d.k_f16 = self.k_f16.data_ptr() if self.k_f16 is not None else None
        d.v_f16 = self.v_f16.data_ptr() if self.v_f16 is not None else None
        if (self.k_f16 is not None) and (self.k_f16.shape != self.k.shape or self.v_f16 is None
                                         or self.v_f16.shape != self.v.shape
                                         or self.k_f16.dtype != torch.float16 or self.v_f16.dtype != torch.float16):
            raise ValueError("the fp16 mirror must be two float16 tensors of the cache's shapes")
        d.dtype = _dtype_code(self.k.dtype)
        if self.block_table is None:
            _, Hkv, cap, dh = self.k.shape
            d.n_kv_heads, d.head_dim, d.capacity = Hkv, dh, cap
            d.page_size, d.block_table, d.max_blocks, d.n_pages = 0, None, 0, 0
        else:
            n_pages, Hkv, ps, dh = self.k.shape
            mb = self.block_table.shape[1]
            d.n_kv_heads, d.head_dim = Hkv, dh
            d.capacity = self.capacity if self.capacity is not None else mb * ps
            d.page_size, d.block_table, d.max_blocks, d.n_pages = ps, self.block_table.data_ptr(), mb, n_pages
        return d


# ----------------------------------------------------------------------------- round steps

def medusa_heads_topk(h, w1, w2, w_lm, topk: int, b1=None, logits_out=None, shared_w2=False):
    """root [T] int32, pool [T, K, topk] int32 (and fills logits_out [T, K+1, V] fp32 if given)."""
    _need_cuda(h, w1, w2, w_lm, b1, logits_out)
    T, d = h.shape
    V = w_lm.shape[0]
    K = w1.shape[0]
    dev = h.device
    stride = 0 if shared_w2 else V * d
    root = torch.empty(T, dtype=torch.int32, device=dev)
    pool = torch.empty((T, K, topk), dtype=torch.int32, device=dev)
    nb = lib().medusa_heads_topk_workspace(T, d, V, K, topk)
    ws = _WS.get("heads", nb, dev)
    check("medusa_heads_topk",
          lib().medusa_heads_topk(_ptr(h), T, d, V, K, _ptr(w1), _ptr(b1), _ptr(w2), stride, _ptr(w_lm),
                                  topk, _dtype_code(h.dtype), _ptr(root), _ptr(pool), _ptr(logits_out),
                                  _ptr(ws), ws.numel(), _stream(dev)))
    return root, pool


def medusa_tree_fill(tmpl: Template, root, pool, L):
    """tokens [B, N], pos [B, N] int32."""
    _need_cuda(root, pool, L)
    B = root.shape[0]
    K = pool.shape[1] if pool.dim() == 3 else 0
    tokens = torch.empty((B, tmpl.n_rows), dtype=torch.int32, device=root.device)
    pos = torch.empty_like(tokens)
    check("medusa_tree_fill",
          lib().medusa_tree_fill(C.byref(tmpl.dev), B, K, _ptr(root), _ptr(pool), _ptr(L), _ptr(tokens),
                                 _ptr(pos), _stream(root.device)))
    return tokens, pos


def medusa_tree_attn_workspace(tmpl: Template, B: int, n_q_heads: int, cache: KVCache, max_prefix: int) -> int:
    d = cache.desc()
    return lib().medusa_tree_attn_workspace(C.byref(tmpl.dev), B, n_q_heads, C.byref(d), max_prefix)


def medusa_tree_attn_verify(tmpl: Template, q, k_new, v_new, cache: KVCache, L, max_prefix: int,
                            rope_base: float = 10000.0, scale: Optional[float] = None, want_lse=False,
                            out=None, ws=None):
    """out [B, N, Hq, dh] fp32, lse [B, N, Hq] fp32 or None, status [B] int32."""
    _need_cuda(q, k_new, v_new, L, out)
    B, N, Hq, dh = q.shape
    dev = q.device
    if scale is None:
        scale = 1.0 / float(dh) ** 0.5
    d = cache.desc()
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float32, device=dev)
    lse = torch.empty((B, N, Hq), dtype=torch.float32, device=dev) if want_lse else None
    status = torch.empty(B, dtype=torch.int32, device=dev)
    nb = lib().medusa_tree_attn_workspace(C.byref(tmpl.dev), B, Hq, C.byref(d), max_prefix)
    if nb == 0:
        raise ValueError("invalid tree attention shapes")
    if ws is None:
        ws = _WS.get("attn", nb, dev)
    check("medusa_tree_attn_verify",
          lib().medusa_tree_attn_verify(C.byref(tmpl.dev), B, Hq, _ptr(q), _ptr(k_new), _ptr(v_new),
                                        C.byref(d), _ptr(L), max_prefix, float(rope_base), float(scale),
                                        _ptr(out), _ptr(lse), _ptr(status), _ptr(ws), ws.numel(),
                                        _stream(dev)))
    return out, lse, status


def medusa_tree_accept(tmpl: Template, logits, tokens, mode: str = "greedy", temperature: float = 1.0,
                       epsilon: float = 0.09, delta: float = 0.3, entropy_guard: bool = False):
    """dict of best_path, accept_len, out_tokens, out_rows, frontier_row (int32 device tensors)."""
    _need_cuda(logits, tokens)
    B, N, V = logits.shape
    dev = logits.device
    W = tmpl.max_depth + 1
    r = {k: torch.empty(B, dtype=torch.int32, device=dev) for k in ("best_path", "accept_len", "frontier_row")}
    r["out_tokens"] = torch.empty((B, W), dtype=torch.int32, device=dev)
    r["out_rows"] = torch.empty((B, W), dtype=torch.int32, device=dev)
    nb = lib().medusa_tree_accept_workspace(C.byref(tmpl.dev), B, V)
    ws = _WS.get("accept", nb, dev)
    m = nat.GREEDY if mode == "greedy" else nat.TYPICAL
    check("medusa_tree_accept",
          lib().medusa_tree_accept(C.byref(tmpl.dev), B, V, _ptr(logits), _dtype_code(logits.dtype),
                                   _ptr(tokens), m, float(temperature), float(epsilon), float(delta),
                                   int(entropy_guard), _ptr(r["best_path"]), _ptr(r["accept_len"]),
                                   _ptr(r["out_tokens"]), _ptr(r["out_rows"]), _ptr(r["frontier_row"]),
                                   _ptr(ws), ws.numel(), _stream(dev)))
    return r


def medusa_tree_accept_commit(tmpl: Template, logits, tokens, cache: KVCache, L, mode: str = "greedy",
                              temperature: float = 1.0, epsilon: float = 0.09, delta: float = 0.3,
                              entropy_guard: bool = False):
    """medusa_tree_accept and medusa_kv_compact of the winner in one: the acceptance dict
    plus L_out and status (int32 device tensors); the cache is compacted in place."""
    _need_cuda(logits, tokens, L)
    B, N, V = logits.shape
    dev = logits.device
    W = tmpl.max_depth + 1
    r = {k: torch.empty(B, dtype=torch.int32, device=dev)
         for k in ("best_path", "accept_len", "frontier_row", "L_out", "status")}
    r["out_tokens"] = torch.empty((B, W), dtype=torch.int32, device=dev)
    r["out_rows"] = torch.empty((B, W), dtype=torch.int32, device=dev)
    nb = lib().medusa_tree_accept_workspace(C.byref(tmpl.dev), B, V)
    ws = _WS.get("accept", nb, dev)
    m = nat.GREEDY if mode == "greedy" else nat.TYPICAL
    d = cache.desc()
    check("medusa_tree_accept_commit",
          lib().medusa_tree_accept_commit(C.byref(tmpl.dev), B, V, _ptr(logits), _dtype_code(logits.dtype),
                                          _ptr(tokens), m, float(temperature), float(epsilon), float(delta),
                                          int(entropy_guard), C.byref(d), _ptr(L), _ptr(r["best_path"]),
                                          _ptr(r["accept_len"]), _ptr(r["out_tokens"]), _ptr(r["out_rows"]),
                                          _ptr(r["frontier_row"]), _ptr(r["L_out"]), _ptr(r["status"]), _ptr(ws),
                                          ws.numel(), _stream(dev)))
    return r


def medusa_tree_accept_hidden(tmpl: Template, hidden, w_lm, tokens, mode: str = "greedy",
                              temperature: float = 1.0, epsilon: float = 0.09, delta: float = 0.3):
    """medusa_tree_accept on the target's final hidden states: the vocabulary projection
    of the internal rows is folded in (hidden [B, N, d] bf16, w_lm [V, d] bf16)."""
    _need_cuda(hidden, w_lm, tokens)
    B, N, d = hidden.shape
    V = w_lm.shape[0]
    dev = hidden.device
    W = tmpl.max_depth + 1
    r = {k: torch.empty(B, dtype=torch.int32, device=dev) for k in ("best_path", "accept_len", "frontier_row")}
    r["out_tokens"] = torch.empty((B, W), dtype=torch.int32, device=dev)
    r["out_rows"] = torch.empty((B, W), dtype=torch.int32, device=dev)
    nb = lib().medusa_tree_accept_hidden_workspace(C.byref(tmpl.dev), B, V, d)
    if nb == 0:
        raise ValueError("invalid acceptance shapes")
    ws = _WS.get("accept_hidden", nb, dev)
    m = nat.GREEDY if mode == "greedy" else nat.TYPICAL
    check("medusa_tree_accept_hidden",
          lib().medusa_tree_accept_hidden(C.byref(tmpl.dev), B, V, d, _ptr(hidden), _ptr(w_lm), _ptr(tokens), m,
                                          float(temperature), float(epsilon), float(delta), _ptr(r["best_path"]),
                                          _ptr(r["accept_len"]), _ptr(r["out_tokens"]), _ptr(r["out_rows"]),
                                          _ptr(r["frontier_row"]), _ptr(ws), ws.numel(), _stream(dev)))
    return r


def medusa_kv_compact(cache: KVCache, tmpl: Template, L, accept_len, out_rows):
    """L_out [B], status [B] int32; the cache is compacted in place."""
    _need_cuda(L, accept_len, out_rows)
    B = L.shape[0]
    dev = L.device
    L_out = torch.empty(B, dtype=torch.int32, device=dev)
    status = torch.empty(B, dtype=torch.int32, device=dev)
    d = cache.desc()
    check("medusa_kv_compact",
          lib().medusa_kv_compact(C.byref(d), C.byref(tmpl.dev), B, _ptr(L), _ptr(accept_len),
                                  _ptr(out_rows), _ptr(L_out), _ptr(status), _stream(dev)))
    return L_out, status


def medusa_kv_compact_layers(caches: Sequence[KVCache], tmpl: Template, L, accept_len, out_rows):
    """medusa_kv_compact for every layer's cache at once; L_out [B], status [B] int32."""
    _need_cuda(L, accept_len, out_rows)
    B = L.shape[0]
    dev = L.device
    L_out = torch.empty(B, dtype=torch.int32, device=dev)
    status = torch.empty(B, dtype=torch.int32, device=dev)
    arr = (nat.MedusaKV * len(caches))(*[c.desc() for c in caches])
    check("medusa_kv_compact_layers",
          lib().medusa_kv_compact_layers(arr, len(caches), C.byref(tmpl.dev), B, _ptr(L), _ptr(accept_len),
                                         _ptr(out_rows), _ptr(L_out), _ptr(status), _stream(dev)))
    return L_out, status


# ----------------------------------------------------------------------------- whole round

class MedusaRound:
    """One verify round recorded as a CUDA graph of the five calls
    (medusa_round_create); launch() replays it with one graph launch.

    The inputs are the device tensors given here, referenced by address: write new
    values into them (copy_) before a launch.  The outputs are tensors allocated here
    and overwritten by every launch: root, pool, tokens, pos, out, lse (or None),
    attn_status, best_path, accept_len, out_tokens, out_rows, frontier_row, L_out,
    compact_status.  The heads run on one frontier row per sequence (h is [B, d]).
    With hidden_target ([B, N, d] bf16, the target's final hidden states of the tree
    rows) acceptance projects the internal rows through w_lm itself
    (medusa_tree_accept_hidden) and logits may be None.  With fuse_commit the winning
    rows are committed by the acceptance kernel itself (medusa_tree_accept_commit):
    one launch fewer, the same results."""

    _OUT = ("root", "pool", "tokens", "pos", "out", "lse", "attn_status", "best_path", "accept_len",
            "out_tokens", "out_rows", "frontier_row", "L_out", "compact_status")

    def __init__(self, tmpl: Template, h, w1, w2, w_lm, topk: int, L, q, k_new, v_new, cache: KVCache,
                 max_prefix: int, logits, mode: str = "greedy", rope_base: float = 10000.0,
                 scale: Optional[float] = None, temperature: float = 1.0, epsilon: float = 0.09,
                 delta: float = 0.3, entropy_guard: bool = False, b1=None, shared_w2: bool = False,
                 want_lse: bool = False, hidden_target=None, fuse_commit: bool = False):
        _need_cuda(h, w1, w2, w_lm, b1, L, q, k_new, v_new, logits, hidden_target)
        B, d = h.shape
        V, K, N = w_lm.shape[0], w1.shape[0], tmpl.n_rows
        Bq, Nq, Hq, dh = q.shape
        if Bq != B or Nq != N or tuple(L.shape) != (B,):
            raise ValueError("inconsistent round shapes")
        if hidden_target is None:
            if logits is None or tuple(logits.shape) != (B, N, V) or logits.dtype != h.dtype:
                raise ValueError("logits must be [B, N, V] in the dtype of the hidden rows")
        elif tuple(hidden_target.shape) != (B, N, d) or hidden_target.dtype != h.dtype:
            raise ValueError("hidden_target must be [B, N, d] in the dtype of the hidden rows")
        dev = h.device
        i32 = dict(dtype=torch.int32, device=dev)
        W = tmpl.max_depth + 1
        self.root = torch.empty(B, **i32)
        self.pool = torch.empty((B, K, topk), **i32)
        self.tokens = torch.empty((B, N), **i32)
        self.pos = torch.empty((B, N), **i32)
        self.out = torch.empty(tuple(q.shape), dtype=torch.float32, device=dev)
        self.lse = torch.empty((B, N, Hq), dtype=torch.float32, device=dev) if want_lse else None
        self.attn_status = torch.empty(B, **i32)
        self.best_path = torch.empty(B, **i32)
        self.accept_len = torch.empty(B, **i32)
        self.out_tokens = torch.empty((B, W), **i32)
        self.out_rows = torch.empty((B, W), **i32)
        self.frontier_row = torch.empty(B, **i32)
        self.L_out = torch.empty(B, **i32)
        self.compact_status = torch.empty(B, **i32)
        # the graph records addresses: keep every input alive as long as the round
        self._inputs = (tmpl, h, w1, w2, w_lm, b1, L, q, k_new, v_new, cache, logits, hidden_target)
        r = nat.MedusaRoundDesc()
        r.tree = tmpl.dev
        r.B, r.dtype = B, _dtype_code(h.dtype)
        r.h, r.d, r.V, r.K, r.topk = h.data_ptr(), d, V, K, topk
        r.w1, r.b1, r.w2 = w1.data_ptr(), (b1.data_ptr() if b1 is not None else None), w2.data_ptr()
        r.w2_head_stride = 0 if shared_w2 else V * d
        r.w_lm, r.root, r.pool = w_lm.data_ptr(), self.root.data_ptr(), self.pool.data_ptr()
        r.L, r.tokens, r.pos = L.data_ptr(), self.tokens.data_ptr(), self.pos.data_ptr()
        r.n_q_heads, r.q, r.k_new, r.v_new = Hq, q.data_ptr(), k_new.data_ptr(), v_new.data_ptr()
        r.cache = cache.desc()
        r.max_prefix = int(max_prefix)
        r.rope_base = float(rope_base)
        r.scale = float(scale) if scale is not None else 1.0 / float(dh) ** 0.5
        r.out, r.lse = self.out.data_ptr(), (self.lse.data_ptr() if self.lse is not None else None)
        r.attn_status = self.attn_status.data_ptr()
        r.logits = logits.data_ptr() if logits is not None else None
        r.hidden_target = hidden_target.data_ptr() if hidden_target is not None else None
        r.fuse_commit = 1 if fuse_commit else 0
        r.mode = nat.GREEDY if mode == "greedy" else nat.TYPICAL
        r.temperature, r.epsilon, r.delta = float(temperature), float(epsilon), float(delta)
        r.entropy_guard = int(entropy_guard)
        r.best_path, r.accept_len = self.best_path.data_ptr(), self.accept_len.data_ptr()
        r.out_tokens, r.out_rows = self.out_tokens.data_ptr(), self.out_rows.data_ptr()
        r.frontier_row = self.frontier_row.data_ptr()
        r.L_out, r.compact_status = self.L_out.data_ptr(), self.compact_status.data_ptr()
        self.desc = r
        nb = lib().medusa_round_workspace(C.byref(r))
        if nb == 0:
            raise ValueError("invalid round arguments")
        self.ws = torch.empty(nb, dtype=torch.uint8, device=dev)
        self.device = dev
        self._handle = C.c_void_p()
        check("medusa_round_create",
              lib().medusa_round_create(C.byref(r), _ptr(self.ws), nb, _stream(dev), C.byref(self._handle)))

    def launch(self, stream: Optional[torch.cuda.Stream] = None):
        """Enqueue the whole round on `stream` (default: the current stream)."""
        s = C.c_void_p((stream or torch.cuda.current_stream(self.device)).cuda_stream)
        check("medusa_round_launch", lib().medusa_round_launch(self._handle, s))

    def results(self) -> dict:
        return {k: getattr(self, k) for k in self._OUT}

    def close(self):
        """Free the graph (after the device has finished every launch)."""
        if self._handle is not None and self._handle.value:
            torch.cuda.synchronize(self.device)
            check("medusa_round_destroy", lib().medusa_round_destroy(self._handle))
        self._handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
