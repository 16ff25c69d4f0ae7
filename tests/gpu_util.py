"""Helpers shared by the GPU parity tests: building inputs from `synth`, moving
them between the devices and the tolerance checks of the parity bar."""
from __future__ import annotations

import numpy as np
import torch

import synth

# Parity bar: fp32 inputs within 1e-5; bf16 inputs (fp32 accumulation) within
# max-abs 2e-2 and relative-L2 1e-3.
F32_ABS = 1e-5
BF16_ABS = 2e-2
BF16_REL_L2 = 1e-3


def to64(t) -> np.ndarray:
    if isinstance(t, np.ndarray):
        return t.astype(np.float64)
    return t.detach().to("cpu", torch.float64).numpy()


def float_parity(got, want, is_f32: bool, what: str = ""):
    got, want = to64(got), to64(want)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite GPU values"
    err = np.abs(got - want)
    if is_f32:
        assert err.max() <= F32_ABS, f"{what}: max abs err {err.max():.3g} > {F32_ABS}"
        return float(err.max()), None
    rel = float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-30))
    assert err.max() <= BF16_ABS, f"{what}: max abs err {err.max():.3g} > {BF16_ABS}"
    assert rel <= BF16_REL_L2, f"{what}: rel-L2 {rel:.3g} > {BF16_REL_L2}"
    return float(err.max()), rel


def topk_parity(ids_gpu, values64, k: int, tol: float) -> int:
    """GPU top-k ids against the oracle's fp64 values of the same row.

    Equal lists pass.  Otherwise each differing rank must be a near tie: the
    oracle value at the GPU's id lies within `tol` of the oracle's value at that
    rank (the two sides rank in different precisions).  Returns the number of
    ranks decided by such near ties."""
    ids_gpu = [int(x) for x in ids_gpu]
    assert len(set(ids_gpu)) == len(ids_gpu)
    order = np.lexsort((np.arange(values64.shape[0]), -values64))[:k]
    amb = 0
    for r in range(k):
        if ids_gpu[r] != int(order[r]):
            assert abs(values64[ids_gpu[r]] - values64[order[r]]) <= tol, (r, ids_gpu, list(order))
            amb += 1
    return amb


def device_tensor(x, dtype, device="cuda"):
    return torch.as_tensor(np.ascontiguousarray(x)).to(device=device, dtype=dtype)


def contiguous_cache(w: synth.Workload, lengths, n_rows, guard=16, device="cuda", fill_tail=0.0):
    """[B, Hkv, cap, dh] caches holding the seeded prefix rows; rows >= L filled with `fill_tail`."""
    ks, vs = synth.prefix_kv(w, lengths, device="cpu")
    cap = int(max(lengths)) + n_rows + guard
    dt = w.torch_dtype
    K = torch.full((w.batch, w.n_kv_heads, cap, w.head_dim), fill_tail, dtype=dt)
    V = torch.full_like(K, fill_tail)
    for b, L in enumerate(lengths):
        K[b, :, :L] = ks[b]
        V[b, :, :L] = vs[b]
    return K.to(device), V.to(device), ks, vs


def paged_cache(w: synth.Workload, lengths, n_rows, device="cuda", fill_tail=0.0):
    """Paged [pages, Hkv, 16, dh] caches with a shuffled block table."""
    lay = synth.paged_layout(w, lengths, n_rows)
    ps = lay.page_size
    ks, vs = synth.prefix_kv(w, lengths, device="cpu")
    dt = w.torch_dtype
    K = torch.full((lay.n_pages, w.n_kv_heads, ps, w.head_dim), fill_tail, dtype=dt)
    V = torch.full_like(K, fill_tail)
    for b, L in enumerate(lengths):
        for r0 in range(0, int(L), ps):
            page = int(lay.block_table[b, r0 // ps])
            n = min(ps, int(L) - r0)
            K[page, :, :n] = ks[b][:, r0:r0 + n]
            V[page, :, :n] = vs[b][:, r0:r0 + n]
    bt = torch.as_tensor(lay.block_table, dtype=torch.int32)     # -1 marks unused entries
    return K.to(device), V.to(device), bt.to(device), lay, ks, vs


def read_paged_row(K, block_table, b, row, ps=16):
    page = int(block_table[b, row // ps])
    return K[page, :, row % ps]


def typical_ambiguous(o, rel: float = 1e-5) -> bool:
    """True when a typical-acceptance decision or the winning tie-break of an oracle
    result lies within `rel` of its threshold, where fp32 and fp64 may differ."""
    if o.margins and min(o.margins) < rel:
        return True
    sc = sorted(o.per_path_score[o.per_path_len == o.accept_len])[::-1]
    if len(sc) >= 2 and sc[0] != sc[1] and sc[0] - sc[1] < rel * max(1.0, abs(sc[0])):
        return True
    return False


def oracle_heads_blocked(h, w1, w2, w_lm, topk: int, block: int = 4096):
    """The oracle's medusa_heads on device-resident weights, with the vocabulary rows of
    W2 and W_LM brought to the host in blocks: the fp64 copies of the larger workloads'
    weights (up to 44 GB) do not fit in host memory at once.  The same oracle functions
    run on slices of their inputs (residual on all of W1; head_logits on each block of
    W2, and on each block of W_LM as a one-head shared projection); ranked_ids then
    selects root and pools from the assembled fp64 logits, as medusa_heads does.
    Returns (root [T], pool [T, K, topk], logits [T, K + 1, V] fp64)."""
    from oracle import heads as oheads
    h64 = to64(h)
    z = oheads.residual(h64, to64(w1))
    T, K, V = h64.shape[0], w1.shape[0], w_lm.shape[0]
    logits = np.empty((T, K + 1, V))
    for v0 in range(0, V, block):
        v1 = min(V, v0 + block)
        logits[:, 1:, v0:v1] = oheads.head_logits(z, to64(w2[:, v0:v1]))
        logits[:, 0, v0:v1] = oheads.head_logits(h64[:, None, :], to64(w_lm[v0:v1]))[:, 0]
    root = np.array([oheads.ranked_ids(logits[t, 0], 1)[0] for t in range(T)], dtype=np.int64)
    pool = np.zeros((T, K, topk), dtype=np.int64)
    for t in range(T):
        for k in range(K):
            pool[t, k] = oheads.ranked_ids(logits[t, 1 + k], topk)
    return root, pool, logits
