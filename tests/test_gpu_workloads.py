"""GPU parity at the five workloads' full sizes, in the launch configuration the
benchmark times.  The oracle checks sampled outputs one by one (head logits at
sampled vocabulary rows, attention at sampled (node, head) pairs) and whole
outputs where it is cheap (fill, acceptance, compaction).  Every step is fed
from the seeded generators, never from an upstream GPU step.
"""
import math

import numpy as np
import pytest
import torch

import synth
from oracle import accept as oacc
from oracle import attention as oatt
from oracle import compact as ocomp
from oracle import heads as oheads
from oracle import round as oround
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    import medusa_speculative_tree_gb300 as m
    from medusa_speculative_tree_gb300 import build
    build.build()
    return m


def templates(m, w):
    acc = synth.rank_accuracy(w.n_heads, 10)
    t_o = oround.template_for(w.template, w.topk, w.n_heads, acc)
    t_g = m.Template(t_o.paths[1:], w.topk, w.n_heads, device="cuda")
    return t_o, t_g, acc


def test_full_round_tiny_fp32(m):
    """The whole chained round on the GPU against the oracle's chained round."""
    w = synth.WORKLOADS["tiny-fp32"]
    t_o, t_g, acc = templates(m, w)
    N = t_o.n_rows
    h, w1, w2, w_lm = synth.head_weights(w)
    q, k, v = synth.tree_qkv(w, N)
    lengths = synth.prefix_lengths(w)
    K, V, ks, vs = gu.contiguous_cache(w, lengths, N)
    for plant in (False, True):
        logits = synth.target_logits(w, N, sub=int(plant))
        o_root, o_pool, _ = oheads.medusa_heads(gu.to64(h), gu.to64(w1), gu.to64(w2), gu.to64(w_lm), w.topk)
        if plant:
            synth.plant_argmax(logits, o_pool, t_o.depth, acc, synth.plant_uniforms(w, N))
        Kd, Vd = K.clone(), V.clone()
        cache = m.KVCache(Kd, Vd)
        Ld = gu.device_tensor(lengths, torch.int32)
        root, pool = m.medusa_heads_topk(h.cuda(), w1.cuda(), w2.cuda(), w_lm.cuda(), w.topk)
        tokens, pos = m.medusa_tree_fill(t_g, root, pool, Ld)
        out, lse, st = m.medusa_tree_attn_verify(t_g, q.cuda(), k.cuda(), v.cuda(), cache, Ld, int(lengths.max()))
        r = m.medusa_tree_accept(t_g, logits.cuda(), tokens, "greedy")
        L_out, st2 = m.medusa_kv_compact(cache, t_g, Ld, r["accept_len"], r["out_rows"])
        torch.cuda.synchronize()

        ck = gu.to64(K[0]).copy()
        cv = gu.to64(V[0]).copy()
        o = oround.run_sequence(t_o, gu.to64(h[0]), gu.to64(w1), gu.to64(w2), gu.to64(w_lm), gu.to64(q[0]),
                                gu.to64(k[0]), gu.to64(v[0]), ck, cv, int(lengths[0]), gu.to64(logits[0]),
                                "greedy", w.rope_base)
        assert int(root[0]) == o.root and (pool[0].cpu().numpy() == o.pool).all()
        assert (tokens[0].cpu().numpy() == o.tokens).all() and (pos[0].cpu().numpy() == o.pos).all()
        gu.float_parity(out[0], o.attn_out, True, "round attention")
        assert int(r["accept_len"][0]) == o.accept.accept_len
        G = o.accept.accept_len + 1
        assert list(r["out_tokens"][0, :G].cpu().numpy()) == list(o.accept.out_tokens)
        assert int(L_out[0]) == o.new_len and int(st[0]) == 0 and int(st2[0]) == 0
        gu.float_parity(Kd[0, :, :o.new_len], ck[:, :o.new_len], True, "compacted K")
        gu.float_parity(Vd[0, :, :o.new_len], cv[:, :o.new_len], True, "compacted V")
        if plant:
            assert o.accept.accept_len > 0


@pytest.mark.parametrize("name", synth.WORKLOAD_ORDER)
def test_heads_full_size_sampled(m, name):
    w = synth.WORKLOADS[name]
    T = w.batch
    h, w1, w2, w_lm = synth.head_weights(w, device="cuda")
    logits = torch.empty((T, w.n_heads + 1, w.vocab), dtype=torch.float32, device="cuda")
    root, pool = m.medusa_heads_topk(h, w1, w2, w_lm, w.topk, logits_out=logits)
    torch.cuda.synchronize()
    rng = np.random.default_rng(7)
    is_f32 = w.dtype == "f32"
    root, pool = root.cpu().numpy(), pool.cpu().numpy()
    for t in range(min(T, 2)):
        rows = []
        for mm in range(w.n_heads + 1):
            ids = list(rng.integers(0, w.vocab, size=24))
            ids += [int(root[t])] if mm == 0 else [int(x) for x in pool[t, mm - 1]]
            rows += [(mm, int(i)) for i in ids]
        # copy just the touched weights to the host
        want = oheads.head_logit_rows(gu.to64(h[t]), lambda kk: gu.to64(w1[kk]),
                                      lambda kk, vv: gu.to64(w2[kk, vv]), lambda vv: gu.to64(w_lm[vv]), rows)
        got = np.array([float(logits[t, mm, v]) for mm, v in rows])
        gu.float_parity(got, want, is_f32, f"{name} sampled head logits")
        # top-k exactness on the kernel's own fp32 logits; oracle ranks agree up to near ties
        gl = logits[t].cpu().numpy().astype(np.float64)
        assert root[t] == np.lexsort((np.arange(w.vocab), -gl[0]))[0]
        for k in range(w.n_heads):
            assert list(pool[t, k]) == list(np.lexsort((np.arange(w.vocab), -gl[1 + k]))[:w.topk])
    del w1, w2, w_lm
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["llama3-8b-256", "longctx-341"])
def test_heads_all_rows_full_size_sampled(m, name):
    """The all-rows variant (every tree row a hidden row: 256 and 341 rows, one and two
    wide tensor-core passes of up to 256 rows) on the full weights: sampled logits of
    rows in every pass against the fp64 oracle, and the top-k of every sampled row exact
    on the kernel's own logits."""
    w = synth.WORKLOADS[name]
    t_o, _, _ = templates(m, w)
    T = t_o.n_rows
    _, w1, w2, w_lm = synth.head_weights(w, device="cuda")
    h = synth.normal((T, w.hidden), 1.0, w.seed, "h", "cuda", w.torch_dtype, sub=1)
    logits = torch.empty((T, w.n_heads + 1, w.vocab), dtype=torch.float32, device="cuda")
    root, pool = m.medusa_heads_topk(h, w1, w2, w_lm, w.topk, logits_out=logits)
    torch.cuda.synchronize()
    rng = np.random.default_rng(11)
    root, pool = root.cpu().numpy(), pool.cpu().numpy()
    for t in sorted({0, 127, 128, min(255, T - 1), min(256, T - 1), T - 1}):
        rows = []
        for mm in range(w.n_heads + 1):
            ids = list(rng.integers(0, w.vocab, size=8))
            ids += [int(root[t])] if mm == 0 else [int(x) for x in pool[t, mm - 1]]
            rows += [(mm, int(i)) for i in ids]
        want = oheads.head_logit_rows(gu.to64(h[t]), lambda kk: gu.to64(w1[kk]),
                                      lambda kk, vv: gu.to64(w2[kk, vv]), lambda vv: gu.to64(w_lm[vv]), rows)
        got = np.array([float(logits[t, mm, v]) for mm, v in rows])
        gu.float_parity(got, want, False, f"{name} all-rows sampled head logits, row {t}")
        gl = logits[t].cpu().numpy().astype(np.float64)
        assert root[t] == np.lexsort((np.arange(w.vocab), -gl[0]))[0]
        for k in range(w.n_heads):
            assert list(pool[t, k]) == list(np.lexsort((np.arange(w.vocab), -gl[1 + k]))[:w.topk])
    del w1, w2, w_lm, logits
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", synth.WORKLOAD_ORDER)
def test_attention_full_size_sampled(m, name):
    w = synth.WORKLOADS[name]
    t_o, t_g, _ = templates(m, w)
    N = t_o.n_rows
    lengths = synth.prefix_lengths(w)
    q, k, v = synth.tree_qkv(w, N, device="cuda")
    paged = w.page_size > 0
    if paged:
        K, V, bt, lay, ks, vs = gu.paged_cache(w, lengths, N, fill_tail=float("nan"))
        cache = m.KVCache(K, V, block_table=bt)
    else:
        K, V, ks, vs = gu.contiguous_cache(w, lengths, N, fill_tail=float("nan"))
        cache = m.KVCache(K, V)
    out, lse, status = m.medusa_tree_attn_verify(t_g, q, k, v, cache, gu.device_tensor(lengths, torch.int32),
                                                 int(lengths.max()), rope_base=w.rope_base, want_lse=True)
    torch.cuda.synchronize()
    assert (status.cpu().numpy() == 0).all()
    assert torch.isfinite(out).all()
    rng = np.random.default_rng(11)
    is_f32 = w.dtype == "f32"
    g = w.group
    got, want = [], []
    for b in range(w.batch):
        L = int(lengths[b])
        for _ in range(6 if w.batch > 1 else 24):
            u = int(rng.integers(0, N))
            hq = int(rng.integers(0, w.n_q_heads))
            kv = hq // g
            o, l = oatt.node_attention_rows(gu.to64(q[b, u, hq]), gu.to64(k[b, :, kv]), gu.to64(v[b, :, kv]),
                                            gu.to64(ks[b][kv]), gu.to64(vs[b][kv]), L, t_o.depth, t_o.mask[u], u,
                                            w.rope_base)
            got.append(gu.to64(out[b, u, hq]))
            want.append(o)
    gu.float_parity(np.stack(got), np.stack(want), is_f32, f"{name} sampled attention")


@pytest.mark.parametrize("name", synth.WORKLOAD_ORDER)
def test_accept_full_size(m, name):
    w = synth.WORKLOADS[name]
    t_o, t_g, acc = templates(m, w)
    N = t_o.n_rows
    root, pool = synth.random_pool(w)
    tokens = np.stack([oround.tree_fill(t_o, root[b], pool[b], 0)[0] for b in range(w.batch)])
    logits = synth.target_logits(w, N)
    if w.plant:
        synth.plant_argmax(logits, pool, t_o.depth, acc, synth.plant_uniforms(w, N))
    ld = logits.cuda()
    for mode in w.accept:
        r = m.medusa_tree_accept(t_g, ld, gu.device_tensor(tokens, torch.int32), mode,
                                 epsilon=w.epsilon, delta=w.delta)
        r = {kk: vv.cpu().numpy() for kk, vv in r.items()}
        skipped = 0
        for b in range(w.batch):
            o = oacc.accept(gu.to64(logits[b]), tokens[b], t_o.retrieve, mode, 1.0, w.epsilon, w.delta)
            if mode == "typical" and gu.typical_ambiguous(o):
                skipped += 1
                continue
            G = o.accept_len + 1
            assert r["accept_len"][b] == o.accept_len
            assert r["best_path"][b] == o.best_path
            assert list(r["out_rows"][b, :G]) == list(o.out_rows)
            assert list(r["out_tokens"][b, :G]) == list(o.out_tokens)
            assert r["frontier_row"][b] == o.frontier_row
        assert skipped <= max(1, w.batch // 8)


@pytest.mark.parametrize("name", synth.WORKLOAD_ORDER)
def test_compact_full_size(m, name):
    w = synth.WORKLOADS[name]
    t_o, t_g, _ = templates(m, w)
    N = t_o.n_rows
    lengths = synth.prefix_lengths(w)
    paged = w.page_size > 0
    if paged:
        K, V, bt, lay, _, _ = gu.paged_cache(w, lengths, N)
        cache = m.KVCache(K, V, block_table=bt)
    else:
        K, V, _, _ = gu.contiguous_cache(w, lengths, N)
        cache = m.KVCache(K, V)
    gen = torch.Generator(device="cuda").manual_seed(3)
    K.copy_(torch.randn(K.shape, generator=gen, device="cuda").to(K.dtype))
    V.copy_(torch.randn(V.shape, generator=gen, device="cuda").to(V.dtype))
    rng = np.random.default_rng(5)
    W = t_o.max_depth + 1
    rows = np.full((w.batch, W), -1, dtype=np.int32)
    alen = np.zeros(w.batch, dtype=np.int32)
    for b in range(w.batch):
        nodes = [x for x in t_o.retrieve[int(rng.integers(0, t_o.n_paths))] if x >= 0]
        alen[b] = len(nodes) - 1
        rows[b, :len(nodes)] = nodes
    Ks, Vs = K.clone(), V.clone()
    L_out, status = m.medusa_kv_compact(cache, t_g, gu.device_tensor(lengths, torch.int32),
                                        gu.device_tensor(alen, torch.int32), gu.device_tensor(rows, torch.int32))
    torch.cuda.synchronize()
    assert (status.cpu().numpy() == 0).all()
    assert list(L_out.cpu().numpy()) == list(lengths + alen + 1)
    for b in range(w.batch):
        L, G = int(lengths[b]), int(alen[b]) + 1
        span = range(L, L + N)
        if paged:
            btc = bt.cpu()
            kb = np.stack([gu.to64(gu.read_paged_row(Ks, btc, b, r)) for r in span], 1)
            vb = np.stack([gu.to64(gu.read_paged_row(Vs, btc, b, r)) for r in span], 1)
            ka = np.stack([gu.to64(gu.read_paged_row(K, btc, b, r)) for r in span], 1)
            va = np.stack([gu.to64(gu.read_paged_row(V, btc, b, r)) for r in span], 1)
        else:
            kb, vb = gu.to64(Ks[b, :, L:L + N]), gu.to64(Vs[b, :, L:L + N])
            ka, va = gu.to64(K[b, :, L:L + N]), gu.to64(V[b, :, L:L + N])
        ocomp.kv_compact(kb, vb, 0, rows[b, :G])
        assert (ka == kb).all() and (va == vb).all()
