"""The whole verify round on the GPU against the oracle's round, on every workload at
full size, element by element.

The GPU side is the library's round graph (medusa_round_create / medusa_round_launch:
heads -> fill -> attention -> acceptance -> compaction recorded once and replayed), the
launch configuration the benchmark times.  The oracle side composes the same five
oracle steps as oracle.round.run_sequence does, per sequence, on the same seeded
inputs ([M7.2] §0x07A round order; [CN] "Mask、位置和 KV 必须一起验证": mask, positions
and K/V are checked together).  The heads run through gu.oracle_heads_blocked because
the fp64 weights of the larger workloads do not fit in host memory at once.

Checked:
  - head logits [T, K+1, V] of every workload within the parity bar (a separate
    medusa_heads_topk call with logits_out), root and pools bit-exact against the
    oracle's top-k (the c19 rule: a differing rank must be a near tie of the fp64
    values, which reseeds the round; reseeds are counted and bounded);
  - tokens and positions bit-exact;
  - the whole attention output [B, N, Hq, dh] within the parity bar;
  - best path, accepted length, published rows and tokens, frontier row bit-exact
    (typical decisions within 1e-5 of their threshold are excluded and counted);
  - L_out, and every cache row [0, L + N) of every sequence after compaction: prefix
    rows unchanged, published rows and the remaining staged rows against the oracle's
    cache (K rotated: within bf16 rounding; V: exact).
"""
import numpy as np
import pytest
import torch

import synth
from oracle import accept as oacc
from oracle import attention as oatt
from oracle import compact as ocomp
from oracle import round as oround
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    import medusa_speculative_tree_gb300 as m
    from medusa_speculative_tree_gb300 import build
    build.build()
    return m


def cache_rows(K, V, bt, b, n_rows, paged):
    """[Hkv, n_rows, dh] float64 copies of cache rows 0 .. n_rows - 1 of sequence b."""
    if paged:
        ps = K.shape[2]
        nb = (n_rows + ps - 1) // ps
        pages = bt[b, :nb].long()
        flat = lambda X: X[pages].permute(1, 0, 2, 3).reshape(X.shape[1], nb * ps, X.shape[3])[:, :n_rows]
        return gu.to64(flat(K)), gu.to64(flat(V))
    return gu.to64(K[b, :, :n_rows]), gu.to64(V[b, :, :n_rows])


@pytest.mark.parametrize("name", synth.WORKLOAD_ORDER)
def test_full_round_against_oracle(m, name):
    w = synth.WORKLOADS[name]
    acc = synth.rank_accuracy(w.n_heads, 10)
    t_o = oround.template_for(w.template, w.topk, w.n_heads, acc)
    t_g = m.Template(t_o.paths[1:], w.topk, w.n_heads, device="cuda")
    N, B = t_o.n_rows, w.batch
    is_f32 = w.dtype == "f32"
    paged = w.page_size > 0
    lengths = synth.prefix_lengths(w)
    _, w1, w2, w_lm = synth.head_weights(w, device="cuda")
    q, k, v = synth.tree_qkv(w, N, device="cuda")
    if paged:
        K, V, bt, _, ks, vs = gu.paged_cache(w, lengths, N)
        cache = m.KVCache(K, V, block_table=bt)
    else:
        K, V, ks, vs = gu.contiguous_cache(w, lengths, N)
        bt = None
        cache = m.KVCache(K, V)
    K0, V0 = K.clone(), V.clone()
    Ld = gu.device_tensor(lengths, torch.int32)

    # Frontier rows: the workload's h, reseeded (sub 1, 2, ...) when an fp32 and an fp64
    # top-k disagree on a near tie.
    reseeds = 0
    for sub in range(3):
        h = synth.normal((B, w.hidden), 1.0, w.seed, "h", "cuda", w.torch_dtype, sub=sub)
        o_root, o_pool, o_logits = gu.oracle_heads_blocked(h, w1, w2, w_lm, w.topk)
        g_logits = torch.empty((B, w.n_heads + 1, w.vocab), dtype=torch.float32, device="cuda")
        g_root, g_pool = m.medusa_heads_topk(h, w1, w2, w_lm, w.topk, logits_out=g_logits)
        torch.cuda.synchronize()
        gu.float_parity(g_logits, o_logits, is_f32, f"{name} head logits")
        g_root, g_pool = g_root.cpu().numpy(), g_pool.cpu().numpy()
        same = (g_root == o_root).all() and (g_pool == o_pool).all()
        if same:
            break
        for b in range(B):                      # a differing rank must be a near tie
            gu.topk_parity([g_root[b]], o_logits[b, 0], 1, 1e-4)
            for kk in range(w.n_heads):
                gu.topk_parity(g_pool[b, kk], o_logits[b, 1 + kk], w.topk, 1e-4)
        reseeds += 1
    assert same, f"{name}: pools still differ after {reseeds} reseeds"
    assert reseeds <= 1

    # target logits, argmax planted on the proposed candidates (the same pool on both sides)
    logits = synth.target_logits(w, N)
    if w.plant:
        synth.plant_argmax(logits, o_pool, t_o.depth, acc, synth.plant_uniforms(w, N))
    mode = w.accept[0]
    rnd = m.MedusaRound(t_g, h, w1, w2, w_lm, w.topk, Ld, q, k, v, cache, int(lengths.max()),
                        logits.to("cuda"), mode=mode, rope_base=w.rope_base, epsilon=w.epsilon,
                        delta=w.delta, want_lse=True)
    K.copy_(K0)
    V.copy_(V0)                                 # creation leaves the cache as it was; be explicit
    rnd.launch()
    torch.cuda.synchronize()
    assert (rnd.attn_status.cpu().numpy() == 0).all()
    assert (rnd.root.cpu().numpy() == o_root).all() and (rnd.pool.cpu().numpy() == o_pool).all()

    skipped = 0
    g_out = rnd.out
    for b in range(B):
        L = int(lengths[b])
        tokens, pos = oround.tree_fill(t_o, o_root[b], o_pool[b], L)
        assert (rnd.tokens[b].cpu().numpy() == tokens).all() and (rnd.pos[b].cpu().numpy() == pos).all()
        ck = np.zeros((w.n_kv_heads, L + N, w.head_dim))
        cv = np.zeros_like(ck)
        ck[:, :L], cv[:, :L] = gu.to64(ks[b]), gu.to64(vs[b])
        o_out, o_lse, kr = oatt.tree_attention(gu.to64(q[b]), gu.to64(k[b]), gu.to64(v[b]), ck, cv, L,
                                               t_o.depth, t_o.mask, w.rope_base)
        gu.float_parity(g_out[b], o_out, is_f32, f"{name} attention output, sequence {b}")
        gu.float_parity(rnd.lse[b], o_lse, True if is_f32 else False, f"{name} lse, sequence {b}")
        ck[:, L:L + N] = np.transpose(kr, (1, 0, 2))
        cv[:, L:L + N] = np.transpose(gu.to64(v[b]), (1, 0, 2))
        o = oacc.accept(gu.to64(logits[b]), tokens, t_o.retrieve, mode, 1.0, w.epsilon, w.delta)
        if mode == "typical" and gu.typical_ambiguous(o):
            skipped += 1
            continue
        G = o.accept_len + 1
        assert int(rnd.accept_len[b]) == o.accept_len, (name, b)
        assert int(rnd.best_path[b]) == o.best_path
        assert list(rnd.out_rows[b, :G].cpu().numpy()) == list(o.out_rows)
        assert list(rnd.out_tokens[b, :G].cpu().numpy()) == list(o.out_tokens)
        assert int(rnd.frontier_row[b]) == o.frontier_row
        new_len = ocomp.kv_compact(ck, cv, L, o.out_rows)
        assert int(rnd.L_out[b]) == new_len and int(rnd.compact_status[b]) == 0
        gk, gv = cache_rows(K, V, bt, b, L + N, paged)
        assert (gk[:, :L] == ck[:, :L]).all() and (gv[:, :L] == cv[:, :L]).all()    # prefix untouched
        tol = 1e-6 if is_f32 else 2.0 ** -8                                           # one rounding of K'
        dk = np.abs(gk[:, L:] - ck[:, L:])
        assert (dk <= tol * np.maximum(np.abs(ck[:, L:]), 1.0)).all(), f"{name} committed K, sequence {b}"
        assert (gv[:, L:] == cv[:, L:]).all(), f"{name} committed V, sequence {b}"
    assert skipped <= max(1, B // 8)
    if w.plant:
        assert int(rnd.accept_len.max()) > 0            # planted argmaxes are accepted somewhere
    rnd.close()
    print(f"{name}: reseeds {reseeds}, typical decisions excluded {skipped}")
