"""Per-sequence templates and trees built on the GPU.

[M7.2] §0x07D leaves a batch whose sequences verify different trees to continuous
batching, and [CN] "局限与适用场景" notes that the best tree size moves with the context
length; the library takes
one template per sequence (a TemplateBatch: the shared descriptor's counts become
bounds and each sequence reads its own template from device memory), and builds the
greedy tree of each sequence's rank accuracies on the GPU
(medusa_tree_greedy_device).

Checked here:
  - the device builder against the oracle's greedy search and compiler
    ([M7.2] §0x04C, [PartII] Part 3): every template array bit-exact, on the
    workloads' accuracy tables, on random tables, on tables with exact weight ties
    and on a table with a value outside [0, 1] (root-only template, MEDUSA_EINVAL);
  - the whole round (heads, fill, attention, acceptance, compaction) on the
    serving batch with two different greedy trees in one batch, against the
    oracle's round of each sequence with its own template; the same through the
    round graph.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import accept as oacc
from oracle import attention as oatt
from oracle import compact as ocomp
from oracle import round as oround
from oracle import tree as otree
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    import medusa_speculative_tree_gb300 as m
    from medusa_speculative_tree_gb300 import build
    build.build()
    return m


def compare_arrays(g, t_o):
    """Device-built template arrays against the oracle's compile of the same paths."""
    N = t_o.n_rows
    assert g["n_rows"] == N and g["max_depth"] == t_o.max_depth and g["n_paths"] == t_o.n_paths
    assert (g["slot"] == t_o.slot).all() and (g["depth"] == t_o.depth).all() and (g["parent"] == t_o.parent).all()
    assert (g["retrieve"] == t_o.retrieve).all()
    kids = np.zeros(N, dtype=int)
    for u in range(1, N):
        kids[t_o.parent[u]] += 1
    internal = [u for u in range(N) if kids[u] > 0]
    assert list(g["internal"]) == internal and g["n_internal"] == len(internal)
    assert list(g["internal_index"]) == [internal.index(u) if kids[u] else -1 for u in range(N)]
    for u in range(N):
        bits = [(int(g["anc"][u, v // 64]) >> (v % 64)) & 1 for v in range(N)]
        assert bits == list(t_o.mask[u].astype(int)), u


def alt_accuracy(n_heads, n_ranks):
    """A second synthetic table, a_k^(i) = 0.9 * 0.85^(k-1) * 0.3^(i-1) (multiplied left to
    right like synth.rank_accuracy): heads that stay accurate deeper, ranks that fall off
    faster, so its greedy 64-row tree is deep and narrow (depth counts 5, 10, 20, 28
    against the workload's 7, 21, 30, 5)."""
    acc = np.empty((n_heads, n_ranks))
    hf = 0.9
    for k in range(n_heads):
        rf = hf
        for i in range(n_ranks):
            acc[k, i] = rf
            rf = rf * 0.3
        hf = hf * 0.85
    return acc


def random_tables(B, K, R, seed):
    rng = np.random.default_rng(seed)
    tabs = []
    for b in range(B):
        if b % 3 == 0:       # quantised values: many exact weight ties
            t = rng.integers(1, 5, size=(K, R)) / 5.0
        else:
            t = np.sort(rng.uniform(0.0, 1.0, size=(K, R)), axis=1)[:, ::-1]
        tabs.append(t)
    return np.stack(tabs)


@pytest.mark.parametrize("case", [
    dict(kind="workloads", budget=63, K=4, R=10, topk=10),
    dict(kind="workloads", budget=255, K=4, R=10, topk=10),
    dict(kind="random", budget=40, K=3, R=6, topk=8, B=9),
    dict(kind="random", budget=120, K=5, R=4, topk=4, B=6),
    dict(kind="random", budget=1, K=2, R=3, topk=3, B=2),
    dict(kind="random", budget=0, K=2, R=3, topk=3, B=2),
    dict(kind="random", budget=500, K=2, R=3, topk=3, B=2),       # every path of depth <= 2 taken (12)
])
def test_device_greedy_tree_matches_oracle(m, case):
    K, R, budget, topk = case["K"], case["R"], case["budget"], case["topk"]
    if case["kind"] == "workloads":
        tabs = np.stack([synth.rank_accuracy(K, R), alt_accuracy(K, R)])
    else:
        tabs = random_tables(case["B"], K, R, seed=budget + 7 * K)
    acc = torch.tensor(tabs, dtype=torch.float64, device="cuda")
    batch, status = m.medusa_tree_greedy_device(acc, budget, topk)
    torch.cuda.synchronize()
    assert (status.cpu().numpy() == 0).all()
    for b in range(tabs.shape[0]):
        paths = otree.greedy_tree(tabs[b], budget)
        t_o = otree.compile_template(paths, topk, K)
        compare_arrays(m.batch_template_arrays(batch, b), t_o)
    assert batch.n_rows == budget + 1


def test_device_greedy_tree_rejects_bad_table(m):
    tabs = np.stack([synth.rank_accuracy(3, 4), synth.rank_accuracy(3, 4)])
    tabs[1, 2, 1] = 1.5                       # outside [0, 1]
    acc = torch.tensor(tabs, dtype=torch.float64, device="cuda")
    batch, status = m.medusa_tree_greedy_device(acc, 10, 4)
    torch.cuda.synchronize()
    assert list(status.cpu().numpy()) == [0, m.api.nat.EINVAL]
    compare_arrays(m.batch_template_arrays(batch, 0), otree.compile_template(otree.greedy_tree(tabs[0], 10), 4, 3))
    g = m.batch_template_arrays(batch, 1)
    assert g["n_rows"] == 1 and g["n_paths"] == 1 and g["max_depth"] == 0 and list(g["retrieve"][0]) == [0]


def run_ragged_round(m, w, tabs, seq_tab, use_graph):
    """The five calls with per-sequence device-built templates against the oracle's round
    of every sequence with its own template."""
    B, N_heads = w.batch, w.n_heads
    budget = w.template[1]
    acc_d = torch.tensor(tabs[seq_tab][:, :, :w.template[2]], dtype=torch.float64, device="cuda")
    batch, st = m.medusa_tree_greedy_device(acc_d, budget, w.topk)
    torch.cuda.synchronize()
    assert (st.cpu().numpy() == 0).all()
    t_os = [oround.template_for(w.template, w.topk, N_heads, tabs[seq_tab[b]]) for b in range(B)]
    NC = batch.n_rows                                     # row stride: the batch bound
    assert NC == max(t.n_rows for t in t_os)
    lengths = synth.prefix_lengths(w)
    h, w1, w2, w_lm = synth.head_weights(w, device="cuda")
    q, k, v = synth.tree_qkv(w, NC, device="cuda")
    paged = w.page_size > 0
    if paged:
        K, V, bt, _, ks, vs = gu.paged_cache(w, lengths, NC)
        cache = m.KVCache(K, V, block_table=bt)
    else:
        K, V, ks, vs = gu.contiguous_cache(w, lengths, NC)
        cache = m.KVCache(K, V)
    Ld = gu.device_tensor(lengths, torch.int32)
    o_root, o_pool, _ = gu.oracle_heads_blocked(h, w1, w2, w_lm, w.topk)
    logits = synth.target_logits(w, NC)
    u01 = synth.plant_uniforms(w, NC)
    for b in range(B):                                   # each sequence planted on its own tree
        synth.plant_argmax(logits[b:b + 1], o_pool[b:b + 1], t_os[b].depth, tabs[seq_tab[b]], u01[b:b + 1])
    mode = w.accept[0]
    if use_graph:
        rnd = m.MedusaRound(batch, h, w1, w2, w_lm, w.topk, Ld, q, k, v, cache, int(lengths.max()),
                            logits.cuda(), mode=mode, rope_base=w.rope_base, epsilon=w.epsilon, delta=w.delta)
        rnd.launch()
        torch.cuda.synchronize()
        root, pool, tokens, pos, out = rnd.root, rnd.pool, rnd.tokens, rnd.pos, rnd.out
        attn_status = rnd.attn_status
        r = {"accept_len": rnd.accept_len, "best_path": rnd.best_path, "out_rows": rnd.out_rows,
             "out_tokens": rnd.out_tokens, "frontier_row": rnd.frontier_row}
        L_out, c_status = rnd.L_out, rnd.compact_status
    else:
        root, pool = m.medusa_heads_topk(h, w1, w2, w_lm, w.topk)
        tokens, pos = m.medusa_tree_fill(batch, root, pool, Ld)
        out, _, attn_status = m.medusa_tree_attn_verify(batch, q, k, v, cache, Ld, int(lengths.max()),
                                                        rope_base=w.rope_base)
        r = m.medusa_tree_accept(batch, logits.cuda(), tokens, mode, epsilon=w.epsilon, delta=w.delta)
        L_out, c_status = m.medusa_kv_compact(cache, batch, Ld, r["accept_len"], r["out_rows"])
        torch.cuda.synchronize()
    assert (attn_status.cpu().numpy() == 0).all()
    assert (root.cpu().numpy() == o_root).all() and (pool.cpu().numpy() == o_pool).all()
    accepted = 0
    for b in range(B):
        t_o, L = t_os[b], int(lengths[b])
        Nb = t_o.n_rows
        o_tok, o_pos = oround.tree_fill(t_o, o_root[b], o_pool[b], L)
        assert (tokens[b, :Nb].cpu().numpy() == o_tok).all() and (pos[b, :Nb].cpu().numpy() == o_pos).all()
        assert (tokens[b, Nb:].cpu().numpy() == -1).all()
        ck = np.zeros((w.n_kv_heads, L + Nb, w.head_dim))
        cv = np.zeros_like(ck)
        ck[:, :L], cv[:, :L] = gu.to64(ks[b]), gu.to64(vs[b])
        o_out, _, kr = oatt.tree_attention(gu.to64(q[b, :Nb]), gu.to64(k[b, :Nb]), gu.to64(v[b, :Nb]), ck, cv, L,
                                           t_o.depth, t_o.mask, w.rope_base)
        gu.float_parity(out[b, :Nb], o_out, w.dtype == "f32", f"ragged attention, sequence {b}")
        ck[:, L:L + Nb] = np.transpose(kr, (1, 0, 2))
        cv[:, L:L + Nb] = np.transpose(gu.to64(v[b, :Nb]), (1, 0, 2))
        o = oacc.accept(gu.to64(logits[b, :Nb]), o_tok, t_o.retrieve, mode, 1.0, w.epsilon, w.delta)
        G = o.accept_len + 1
        assert int(r["accept_len"][b]) == o.accept_len and int(r["best_path"][b]) == o.best_path
        assert list(r["out_rows"][b, :G].cpu().numpy()) == list(o.out_rows)
        assert list(r["out_tokens"][b, :G].cpu().numpy()) == list(o.out_tokens)
        assert int(r["frontier_row"][b]) == o.frontier_row
        accepted += o.accept_len
        new_len = ocomp.kv_compact(ck, cv, L, o.out_rows)
        assert int(L_out[b]) == new_len and int(c_status[b]) == 0
        if paged:
            nb_ = (L + Nb + 15) // 16
            pages = bt[b, :nb_].long()
            flat = lambda X: X[pages].permute(1, 0, 2, 3).reshape(X.shape[1], nb_ * 16, X.shape[3])[:, :L + Nb]
            gk, gv = gu.to64(flat(K)), gu.to64(flat(V))
        else:
            gk, gv = gu.to64(K[b, :, :L + Nb]), gu.to64(V[b, :, :L + Nb])
        assert (gk[:, :L] == ck[:, :L]).all() and (gv[:, :L] == cv[:, :L]).all()
        dk = np.abs(gk[:, L:] - ck[:, L:])
        assert (dk <= 2.0 ** -8 * np.maximum(np.abs(ck[:, L:]), 1.0)).all()
        assert (gv[:, L:] == cv[:, L:]).all()
    assert accepted > 0
    return t_os


@pytest.mark.parametrize("use_graph", [False, True])
def test_serving_batch_with_two_trees(m, use_graph):
    """The serving batch (16 sequences, paged cache, shared heads) with two different
    64-row greedy trees: even sequences the workload's table, odd ones another."""
    w = synth.WORKLOADS["serving-b16-paged"]
    tabs = np.stack([synth.rank_accuracy(w.n_heads, 10), alt_accuracy(w.n_heads, 10)])
    seq_tab = np.arange(w.batch) % 2
    t_os = run_ragged_round(m, w, tabs, seq_tab, use_graph)
    assert t_os[0].n_rows == t_os[1].n_rows == 64
    assert not np.array_equal(t_os[0].parent, t_os[1].parent)     # two different trees


def test_ragged_row_counts_small(m):
    """Templates of different sizes in one batch (4, 12 and 21 rows; bf16, GQA,
    contiguous cache): rows past a sequence's own are neither read nor written."""
    w = synth.small_variant(synth.WORKLOADS["llama3-8b-256"], batch=3, prefix_len=300, n_q_heads=8,
                            n_kv_heads=2, hidden=256, vocab=3000, template=("greedy", 20, 4), topk=4)
    tabs = np.stack([synth.rank_accuracy(4, 4), alt_accuracy(4, 4), np.full((4, 4), 0.05)])
    t_os = [otree.compile_template(otree.greedy_tree(tabs[b], bud), 4, 4) for b, bud in enumerate([3, 11, 20])]
    # one batch of host-compiled templates of the three sizes
    t_gs = [m.Template(t.paths[1:], 4, 4, device="cuda") for t in t_os]
    tb = m.TemplateBatch(t_gs, [0, 1, 2])
    assert tb.n_rows == 21
    N = tb.n_rows
    lengths = synth.prefix_lengths(w)
    q, k, v = synth.tree_qkv(w, N, device="cuda")
    K, V, ks, vs = gu.contiguous_cache(w, lengths, N, fill_tail=float("nan"))
    out = torch.full((w.batch, N, w.n_q_heads, w.head_dim), 9.0, device="cuda")
    _, _, status = m.medusa_tree_attn_verify(tb, q, k, v, m.KVCache(K, V), gu.device_tensor(lengths, torch.int32),
                                             int(lengths.max()), rope_base=w.rope_base, out=out)
    torch.cuda.synchronize()
    assert (status.cpu().numpy() == 0).all()
    for b in range(3):
        t_o = t_os[b]
        Nb, L = t_o.n_rows, int(lengths[b])
        o, _, _ = oatt.tree_attention(gu.to64(q[b, :Nb]), gu.to64(k[b, :Nb]), gu.to64(v[b, :Nb]), gu.to64(ks[b]),
                                      gu.to64(vs[b]), L, t_o.depth, t_o.mask, w.rope_base)
        gu.float_parity(out[b, :Nb], o, False, f"attention, {Nb} rows")
        assert (out[b, Nb:] == 9.0).all()                 # rows past the sequence's own: untouched
