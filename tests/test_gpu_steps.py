"""GPU parity of each round step against the fp64 oracle on identical seeded inputs.

Sizes here are ones the oracle finishes in seconds while still spanning several
tiles, a ragged tail, GQA groups, paged caches and the degenerate cases
(root-only tree, empty prefix, deep chains, multiword masks).
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
from oracle import tree as otree
from oracle.round import tree_fill as o_fill
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    import medusa_speculative_tree_gb300 as m
    from medusa_speculative_tree_gb300 import build
    build.build()
    return m


def make_template(m, paths, topk, n_heads=0):
    return m.Template(paths, topk, n_heads, device="cuda"), otree.compile_template(paths, topk)


# ----------------------------------------------------------------------------- fill

@pytest.mark.parametrize("name", synth.WORKLOAD_ORDER)
def test_tree_fill(m, name):
    w = synth.WORKLOADS[name]
    acc = synth.rank_accuracy(w.n_heads, 10)
    from oracle.round import template_for
    t_o = template_for(w.template, w.topk, w.n_heads, acc)
    t_g = m.Template(t_o.paths[1:], w.topk, w.n_heads, device="cuda")
    root, pool = synth.random_pool(w)
    L = synth.prefix_lengths(w)
    tok, pos = m.medusa_tree_fill(t_g, gu.device_tensor(root, torch.int32), gu.device_tensor(pool, torch.int32),
                                  gu.device_tensor(L, torch.int32))
    tok, pos = tok.cpu().numpy(), pos.cpu().numpy()
    for b in range(w.batch):
        wt, wp = o_fill(t_o, root[b], pool[b], L[b])
        assert (tok[b] == wt).all() and (pos[b] == wp).all()


# ----------------------------------------------------------------------------- heads

@pytest.mark.parametrize("case", [
    dict(T=1, d=256, V=1000, K=2, topk=3, dt=torch.float32),
    dict(T=1, d=512, V=5003, K=4, topk=10, dt=torch.bfloat16),
    dict(T=1, d=6144, V=3001, K=3, topk=10, dt=torch.bfloat16),   # weight stream, rows in two halves
    dict(T=3, d=1024, V=4000, K=3, topk=10, dt=torch.bfloat16),
    dict(T=16, d=4096, V=2048, K=2, topk=10, dt=torch.bfloat16),
    dict(T=128, d=256, V=1000, K=2, topk=5, dt=torch.bfloat16),   # tensor-core stream, one pass of pairs
    dict(T=150, d=256, V=1000, K=2, topk=5, dt=torch.bfloat16),   # one wide pass (single rows, fp16 z)
    dict(T=300, d=512, V=777, K=3, topk=8, dt=torch.bfloat16),    # two wide passes, ragged vocabulary group
    dict(T=5, d=128, V=300, K=1, topk=32, dt=torch.float32),
])
def test_heads_topk(m, case):
    T, d, V, K, topk, dt = case["T"], case["d"], case["V"], case["K"], case["topk"], case["dt"]
    seed = 77 + T + d
    h = synth.normal((T, d), 1.0, seed, "h", dtype=dt)
    w1 = synth.normal((K, d, d), 0.02, seed, "w1", dtype=dt)
    w2 = synth.normal((K, V, d), 1 / math.sqrt(d), seed, "w2", dtype=dt)
    w_lm = synth.normal((V, d), 1 / math.sqrt(d), seed, "w_lm", dtype=dt)
    logits = torch.empty((T, K + 1, V), dtype=torch.float32, device="cuda")
    root, pool = m.medusa_heads_topk(h.cuda(), w1.cuda(), w2.cuda(), w_lm.cuda(), topk, logits_out=logits)
    o_root, o_pool, o_logits = oheads.medusa_heads(gu.to64(h), gu.to64(w1), gu.to64(w2), gu.to64(w_lm), topk)
    gu.float_parity(logits, o_logits, dt == torch.float32, "head logits")
    root, pool = root.cpu().numpy(), pool.cpu().numpy()
    # Near ties the fp32 and fp64 rankings may order differently.  Pairs (T <= 128) keep z
    # to ~2^-16, so logits agree to ~1e-5.  Wide passes (T > 128) keep z in fp16: each
    # element carries a relative rounding of at most 2^-11, so a logit errs by about
    # 2^-11 / sqrt(3) * ||W2 o z||_2 ~ 3e-4 (std) here, and ranks within 4e-3 are near ties.
    tol = 4e-3 if (dt == torch.bfloat16 and T > 128) else 1e-4
    for t in range(T):
        gu.topk_parity([root[t]], o_logits[t, 0], 1, tol=tol)
        for k in range(K):
            gu.topk_parity(pool[t, k], o_logits[t, 1 + k], topk, tol=tol)
        # the top-k kernel itself is exact on its own fp32 inputs
        gl = logits[t].cpu().numpy().astype(np.float64)
        assert root[t] == np.lexsort((np.arange(V), -gl[0]))[0]
        for k in range(K):
            assert list(pool[t, k]) == list(np.lexsort((np.arange(V), -gl[1 + k]))[:topk])


def test_heads_shared_projection_and_bias(m):
    T, d, V, K, topk = 2, 256, 777, 3, 5
    s = 5
    h = synth.normal((T, d), 1.0, s, "h")
    w1 = synth.normal((K, d, d), 0.05, s, "w1")
    b1 = synth.normal((K, d), 0.5, s, "b1")
    w_lm = synth.normal((V, d), 0.1, s, "w_lm")
    logits = torch.empty((T, K + 1, V), dtype=torch.float32, device="cuda")
    root, pool = m.medusa_heads_topk(h.cuda(), w1.cuda(), w_lm.cuda(), w_lm.cuda(), topk, b1=b1.cuda(),
                                     logits_out=logits, shared_w2=True)
    _, _, o_logits = oheads.medusa_heads(gu.to64(h), gu.to64(w1), gu.to64(w_lm), gu.to64(w_lm), topk,
                                         b1=gu.to64(b1))
    gu.float_parity(logits, o_logits, True, "shared-projection logits")


# ----------------------------------------------------------------------------- attention

def same_as_mirror(cache):
    """The fp16 mirror holds fp16(bf16 value) of every cache element (NaN where NaN)."""
    for c16, c in ((cache.k_f16, cache.k), (cache.v_f16, cache.v)):
        want = c.to(torch.float16)
        assert bool(((c16 == want) | (c16.isnan() & want.isnan())).all())


def attn_case(m, w, paths, lengths, paged=False, fill_tail=0.0, want_lse=True, mirror=False):
    """Run GPU tree attention and the dense oracle on the same inputs (with mirror, on a
    bf16 cache carrying an fp16 mirror, which must again mirror the cache afterwards)."""
    t_g, t_o = make_template(m, paths, w.topk)
    N = t_o.n_rows
    q, k, v = synth.tree_qkv(w, N)
    if paged:
        K, V, bt, lay, ks, vs = gu.paged_cache(w, lengths, N, fill_tail=fill_tail)
        cache = m.KVCache(K, V, block_table=bt)
    else:
        K, V, ks, vs = gu.contiguous_cache(w, lengths, N, fill_tail=fill_tail)
        cache = m.KVCache(K, V)
    if mirror:
        cache.add_mirror()
    Ld = gu.device_tensor(lengths, torch.int32)
    out, lse, status = m.medusa_tree_attn_verify(t_g, q.cuda(), k.cuda(), v.cuda(), cache, Ld,
                                                 int(max(lengths)), rope_base=w.rope_base, want_lse=want_lse)
    torch.cuda.synchronize()
    assert (status.cpu().numpy() == 0).all()
    if mirror:
        same_as_mirror(cache)
    is_f32 = w.dtype == "f32"
    for b, L in enumerate(lengths):
        o_out, o_lse, o_kr = oatt.tree_attention(gu.to64(q[b]), gu.to64(k[b]), gu.to64(v[b]), gu.to64(ks[b]),
                                                 gu.to64(vs[b]), int(L), t_o.depth, t_o.mask, w.rope_base)
        gu.float_parity(out[b], o_out, is_f32, f"attn out b={b}")
        if want_lse:
            gu.float_parity(lse[b], o_lse, True if is_f32 else False, f"lse b={b}")
        # staged rows L + u hold the rotated tree keys and the tree values
        for u in range(N):
            if paged:
                krow = gu.read_paged_row(K, bt.cpu(), b, int(L) + u)
                vrow = gu.read_paged_row(V, bt.cpu(), b, int(L) + u)
            else:
                krow, vrow = K[b, :, int(L) + u], V[b, :, int(L) + u]
            kk, vv = gu.to64(krow), gu.to64(vrow)
            tol = 1e-6 if is_f32 else 2.0 ** -8
            assert np.all(np.abs(kk - o_kr[u]) <= tol * np.maximum(np.abs(o_kr[u]), 1.0))
            assert (vv == gu.to64(v[b, u])).all()
    return out


def test_attn_tiny_fp32(m):
    w = synth.WORKLOADS["tiny-fp32"]
    attn_case(m, w, otree.regular_paths((2, 3)), synth.prefix_lengths(w))


@pytest.mark.parametrize("dt", ["f32", "bf16", "bf16+mirror"])
@pytest.mark.parametrize("L", [0, 1, 37, 300])
def test_attn_ragged_prefix_gqa(m, dt, L):
    w = synth.small_variant(synth.WORKLOADS["llama3-8b-256"], dtype=dt.split("+")[0], prefix_len=L, seed=2000 + L)
    acc = synth.rank_accuracy(4, 10)
    attn_case(m, w, otree.greedy_tree(acc, 40), synth.prefix_lengths(w), mirror=dt.endswith("mirror"))


def test_attn_root_only_and_deep_chain(m):
    w = synth.small_variant(synth.WORKLOADS["vicuna7b-64"], n_q_heads=4, n_kv_heads=4, prefix_len=129,
                            seed=31)
    attn_case(m, w, [], synth.prefix_lengths(w))
    chain = [tuple([0] * t) for t in range(1, 17)]
    attn_case(m, w, chain, synth.prefix_lengths(w))


@pytest.mark.parametrize("dh", [64, 128])
def test_attn_fp32_deep_chain_and_multiword_mask(m, dh):
    """The CUDA-core kernel (fp32) where a row has many ancestors: a 16-deep chain (17
    ancestor-or-self rows, read in groups of four with a partial last group) and the
    341-row Cartesian tree (six mask words, ancestors spread over several words), with
    NaN in the cache rows past L + N."""
    w = synth.small_variant(synth.WORKLOADS["longctx-341"], dtype="f32", n_q_heads=4, n_kv_heads=2,
                            head_dim=dh, prefix_len=150, seed=61 + dh)
    chain = [tuple([0] * t) for t in range(1, 17)]
    attn_case(m, w, chain, synth.prefix_lengths(w), fill_tail=float("nan"))
    attn_case(m, w, otree.regular_paths((4, 4, 4, 4)), synth.prefix_lengths(w), fill_tail=float("nan"))


@pytest.mark.parametrize("mirror", [False, True])
def test_attn_multiword_mask_and_nan_tail(m, mirror):
    """341 rows (six 64-bit mask words); cache rows past L + N hold NaN and must stay unread."""
    w = synth.small_variant(synth.WORKLOADS["longctx-341"], n_q_heads=16, n_kv_heads=2, prefix_len=200, seed=41)
    attn_case(m, w, otree.regular_paths((4, 4, 4, 4)), synth.prefix_lengths(w), fill_tail=float("nan"),
              mirror=mirror)


@pytest.mark.parametrize("mirror", [False, True])
def test_attn_paged_batch(m, mirror):
    w = synth.small_variant(synth.WORKLOADS["serving-b16-paged"], batch=4, prefix_range=(20, 700), seed=51)
    acc = synth.rank_accuracy(4, 10)
    attn_case(m, w, otree.greedy_tree(acc, 63), synth.prefix_lengths(w), paged=True, fill_tail=float("nan"),
              mirror=mirror)


@pytest.mark.parametrize("shape", ["1,2", "1,4", "2,2"])
@pytest.mark.parametrize("splits", [1, 2, 3, 5, 8])
def test_attn_every_shape_and_split_count(m, monkeypatch, shape, splits):
    """The tensor-core kernel in each of its shapes (query tiles per CTA, stages) and at
    several split counts, on a paged GQA batch of ragged lengths with a NaN tail: the
    splits' cluster merge and the per-sequence spreading of tiles over them (with an
    fp16 mirror at odd split counts)."""
    monkeypatch.setenv("MEDUSA_ATTN_TC_SHAPE", shape)
    monkeypatch.setenv("MEDUSA_ATTN_TC_SPLITS", str(splits))
    w = synth.small_variant(synth.WORKLOADS["serving-b16-paged"], batch=3, seed=700 + splits)
    acc = synth.rank_accuracy(4, 10)
    lengths = np.array([1337, 3, 650])   # 21 / 1 / 11 tiles of 64 keys: some splits get none
    attn_case(m, w, otree.greedy_tree(acc, 63), lengths, paged=True, fill_tail=float("nan"), mirror=splits % 2 == 1)


@pytest.mark.parametrize("shape", ["1,2", "2,2"])
@pytest.mark.parametrize("splits", [1, 3])
def test_attn_rising_scores_rescale(m, monkeypatch, shape, splits):
    """Prefix scores that rise by about 12 (log2 units) every 64 keys: the row max of every
    half of a 128-key tile exceeds the running reference by more than 2^8, so the online
    softmax raises its reference again and again (rescaling O, l and, in the second half
    of a tile, the P already written).  The rise comes from dimension 63 of the queries
    and prefix keys (the lowest-frequency rotary pair, which barely turns at these
    positions); the last keys dominate the tree block, and the scores stay small enough
    for the fp16 operands."""
    monkeypatch.setenv("MEDUSA_ATTN_TC_SHAPE", shape)
    monkeypatch.setenv("MEDUSA_ATTN_TC_SPLITS", str(splits))
    w = synth.small_variant(synth.WORKLOADS["llama3-8b-256"], batch=2, n_q_heads=8, n_kv_heads=2,
                            prefix_len=700, seed=77)
    acc = synth.rank_accuracy(4, 10)
    t_g, t_o = make_template(m, otree.greedy_tree(acc, 40), w.topk)
    N = t_o.n_rows
    lengths = np.array([704, 700])
    q, k, v = synth.tree_qkv(w, N)
    ks, vs = synth.prefix_kv(w, lengths)
    c = w.head_dim ** -0.5 * np.log2(np.e)               # score (log2 units) per unit of q . k
    q[..., 63], q[..., 127] = 8.0, 0.0
    for b, L in enumerate(lengths):
        level = -112.0 + 12.0 * (np.arange(L) // 64)      # log2 units, rising per 64 keys to +8
        ks[b][:, :, 63] = torch.as_tensor(level / (8.0 * c), dtype=torch.float64).to(ks[b].dtype)
        ks[b][:, :, 127] = 0.0
    cap = int(lengths.max()) + N + 16
    K = torch.zeros((w.batch, w.n_kv_heads, cap, w.head_dim), dtype=w.torch_dtype)
    V = torch.zeros_like(K)
    for b, L in enumerate(lengths):
        K[b, :, :L], V[b, :, :L] = ks[b], vs[b]
    cache = m.KVCache(K.cuda(), V.cuda())
    out, lse, status = m.medusa_tree_attn_verify(t_g, q.cuda(), k.cuda(), v.cuda(), cache,
                                                 gu.device_tensor(lengths, torch.int32), int(lengths.max()),
                                                 rope_base=w.rope_base, want_lse=True)
    torch.cuda.synchronize()
    assert (status.cpu().numpy() == 0).all()
    for b, L in enumerate(lengths):
        o_out, o_lse, _ = oatt.tree_attention(gu.to64(q[b]), gu.to64(k[b]), gu.to64(v[b]), gu.to64(ks[b]),
                                              gu.to64(vs[b]), int(L), t_o.depth, t_o.mask, w.rope_base)
        gu.float_parity(out[b], o_out, False, f"attn out b={b}")
        gu.float_parity(lse[b], o_lse, False, f"lse b={b}")


@pytest.mark.parametrize("mirror", [False, True])
def test_attn_head_dim_64_bf16(m, mirror):
    """The CUDA-core kernel on a bf16 cache (head_dim 64); with an fp16 mirror its staged
    tree rows must reach the mirror too."""
    w = synth.small_variant(synth.WORKLOADS["vicuna7b-64"], n_q_heads=8, n_kv_heads=2, head_dim=64,
                            prefix_len=513, seed=61)
    attn_case(m, w, otree.regular_paths((3, 2)), synth.prefix_lengths(w), mirror=mirror)


def test_attn_capacity_error_leaves_sequence_alone(m):
    w = synth.small_variant(synth.WORKLOADS["tiny-fp32"], batch=2, seed=71)
    paths = otree.regular_paths((2, 3))
    t_g, _ = make_template(m, paths, w.topk)
    N = t_g.n_rows
    lengths = np.array([64, 64])
    q, k, v = synth.tree_qkv(w, N)
    K, V, _, _ = gu.contiguous_cache(w, lengths, N, guard=0)
    cache = m.KVCache(K, V)
    Ld = gu.device_tensor([64, 66], torch.int32)          # sequence 1 would overflow by 2 rows
    before = K[1].clone()
    out = torch.full((2, N, w.n_q_heads, w.head_dim), 7.0, device="cuda")
    with pytest.raises(Exception):
        m.medusa_tree_attn_verify(t_g, q.cuda(), k.cuda(), v.cuda(), cache, Ld, 66)   # host-visible bound
    _, _, status = m.medusa_tree_attn_verify(t_g, q.cuda(), k.cuda(), v.cuda(), cache, Ld, 64, out=out)
    torch.cuda.synchronize()
    assert list(status.cpu().numpy()) == [0, -2]
    assert torch.equal(K[1], before)
    assert (out[1] == 7.0).all()


def test_attn_workspace_reuse_is_clean(m):
    """Calls of different shapes (split counts and numbers of work units) share one
    workspace: the scratch partials of a small call must never land where a later,
    larger call keeps its ticket counters."""
    w = synth.small_variant(synth.WORKLOADS["llama3-8b-256"], dtype="f32", prefix_len=900, seed=81)
    small = otree.regular_paths((3, 2))
    big = otree.greedy_tree(synth.rank_accuracy(4, 10), 63)
    for L, paths, hq in ((900, small, 8), (40, big, 32), (900, small, 8), (0, big, 16), (511, small, 32),
                         (700, big, 32)):
        wl = synth.small_variant(w, prefix_len=L, n_q_heads=hq)
        attn_case(m, wl, paths, synth.prefix_lengths(wl), want_lse=False)


# ----------------------------------------------------------------------------- acceptance

def test_accept_page_fixtures(m):
    """The nine-row fixtures of the acceptance pins, on the GPU (fp32 logits)."""
    from tests import test_oracle_accept_compact as AC
    g, t_o, tokens = AC.a31()
    t_g = m.Template(t_o.paths[1:], 10, device="cuda")
    for fx, mode, want in [(AC.fixture_one, "greedy", [11, 21, 31]), (AC.fixture_one, "typical", [11, 22, 31]),
                           (AC.fixture_two, "typical", [11, 21, 31])]:
        logits = torch.tensor(fx(), dtype=torch.float32, device="cuda")[None]
        r = m.medusa_tree_accept(t_g, logits, gu.device_tensor(tokens[None], torch.int32), mode)
        G = int(r["accept_len"][0]) + 1
        assert list(r["out_tokens"][0, :G].cpu().numpy()) == want


@pytest.mark.parametrize("mode,guard", [("greedy", False), ("typical", False), ("typical", True)])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_accept_planted(m, mode, guard, dt):
    w = synth.small_variant(synth.WORKLOADS["vicuna7b-64"], batch=6, vocab=5000, dtype=dt, seed=91)
    acc = synth.rank_accuracy(4, 10)
    t_o = otree.compile_template(otree.greedy_tree(acc, 63), 10)
    t_g = m.Template(t_o.paths[1:], 10, device="cuda")
    root, pool = synth.random_pool(w)
    tokens = np.stack([o_fill(t_o, root[b], pool[b], 0)[0] for b in range(w.batch)])
    logits = synth.target_logits(w, t_o.n_rows)
    synth.plant_argmax(logits, pool, t_o.depth, acc, synth.plant_uniforms(w, t_o.n_rows))
    r = m.medusa_tree_accept(t_g, logits.cuda(), gu.device_tensor(tokens, torch.int32), mode,
                             epsilon=w.epsilon, delta=w.delta, entropy_guard=guard)
    r = {k: v.cpu().numpy() for k, v in r.items()}
    lens, skipped = [], 0
    for b in range(w.batch):
        o = oacc.accept(gu.to64(logits[b]), tokens[b], t_o.retrieve, mode, 1.0, w.epsilon, w.delta, guard)
        if mode == "typical" and gu.typical_ambiguous(o):
            skipped += 1          # fp32 and fp64 may legitimately decide this sequence differently
            continue
        assert r["accept_len"][b] == o.accept_len
        G = o.accept_len + 1
        assert list(r["out_rows"][b, :G]) == list(o.out_rows)
        assert list(r["out_tokens"][b, :G]) == list(o.out_tokens)
        assert (r["out_rows"][b, G:] == -1).all()
        assert r["frontier_row"][b] == o.frontier_row
        assert r["best_path"][b] == o.best_path
        lens.append(o.accept_len)
    assert skipped <= 1
    assert max(lens) > 0          # planting produced accepted edges


@pytest.mark.parametrize("mode", ["greedy", "typical"])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_accept_ties_and_masked_runs(m, mode, dt):
    """Row statistics at their edge cases, decisions equal to the oracle's: runs of
    -inf logits (masked vocabulary) covering one whole 16384-logit chunk, whole 16-byte
    vectors and an unaligned stretch, with planted candidates inside them; and every
    planted maximum repeated at a second id, lower than the candidate's in half of the
    rows (the lowest id is the argmax, so greedy must then reject that candidate) and
    higher in the other half, in another chunk or in the same vector."""
    w = synth.small_variant(synth.WORKLOADS["vicuna7b-64"], batch=4, vocab=40000, dtype="f32", seed=93)
    acc = synth.rank_accuracy(4, 10)
    t_o = otree.compile_template(otree.greedy_tree(acc, 63), 10)
    t_g = m.Template(t_o.paths[1:], 10, device="cuda")
    root, pool = synth.random_pool(w)
    tokens = np.stack([o_fill(t_o, root[b], pool[b], 0)[0] for b in range(w.batch)])
    logits = synth.target_logits(w, t_o.n_rows)
    for lo, hi in [(16384, 32768), (1024, 1088), (5003, 5011)]:
        logits[:, :, lo:hi] = -math.inf
    synth.plant_argmax(logits, pool, t_o.depth, acc, synth.plant_uniforms(w, t_o.n_rows))
    n_tied = 0
    for b in range(w.batch):
        for u in range(t_o.n_rows):
            row = logits[b, u]
            p = int(torch.argmax(row))
            if p == 0 or p == w.vocab - 1:
                continue
            # a second id with the same maximum: below p for even rows, above for odd; in
            # p's own 16-byte vector when there is room, else in another vector or chunk
            if u % 2 == 0:
                q = p - 1 if p % 4 != 0 else p // 2
            else:
                q = p + 1 if (p + 1) % 4 != 0 else min(w.vocab - 1, p + 16383)
            row[q] = row[p]
            n_tied += 1
    if dt == "bf16":
        logits = logits.to(torch.bfloat16)
    r = m.medusa_tree_accept(t_g, logits.cuda(), gu.device_tensor(tokens, torch.int32), mode,
                             epsilon=w.epsilon, delta=w.delta)
    r = {k: v.cpu().numpy() for k, v in r.items()}
    skipped = 0
    for b in range(w.batch):
        o = oacc.accept(gu.to64(logits[b]), tokens[b], t_o.retrieve, mode, 1.0, w.epsilon, w.delta, False)
        if mode == "typical" and gu.typical_ambiguous(o):
            skipped += 1
            continue
        assert r["accept_len"][b] == o.accept_len, b
        G = o.accept_len + 1
        assert list(r["out_rows"][b, :G]) == list(o.out_rows)
        assert list(r["out_tokens"][b, :G]) == list(o.out_tokens)
        assert r["best_path"][b] == o.best_path
    assert skipped <= 1 and n_tied > 0


def test_accept_root_only_template(m):
    t_g = m.Template([], 4, device="cuda")
    logits = torch.randn(2, 1, 100, device="cuda")
    tokens = torch.tensor([[5], [9]], dtype=torch.int32, device="cuda")
    r = m.medusa_tree_accept(t_g, logits, tokens, "typical")
    assert list(r["accept_len"].cpu()) == [0, 0]
    assert list(r["out_tokens"][:, 0].cpu()) == [5, 9]


# ----------------------------------------------------------------------------- compaction

@pytest.mark.parametrize("paged", [False, True])
@pytest.mark.parametrize("mirror", [False, True])
def test_kv_compact(m, paged, mirror):
    w = synth.small_variant(synth.WORKLOADS["serving-b16-paged"], batch=5, prefix_range=(1, 300), seed=101,
                            page_size=16 if paged else 0)
    acc = synth.rank_accuracy(4, 10)
    t_o = otree.compile_template(otree.greedy_tree(acc, 63), 10)
    t_g = m.Template(t_o.paths[1:], 10, device="cuda")
    lengths = synth.prefix_lengths(w)
    N = t_o.n_rows
    if paged:
        K, V, bt, lay, _, _ = gu.paged_cache(w, lengths, N)
        cache = m.KVCache(K, V, block_table=bt)
    else:
        K, V, _, _ = gu.contiguous_cache(w, lengths, N)
        cache = m.KVCache(K, V)
    # distinct content in every staged row
    g = torch.Generator(device="cpu").manual_seed(5)
    K.copy_(torch.randn(K.shape, generator=g).to(K.dtype))
    V.copy_(torch.randn(V.shape, generator=g).to(V.dtype))
    if mirror:
        cache.add_mirror()
    rng = np.random.default_rng(3)
    W = t_o.max_depth + 1
    rows = np.full((w.batch, W), -1, dtype=np.int32)
    alen = np.zeros(w.batch, dtype=np.int32)
    for b in range(w.batch):
        p = int(rng.integers(0, t_o.n_paths))
        nodes = [x for x in t_o.retrieve[p] if x >= 0]
        a = int(rng.integers(0, len(nodes)))
        alen[b] = a
        rows[b, :a + 1] = nodes[:a + 1]
    Kh, Vh = K.cpu(), V.cpu()
    L_out, status = m.medusa_kv_compact(cache, t_g, gu.device_tensor(lengths, torch.int32),
                                        gu.device_tensor(alen, torch.int32), gu.device_tensor(rows, torch.int32))
    torch.cuda.synchronize()
    assert (status.cpu().numpy() == 0).all()
    assert list(L_out.cpu().numpy()) == list(lengths + alen + 1)
    if mirror:
        same_as_mirror(cache)
    for b in range(w.batch):
        L = int(lengths[b])
        G = int(alen[b]) + 1
        cap = L + N + 16
        if paged:
            kb = np.stack([gu.to64(gu.read_paged_row(Kh, bt.cpu(), b, r)) for r in range(cap)], axis=1)
            vb = np.stack([gu.to64(gu.read_paged_row(Vh, bt.cpu(), b, r)) for r in range(cap)], axis=1)
            ka = np.stack([gu.to64(gu.read_paged_row(K.cpu(), bt.cpu(), b, r)) for r in range(cap)], axis=1)
            va = np.stack([gu.to64(gu.read_paged_row(V.cpu(), bt.cpu(), b, r)) for r in range(cap)], axis=1)
        else:
            kb, vb = gu.to64(Kh[b, :, :cap]), gu.to64(Vh[b, :, :cap])
            ka, va = gu.to64(K[b, :, :cap]), gu.to64(V[b, :, :cap])
        new_len = ocomp.kv_compact(kb, vb, L, rows[b, :G])
        assert new_len == L + G
        assert (ka == kb).all() and (va == vb).all()


@pytest.mark.parametrize("paged,n_layers,mirror", [(False, 5, False), (True, 3, True), (False, 130, False),
                                                   (False, 70, True)])
def test_kv_compact_layers(m, paged, n_layers, mirror):
    """Every layer's cache compacted by one call, against the oracle's compaction of
    each layer; a sequence with an invalid path stays untouched in every layer; more
    than 128 layers take several launches with status and L_out written once (70
    layers with fp16 mirrors are 140 caches: two launches as well)."""
    if n_layers > 8 and not mirror:      # many small layers: fp32, one KV head of 64 dims
        w = synth.small_variant(synth.WORKLOADS["tiny-fp32"], batch=4, n_kv_heads=1, n_q_heads=1,
                                prefix_len=None, prefix_range=(1, 120), seed=141)
    else:
        w = synth.small_variant(synth.WORKLOADS["serving-b16-paged"], batch=4, prefix_range=(1, 300),
                                seed=131 + n_layers, page_size=16 if paged else 0)
    acc = synth.rank_accuracy(4, 10)
    t_o = otree.compile_template(otree.greedy_tree(acc, 63), 10)
    t_g = m.Template(t_o.paths[1:], 10, device="cuda")
    lengths = synth.prefix_lengths(w)
    N, W = t_o.n_rows, t_o.max_depth + 1
    g = torch.Generator(device="cpu").manual_seed(17 + n_layers)
    caches, Ks, Vs = [], [], []
    bt = None
    for layer in range(n_layers):
        if paged:
            K, V, bt_l, lay, _, _ = gu.paged_cache(w, lengths, N)
            bt = bt_l if bt is None else bt            # one block table for every layer
            caches.append(m.KVCache(K, V, block_table=bt))
        else:
            K, V, _, _ = gu.contiguous_cache(w, lengths, N)
            caches.append(m.KVCache(K, V))
        K.copy_(torch.randn(K.shape, generator=g).to(K.dtype))
        V.copy_(torch.randn(V.shape, generator=g).to(V.dtype))
        if mirror:
            caches[-1].add_mirror()
        Ks.append(K)
        Vs.append(V)
    rng = np.random.default_rng(7 + n_layers)
    rows = np.full((w.batch, W), -1, dtype=np.int32)
    alen = np.zeros(w.batch, dtype=np.int32)
    for b in range(w.batch):
        p = int(rng.integers(0, t_o.n_paths))
        nodes = [x for x in t_o.retrieve[p] if x >= 0]
        a = int(rng.integers(1, len(nodes))) if len(nodes) > 1 else 0
        alen[b] = a
        rows[b, :a + 1] = nodes[:a + 1]
    bad = w.batch - 1                    # its second row is not a child of the root
    deep = next(u for u in range(1, N) if t_o.parent[u] != 0)
    rows[bad] = -1
    rows[bad, :2] = [0, deep]
    alen[bad] = 1
    before = [(K.cpu().clone(), V.cpu().clone()) for K, V in zip(Ks, Vs)]
    Ld = gu.device_tensor(lengths, torch.int32)
    L_out, status = m.medusa_kv_compact_layers(caches, t_g, Ld, gu.device_tensor(alen, torch.int32),
                                               gu.device_tensor(rows, torch.int32))
    torch.cuda.synchronize()
    st = status.cpu().numpy()
    assert st[bad] == -7 and (np.delete(st, bad) == 0).all()
    want_L = lengths + alen + 1
    want_L[bad] = lengths[bad]
    assert list(L_out.cpu().numpy()) == list(want_L)
    for layer in range(n_layers):
        Kb, Vb = before[layer]
        Ka, Va = Ks[layer].cpu(), Vs[layer].cpu()
        for b in range(w.batch):
            L = int(lengths[b])
            cap = L + N + 16 if not paged else L + N
            if paged:
                kb = np.stack([gu.to64(gu.read_paged_row(Kb, bt.cpu(), b, r)) for r in range(cap)], axis=1)
                vb = np.stack([gu.to64(gu.read_paged_row(Vb, bt.cpu(), b, r)) for r in range(cap)], axis=1)
                ka = np.stack([gu.to64(gu.read_paged_row(Ka, bt.cpu(), b, r)) for r in range(cap)], axis=1)
                va = np.stack([gu.to64(gu.read_paged_row(Va, bt.cpu(), b, r)) for r in range(cap)], axis=1)
            else:
                kb, vb = gu.to64(Kb[b, :, :cap]), gu.to64(Vb[b, :, :cap])
                ka, va = gu.to64(Ka[b, :, :cap]), gu.to64(Va[b, :, :cap])
            if b != bad:
                ocomp.kv_compact(kb, vb, L, rows[b, :alen[b] + 1])
            assert np.array_equal(ka, kb) and np.array_equal(va, vb), (layer, b)
        if mirror:
            same_as_mirror(caches[layer])


def test_kv_compact_rejects_bad_paths(m):
    w = synth.small_variant(synth.WORKLOADS["tiny-fp32"], batch=4, seed=111)
    t_o = otree.compile_template(otree.regular_paths((2, 3)), 3)
    t_g = m.Template(t_o.paths[1:], 3, device="cuda")
    lengths = np.array([10, 10, 10, 10])
    K, V, _, _ = gu.contiguous_cache(w, lengths, t_o.n_rows)
    cache = m.KVCache(K, V)
    W = t_o.max_depth + 1
    rows = np.full((4, W), -1, dtype=np.int32)
    rows[0, :2] = [0, 1]          # valid
    rows[1, :2] = [0, 4]          # row 4 is not a child of the root
    rows[2, :3] = [0, 1, 9]       # out of range
    rows[3, :2] = [1, 3]          # does not start at the root
    alen = np.array([1, 1, 2, 1], dtype=np.int32)
    before = K.clone()
    L_out, status = m.medusa_kv_compact(cache, t_g, gu.device_tensor(lengths, torch.int32),
                                        gu.device_tensor(alen, torch.int32), gu.device_tensor(rows, torch.int32))
    torch.cuda.synchronize()
    assert list(status.cpu().numpy()) == [0, -7, -7, -7]
    assert list(L_out.cpu().numpy()) == [12, 10, 10, 10]
    assert torch.equal(K[1:], before[1:])
