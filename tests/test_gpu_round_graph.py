"""The whole round as one CUDA graph (medusa_round_create / medusa_round_launch)
against the same five calls issued one by one: every output bit for bit, replays
stable, and new input values written in place picked up by the next launch."""
import pytest
import torch

import bench
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    import medusa_speculative_tree_gb300 as m
    from medusa_speculative_tree_gb300 import build
    build.build()
    return m


def eager(rd):
    """The five calls one by one; every output cloned."""
    root, pool = rd.heads()
    tokens, pos = rd.fill(root, pool)
    out, _, st = rd.attn()
    r = rd.accept(tokens)
    L_out, st2 = rd.compact(r)
    torch.cuda.synchronize()
    res = {"root": root, "pool": pool, "tokens": tokens, "pos": pos, "out": out, "attn_status": st,
           "L_out": L_out, "compact_status": st2}
    res.update(r)
    return {k: v.clone() for k, v in res.items()}


def make_round(m, rd):
    w = rd.w
    return m.MedusaRound(rd.tmpl, rd.h, rd.w1, rd.w2, rd.w_lm, w.topk, rd.L, rd.q, rd.k, rd.v, rd.cache,
                         rd.max_L, rd.logits, mode=rd.mode, rope_base=w.rope_base, epsilon=w.epsilon,
                         delta=w.delta)


def same(graph, ref, what):
    for k, v in ref.items():
        g = getattr(graph, k)
        assert g.shape == v.shape and torch.equal(g, v), (what, k)


def cache_rows(rd, upto):
    """K and V rows [0, upto) of every sequence, as dense tensors."""
    if rd.w.page_size:
        bt = rd.cache.block_table.long()
        nb = (upto + 15) // 16
        k = rd.K[bt[:, :nb]].transpose(2, 3).reshape(rd.w.batch, nb * 16, rd.w.n_kv_heads, -1)[:, :upto]
        v = rd.V[bt[:, :nb]].transpose(2, 3).reshape(rd.w.batch, nb * 16, rd.w.n_kv_heads, -1)[:, :upto]
        return k.clone(), v.clone()
    return rd.K[:, :, :upto].clone(), rd.V[:, :, :upto].clone()


@pytest.mark.parametrize("name", ["tiny-fp32", "vicuna7b-64", "serving-b16-paged"])
def test_round_graph_matches_the_five_calls(m, name):
    w = synth.WORKLOADS[name]
    rd = bench.Round(m, w, torch.device("cuda"))
    ref = eager(rd)
    upto = rd.max_L + rd.tmpl.max_depth + 1
    k_ref, v_ref = cache_rows(rd, upto)
    rnd = make_round(m, rd)
    for rep in range(3):                      # replays give the same round
        rnd.launch()
        torch.cuda.synchronize()
        same(rnd, ref, f"{name} launch {rep}")
        assert (rnd.attn_status == 0).all() and (rnd.compact_status == 0).all()
    k_g, v_g = cache_rows(rd, upto)
    assert torch.equal(k_g, k_ref) and torch.equal(v_g, v_ref)

    # new inputs written into the same buffers: another frontier row and a prefix
    # three rows shorter, so positions, attention and the published rows all move
    rd.h.copy_(torch.roll(rd.h, 1, dims=1))
    rd.L.sub_(3)
    rd2 = eager(rd)
    assert not torch.equal(rd2["pos"], ref["pos"])
    rnd.launch()
    torch.cuda.synchronize()
    same(rnd, rd2, f"{name} after in-place update")
    rnd.close()


def test_round_create_reports_a_bad_call(m):
    """A descriptor that fails one of the recorded calls' own checks (here the heads:
    top-k wider than the vocabulary) returns that call's status and creates nothing."""
    from medusa_speculative_tree_gb300._native import MedusaError, EINVAL
    w = synth.WORKLOADS["tiny-fp32"]
    rd = bench.Round(m, w, torch.device("cuda"))
    with pytest.raises(MedusaError) as e:
        m.MedusaRound(rd.tmpl, rd.h, rd.w1, rd.w2, rd.w_lm, w.vocab + 1, rd.L, rd.q, rd.k, rd.v, rd.cache,
                      rd.max_L, rd.logits)
    assert e.value.status == EINVAL
    # the context is still usable
    ref = eager(rd)
    assert int(ref["attn_status"][0]) == 0


def test_round_graph_with_hidden_state_acceptance(m):
    """Step 4 as medusa_tree_accept_hidden (the target's hidden states instead of
    logits): the graph equals the five eager calls bit for bit, logits unused."""
    w = synth.WORKLOADS["vicuna7b-64"]
    rd = bench.Round(m, w, torch.device("cuda"))
    hid = synth.normal((w.batch, rd.N, w.hidden), 1.0, w.seed, "h", rd.dev, w.torch_dtype, sub=3)
    root, pool = rd.heads()
    tokens, pos = rd.fill(root, pool)
    out, _, st = rd.attn()
    r = m.medusa_tree_accept_hidden(rd.tmpl, hid, rd.w_lm, tokens, "typical", epsilon=w.epsilon, delta=w.delta)
    L_out, st2 = rd.compact(r)
    torch.cuda.synchronize()
    ref = {"root": root, "pool": pool, "tokens": tokens, "pos": pos, "out": out, "attn_status": st,
           "L_out": L_out, "compact_status": st2}
    ref.update(r)
    ref = {k: v.clone() for k, v in ref.items()}
    rnd = m.MedusaRound(rd.tmpl, rd.h, rd.w1, rd.w2, rd.w_lm, w.topk, rd.L, rd.q, rd.k, rd.v, rd.cache, rd.max_L,
                        None, mode="typical", rope_base=w.rope_base, epsilon=w.epsilon, delta=w.delta,
                        hidden_target=hid)
    for rep in range(2):
        rnd.launch()
        torch.cuda.synchronize()
        same(rnd, ref, f"hidden-state round, launch {rep}")
    assert int(rnd.accept_len[0]) >= 0
    rnd.close()
    # the same with the commit fused into the acceptance kernel
    upto = rd.max_L + rd.tmpl.n_rows
    k0, v0 = cache_rows(rd, upto)
    rnd = m.MedusaRound(rd.tmpl, rd.h, rd.w1, rd.w2, rd.w_lm, w.topk, rd.L, rd.q, rd.k, rd.v, rd.cache, rd.max_L,
                        None, mode="typical", rope_base=w.rope_base, epsilon=w.epsilon, delta=w.delta,
                        hidden_target=hid, fuse_commit=True)
    rnd.launch()
    torch.cuda.synchronize()
    same(rnd, ref, "hidden-state round with the fused commit")
    k1, v1 = cache_rows(rd, upto)
    assert torch.equal(k1, k0) and torch.equal(v1, v0)
    rnd.close()


@pytest.mark.parametrize("name", synth.WORKLOAD_ORDER)
def test_fused_commit_equals_accept_then_compact(m, name):
    """medusa_tree_accept_commit against medusa_tree_accept + medusa_kv_compact: the
    acceptance outputs, L_out, status and every cache row the same; a sequence whose
    L + N exceeds the capacity gets MEDUSA_ECAPACITY and is left untouched; and the
    round graph with the fused commit equals the five eager calls."""
    w = synth.WORKLOADS[name]
    rd = bench.Round(m, w, torch.device("cuda"))
    ref = eager(rd)                          # stages the tree rows, separate compaction
    upto = rd.max_L + rd.tmpl.n_rows
    k0, v0 = cache_rows(rd, upto)
    rnd = m.MedusaRound(rd.tmpl, rd.h, rd.w1, rd.w2, rd.w_lm, w.topk, rd.L, rd.q, rd.k, rd.v, rd.cache, rd.max_L,
                        rd.logits, mode=rd.mode, rope_base=w.rope_base, epsilon=w.epsilon, delta=w.delta,
                        fuse_commit=True)
    rnd.launch()
    torch.cuda.synchronize()
    same(rnd, ref, f"{name} fused-commit round")
    k1, v1 = cache_rows(rd, upto)
    assert torch.equal(k1, k0) and torch.equal(v1, v0)
    rnd.close()

    # the standalone call, after restaging the tree rows (attention) each time
    tokens = ref["tokens"]
    rd.attn()
    r_sep = rd.accept(tokens)
    L_sep, st_sep = rd.compact(r_sep)
    torch.cuda.synchronize()
    k_sep, v_sep = cache_rows(rd, upto)
    rd.attn()
    r_f = m.medusa_tree_accept_commit(rd.tmpl, rd.logits, tokens, rd.cache, rd.L, rd.mode, epsilon=w.epsilon,
                                      delta=w.delta)
    torch.cuda.synchronize()
    for k in ("best_path", "accept_len", "out_tokens", "out_rows", "frontier_row"):
        assert torch.equal(r_f[k], r_sep[k]), k
    assert torch.equal(r_f["L_out"], L_sep) and torch.equal(r_f["status"], st_sep)
    k_f, v_f = cache_rows(rd, upto)
    assert torch.equal(k_f, k_sep) and torch.equal(v_f, v_sep)

    # capacity failure: sequence 0 claims a prefix that leaves no room for the tree
    if not w.page_size:
        cap = rd.K.shape[2]
        L_bad = rd.L.clone()
        L_bad[0] = cap - rd.tmpl.n_rows + 1
        before_k, before_v = rd.K.clone(), rd.V.clone()
        r_b = m.medusa_tree_accept_commit(rd.tmpl, rd.logits, tokens, rd.cache, L_bad, rd.mode, epsilon=w.epsilon,
                                          delta=w.delta)
        torch.cuda.synchronize()
        assert int(r_b["status"][0]) == -2 and int(r_b["L_out"][0]) == int(L_bad[0])
        assert torch.equal(rd.K[0], before_k[0]) and torch.equal(rd.V[0], before_v[0])
