"""Pins of the oracle's whole round (oracle.round.run_sequence) on a worked example.

The round's steps are pinned one by one elsewhere; this file checks how the round
wires them together, on inputs small enough to work out by hand from the pages:

- heads ([M7.2] §0x02A): with W1 = 0 the residual is z = h + SiLU(0) = h, so with
  h = e_0 every logit is column 0 of its matrix, and the ids follow by inspection;
- candidate gather ([M7.2] §0x04A): slot(p) = 1 + (t - 1) TOPK + r_t on the canonical
  rows of widths (2, 2);
- positions ([M7.2] §0x01B): a node at depth t sits at sequence position L + t, so a
  rotated 2-element key (1, 0) points at angle L + t (one RoPE pair, frequency 1);
- staging and compaction ([M7.2] §0x06A, §0x06B): the accepted path's rows land at
  cache rows L, L + 1, ... and the committed length is L + a + 1;
- greedy acceptance ([PartII] Part 7) on planted target argmaxes.

A mistake in the wiring (positions without L, staging at L + depth instead of
L + u, a pool read in the wrong order, compaction of the wrong path) fails here.
"""
import math

import numpy as np
import pytest

from oracle import attention, round as oround, tree


pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

L = 3
D = 4          # hidden size
V = 6          # vocabulary
TOPK = 2


def _inputs():
    h = np.zeros(D)
    h[0] = 1.0
    w1 = np.zeros((2, D, D))
    w_lm = np.zeros((V, D))
    w_lm[3, 0] = 5.0                      # root = 3
    w2 = np.zeros((2, V, D))
    w2[0, 1, 0], w2[0, 4, 0] = 4.0, 3.0   # head 0 ranks ids 1, 4
    w2[1, 0, 0], w2[1, 5, 0] = 2.0, 1.0   # head 1 ranks ids 0, 5
    tmpl = oround.template_for(("regular", (2, 2)), TOPK, 2)
    N = tmpl.n_rows
    rng = np.random.default_rng(7)
    q = rng.standard_normal((N, 1, 2))
    k_new = np.tile(np.array([1.0, 0.0]), (N, 1, 1))
    v_new = rng.standard_normal((N, 1, 2))
    cap = L + N
    cache_k = rng.standard_normal((1, cap, 2))
    cache_v = rng.standard_normal((1, cap, 2))
    # Target logits: row 0 prefers token 1 (node (0,)), row 1 prefers token 0 (node
    # (0, 0)); every other row prefers token 2, which no candidate carries.
    logits = np.zeros((N, V))
    logits[:, 2] = 1.0
    logits[0, 1] = 9.0
    logits[1, 0] = 9.0
    return tmpl, h, w1, w2, w_lm, q, k_new, v_new, cache_k, cache_v, logits


def test_round_worked_example():
    tmpl, h, w1, w2, w_lm, q, k_new, v_new, cache_k, cache_v, logits = _inputs()
    prefix_k, prefix_v = cache_k[:, :L].copy(), cache_v[:, :L].copy()
    ck, cv = cache_k.copy(), cache_v.copy()
    r = oround.run_sequence(tmpl, h, w1, w2, w_lm, q, k_new, v_new, ck, cv, L, logits,
                            mode="greedy", base=10000.0)

    # Canonical rows of widths (2, 2): (), (0,), (1,), (0,0), (0,1), (1,0), (1,1).
    assert [tuple(p) for p in tmpl.paths] == [(), (0,), (1,), (0, 0), (0, 1), (1, 0), (1, 1)]
    assert r.root == 3
    assert r.pool.tolist() == [[1, 4], [0, 5]]
    # cand = [3, 1, 4, 0, 5]; slots 0, 1, 2, 3, 4, 3, 4.
    assert r.tokens.tolist() == [3, 1, 4, 0, 5, 0, 5]
    assert r.pos.tolist() == [3, 4, 4, 5, 5, 5, 5]
    assert r.head_logits.shape == (3, V)
    assert r.head_logits[0].tolist() == [0, 0, 0, 5, 0, 0]

    # Each staged key (1, 0) rotated to angle L + depth, length 1.
    for u in range(tmpl.n_rows):
        x, y = r.staged_k[u, 0]
        assert math.hypot(x, y) == pytest.approx(1.0, abs=1e-14)
        ang = L + int(tmpl.depth[u])
        assert math.cos(ang) == pytest.approx(x, abs=1e-14)
        assert math.sin(ang) == pytest.approx(y, abs=1e-14)

    # Attention of every node equals plain causal attention along its own path.
    for u in range(tmpl.n_rows):
        ref = attention.path_attention(q, k_new, v_new, prefix_k, prefix_v, L, tmpl.parent, u, 0)
        np.testing.assert_allclose(r.attn_out[u, 0], ref, rtol=0, atol=1e-13)

    # Greedy: path (0, 0) accepts both edges, (0, 1) one, the (1, *) paths none.
    acc = r.accept
    assert acc.accept_len == 2
    assert acc.out_rows.tolist() == [0, 1, 3]
    assert acc.out_tokens.tolist() == [3, 1, 0]
    assert acc.frontier_row == 3
    assert sorted(acc.per_path_len.tolist()) == [0, 0, 1, 2]
    assert r.new_len == L + 3

    # Prefix rows untouched; rows L, L+1, L+2 hold the staged rows of nodes 0, 1, 3.
    np.testing.assert_array_equal(ck[:, :L], prefix_k)
    np.testing.assert_array_equal(cv[:, :L], prefix_v)
    for j, u in enumerate([0, 1, 3]):
        np.testing.assert_array_equal(ck[0, L + j], r.staged_k[u, 0])
        np.testing.assert_array_equal(cv[0, L + j], v_new[u, 0])


def test_round_nothing_accepted_commits_root_only():
    """Every target argmax is a token no candidate carries: a = 0, one row committed."""
    tmpl, h, w1, w2, w_lm, q, k_new, v_new, cache_k, cache_v, logits = _inputs()
    logits = np.zeros_like(logits)
    logits[:, 2] = 1.0
    ck, cv = cache_k.copy(), cache_v.copy()
    r = oround.run_sequence(tmpl, h, w1, w2, w_lm, q, k_new, v_new, ck, cv, L, logits)
    assert r.accept.accept_len == 0
    assert r.accept.out_rows.tolist() == [0]
    assert r.accept.out_tokens.tolist() == [3]
    assert r.new_len == L + 1
    np.testing.assert_array_equal(ck[0, L], r.staged_k[0, 0])
    np.testing.assert_array_equal(cv[0, L], v_new[0, 0])


def test_round_template_is_the_compiled_regular_tree():
    """template_for on a regular spec is compile_template of the regular paths."""
    a = oround.template_for(("regular", (2, 2)), TOPK, 2)
    b = tree.compile_template(tree.regular_paths((2, 2)), TOPK, 2)
    assert a.slot.tolist() == b.slot.tolist() == [0, 1, 2, 3, 4, 3, 4]
    assert a.depth.tolist() == [0, 1, 1, 2, 2, 2, 2]
    assert a.parent.tolist() == [-1, 0, 0, 1, 1, 2, 2]
