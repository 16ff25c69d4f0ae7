"""Plausible mistakes planted in the oracle (on the CPU) must be caught by the pins.

Each test swaps one oracle function for a mutated copy, re-runs the relevant pin
and asserts that it now fails.  Mutations follow the failure lists of
[M7.2] §0x03F, §0x04G and §0x06E.
"""
import math

import numpy as np
import pytest

from oracle import accept, attention, compact, tree
import tests.test_oracle_accept_compact as AC
import tests.test_oracle_tree as TT
import tests.test_oracle_attention as TA


def fails(fn):
    try:
        fn()
    except AssertionError:
        return True
    return False


def test_positions_by_packed_row(monkeypatch):
    real = tree.compile_template

    def mutated(paths, topk, n_heads=None):
        t = real(paths, topk, n_heads)
        t.depth = np.arange(t.n_rows)            # positions follow packed order
        return t
    monkeypatch.setattr(tree, "compile_template", mutated)
    assert fails(TT.test_a31_nine_row_fixture)


def test_sibling_leak(monkeypatch):
    real = tree.compile_template

    def mutated(paths, topk, n_heads=None):
        t = real(paths, topk, n_heads)
        t.mask = np.tril(np.ones_like(t.mask))   # ordinary causal mask over packed rows
        return t
    monkeypatch.setattr(tree, "compile_template", mutated)
    assert fails(TT.test_seven_node_example)
    monkeypatch.setattr(tree, "compile_template", real)
    t, q, k, v, pk, pv, L = TA._case(0, (2, 3))
    out, _, _ = attention.tree_attention(q, k, v, pk, pv, L, t.depth, np.tril(np.ones_like(t.mask)))
    want = attention.path_attention(q, k, v, pk, pv, L, t.parent, t.n_rows - 1, 0)
    assert not np.allclose(out[-1, 0], want)


def test_hidden_prefix_key(monkeypatch):
    real = attention.visibility

    def mutated(L, mask):
        vis = real(L, mask)
        vis[:, 0] = False                        # one prompt key hidden from every query
        return vis
    monkeypatch.setattr(attention, "visibility", mutated)
    assert fails(lambda: TA.test_tree_equals_independent_path_attention(0, (2, 3)))


def test_rope_sign(monkeypatch):
    real = attention.rope
    monkeypatch.setattr(attention, "rope", lambda x, pos, base=10000.0: real(x, -np.asarray(pos), base))
    assert fails(TA.test_rope_dh2_is_a_plane_rotation)


def test_self_aligned_logits(monkeypatch):
    real = accept.accept

    def mutated(logits, tokens, retrieve, mode="greedy", *a, **kw):
        # compare each candidate with the argmax of its own row instead of its parent's
        shifted = np.asarray(logits).copy()
        for row in retrieve:
            nodes = [u for u in row if u >= 0]
            for a_, b_ in zip(nodes, nodes[1:]):
                shifted[a_] = np.asarray(logits)[b_]
        return real(shifted, tokens, retrieve, mode, *a, **kw)
    monkeypatch.setattr(accept, "accept", mutated)
    assert fails(AC.test_greedy_winner_a31)


def test_threshold_max_instead_of_min(monkeypatch):
    monkeypatch.setattr(accept, "min", max, raising=False)
    assert fails(AC.test_typical_winner_a31)


def test_entropy_sign(monkeypatch):
    real = accept.row_stats

    def mutated(*a, **kw):
        st = real(*a, **kw)
        st.entropy = -st.entropy
        return st
    monkeypatch.setattr(accept, "row_stats", mutated)
    assert fails(AC.test_typical_winner_a31)


def test_raw_probability_tie_break(monkeypatch):
    monkeypatch.setattr(accept, "edge_score", math.exp)   # sum raw probabilities instead
    assert fails(AC.test_typical_tie_break_uses_log_likelihood)


def test_non_prefix_counting(monkeypatch):
    real = accept.accept

    def mutated(logits, tokens, retrieve, mode="greedy", *a, **kw):
        r = real(logits, tokens, retrieve, mode, *a, **kw)
        # count every matching edge of the chosen path, not only the leading ones
        nodes = [u for u in retrieve[r.best_path] if u >= 0]
        am = [int(np.argmax(logits[u])) for u in nodes]
        r.accept_len = sum(int(tokens[b] == am[j]) for j, b in enumerate(nodes[1:]))
        return r
    monkeypatch.setattr(accept, "accept", mutated)
    assert fails(AC.test_prefix_only_counting)


def test_publish_a_rows_instead_of_a_plus_one(monkeypatch):
    real = accept.accept

    def mutated(*a, **kw):
        r = real(*a, **kw)
        r.out_rows = r.out_rows[:-1] if len(r.out_rows) > 1 else r.out_rows
        return r
    monkeypatch.setattr(accept, "accept", mutated)
    assert fails(AC.test_typical_winner_a31)


def test_compact_without_snapshot(monkeypatch):
    def mutated(cache_k, cache_v, L, rows):
        rows = np.asarray(rows)
        for j in reversed(range(len(rows))):     # in-place, last edge first, no snapshot
            cache_k[:, L + j] = cache_k[:, L + rows[j]]
            cache_v[:, L + j] = cache_v[:, L + rows[j]]
        return L + len(rows)
    monkeypatch.setattr(compact, "kv_compact", mutated)
    assert fails(AC.test_compact_overlap_needs_snapshot)


def test_contiguous_commit_by_length(monkeypatch):
    def mutated(L, rows):
        n = len(rows)
        return L + np.arange(n), L + np.arange(n)
    monkeypatch.setattr(compact, "compaction_map", mutated)
    assert fails(AC.test_commit_trace)


def test_greedy_tree_wrong_tie_rule(monkeypatch):
    monkeypatch.setattr(tree, "_before", lambda wa, pa, wb, pb, rel=1e-12: wa < wb)
    assert fails(TT.test_greedy_toy_order)


def _row_stats_with_entropy(entropy_fn):
    """row_stats whose guarded entropy is computed by `entropy_fn(p)` (mutated copies)."""
    real = accept.row_stats

    def mutated(logits_row, temperature=1.0, entropy_guard=False):
        st = real(logits_row, temperature, entropy_guard)
        if entropy_guard:
            x = np.asarray(logits_row, dtype=np.float64) / float(temperature)
            e = np.exp(x - x.max())
            st.entropy = float(entropy_fn(e / e.sum()))
        return st
    return mutated


def test_guard_added_outside_the_log(monkeypatch):
    # -sum p (ln p + 1e-5): the guard added after the logarithm
    monkeypatch.setattr(accept, "row_stats", _row_stats_with_entropy(
        lambda p: -(p[p > 0] * (np.log(p[p > 0]) + 1e-5)).sum()))
    assert fails(AC.test_guarded_entropy_closed_forms)
    assert fails(AC.test_typical_decision_follows_the_guard)


def test_guard_only_on_zero_probabilities(monkeypatch):
    # the guard applied only where p = 0, i.e. the exact entropy everywhere else
    monkeypatch.setattr(accept, "row_stats", _row_stats_with_entropy(
        lambda p: -(p * np.log(np.where(p > 0, p, 1e-5))).sum()))
    assert fails(AC.test_guarded_entropy_closed_forms)
    assert fails(AC.test_typical_decision_follows_the_guard)


def test_guard_weighting_the_guard_too(monkeypatch):
    # -sum (p + 1e-5) ln(p + 1e-5): the guard also in the weight
    monkeypatch.setattr(accept, "row_stats", _row_stats_with_entropy(
        lambda p: -((p + 1e-5) * np.log(p + 1e-5)).sum()))
    assert fails(AC.test_guarded_entropy_closed_forms)


def test_log_prob_without_temperature(monkeypatch):
    # the candidate's logit taken unscaled while the statistics are scaled by 1 / T
    monkeypatch.setattr(accept, "log_prob",
                        lambda row, tok, st, temperature=1.0: float(np.float64(row[tok]) - st.m - st.log_z))
    assert fails(AC.test_temperature_two_closed_form)


# ---- the whole round (pins in tests/test_oracle_round.py) --------------------------

def test_round_pool_read_rank_major(monkeypatch):
    """cand taken rank by rank across the heads instead of head by head."""
    import oracle.round as oround
    import tests.test_oracle_round as TR

    def mutated(tmpl, root, pool, L):
        cand = np.concatenate([[int(root)], np.asarray(pool, dtype=np.int64).T.reshape(-1)])
        return cand[tmpl.slot].astype(np.int64), (int(L) + tmpl.depth).astype(np.int64)
    monkeypatch.setattr(oround, "tree_fill", mutated)
    assert fails(TR.test_round_worked_example)


def test_round_keys_rotated_without_prefix_offset(monkeypatch):
    """Staged tree keys rotated at depth(u) instead of L + depth(u)."""
    import tests.test_oracle_round as TR
    real = attention.tree_attention

    def mutated(q, k_new, v_new, pk, pv, L, depth, mask, base=10000.0, scale=None):
        out, lse, _ = real(q, k_new, v_new, pk, pv, L, depth, mask, base, scale)
        return out, lse, attention.rope(k_new, np.asarray(depth)[:, None], base)
    monkeypatch.setattr(attention, "tree_attention", mutated)
    assert fails(TR.test_round_worked_example)


def test_round_commits_by_depth(monkeypatch):
    """The accepted path's rows copied from L + depth instead of their staged rows L + u."""
    import tests.test_oracle_round as TR
    real = compact.kv_compact

    def mutated(cache_k, cache_v, L, rows):
        depth_rows = np.arange(len(rows))        # row j of the path sits at depth j
        return real(cache_k, cache_v, L, depth_rows)
    monkeypatch.setattr(compact, "kv_compact", mutated)
    assert fails(TR.test_round_worked_example)
