"""Pins for the template compiler, regular trees and greedy tree search of the oracle."""
import itertools
import json
import os

import numpy as np
import pytest

from oracle import cost, tree
from oracle.round import template_for, tree_fill
import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ----------------------------------------------------------------------------- worked examples

def test_a31_nine_row_fixture():
    g = gold("a31_nine_row.json")
    t = tree.compile_template(g["paths"], g["topk"])
    assert t.n_rows == 9
    L = g["prefix_len"]
    assert list(L + t.depth) == g["positions"]
    from oracle.attention import visibility
    assert list(visibility(L, t.mask).shape) == g["rect_mask_shape"]
    assert t.n_paths == g["n_paths"]
    assert list(L + np.arange(t.n_rows)) == g["staged_rows"]
    counts = {s: int((t.slot == s).sum()) for s in g["slots_occurring_twice"]}
    assert all(c == 2 for c in counts.values())
    pool = np.array([g["head0_ranks"], g["head1_ranks"]])
    tokens, pos = tree_fill(t, g["root_token"], pool, L)
    assert list(tokens) == [11, 21, 22, 31, 32, 33, 31, 32, 33]
    assert list(pos) == g["positions"]


def test_seven_node_example():
    g = gold("seven_node.json")
    t = tree.compile_template(tree.regular_paths(g["widths"]), topk=2)
    sym = g["symbols"]
    pool = np.array([[sym["b"], sym["u"]], [sym["c"], sym["v"]]])
    tokens, pos = tree_fill(t, sym["a"], pool, L=100)
    assert list(tokens) == g["tokens"]
    assert list(pos - 100) == g["position_offsets"]
    names = g["node_order"]
    row_cu = names.index("c|u")
    seen = {names[v] for v in range(t.n_rows) if t.mask[row_cu, v]}
    assert seen == set(g["visible_from_c|u"])
    # the four paths as a plain batch would take 4 * 3 token slots; the tree needs 7 rows
    assert t.n_paths * (t.max_depth + 1) == g["paths_as_batch_tokens"]
    assert t.n_rows == 7


@pytest.mark.parametrize("case", gold("counts.json")["regular"])
def test_regular_counts(case):
    w = case["widths"]
    t = tree.compile_template(tree.regular_paths(w), topk=max(w))
    if "nodes" in case:
        assert t.n_rows - 1 == case["nodes"]
        assert tree.regular_node_count(w) == case["nodes"]
    if "paths" in case:
        assert t.n_paths == case["paths"]


def test_cartesian_top4_needs_six_mask_words():
    t = tree.compile_template(tree.regular_paths((4, 4, 4, 4)), topk=4)
    assert t.n_rows == 341
    assert -(-t.n_rows // 64) == 6
    assert t.n_paths == 256 and t.retrieve.shape[1] == 5


def test_cost_ledgers():
    g = gold("counts.json")
    hl = g["head_ledger"]
    d, V, K, R = hl["d"], hl["V"], hl["K"], hl["R_h"]
    assert cost.residual_block_params(d) == hl["residual_block_params"]
    assert V * d == hl["projection_params"]
    assert cost.head_params_independent(K, R, d, V) == hl["independent_params"]
    assert cost.head_params_shared(K, R, d) == hl["shared_params"]
    assert K * V * d == hl["projection_macs_one_row"]
    assert cost.head_flops(K, 1, R, d, V) == 2 * K * (d * d + V * d)
    kv = g["kv_ledger"]
    per = cost.kv_bytes_per_node(kv["layers"], kv["H_kv"], kv["d_h"], kv["bytes"])
    assert per == kv["bytes_per_node"]
    assert per * kv["nodes"] == kv["tree_bytes"]


# ----------------------------------------------------------------------------- invariants

def _random_prefix_closed(rng, topk, depth, n):
    paths = set()
    while len(paths) < n:
        L = int(rng.integers(1, depth + 1))
        p = tuple(int(x) for x in rng.integers(0, topk, size=L))
        for t in range(1, L + 1):
            paths.add(p[:t])
    return sorted(paths)


@pytest.mark.parametrize("seed", range(6))
def test_buffer_identities(seed):
    """Mask axioms and the inverse identities of the four buffers."""
    rng = np.random.default_rng(seed)
    topk = int(rng.integers(2, 6))
    t = tree.compile_template(_random_prefix_closed(rng, topk, 4, 20), topk)
    N = t.n_rows
    M = t.mask
    assert M.diagonal().all()                                   # reflexive
    assert M[:, 0].all()                                        # the root is everyone's ancestor
    for u in range(N):                                          # ancestor-transitive
        for v in np.flatnonzero(M[u]):
            assert (M[u] | ~M[v]).all()
    for u in range(1, N):                                       # siblings never see each other
        for v in range(1, N):
            if u != v and t.parent[u] == t.parent[v]:
                assert not M[u, v]
    for u in range(N):                                          # depth = path length; parent row smaller
        assert t.depth[u] == len(t.paths[u])
        assert u == 0 or t.parent[u] < u
        assert M[u].sum() == t.depth[u] + 1
    pool = rng.integers(1000, 2000, size=(4, topk))
    tokens, _ = tree_fill(t, 7, pool, 0)
    cand = np.concatenate([[7], pool.reshape(-1)])
    assert (cand[t.slot] == tokens).all()
    for row in t.retrieve:
        nodes = [int(x) for x in row if x >= 0]
        assert nodes[0] == 0
        assert all(x == -1 for x in row[len(nodes):])
        for a, b in zip(nodes, nodes[1:]):
            assert t.parent[b] == a and M[b, a]
        leaf = nodes[-1]
        assert not any(t.parent[c] == leaf for c in range(N))   # maximal paths end at leaves
        for j, node in enumerate(nodes):                       # token at depth j of the path
            p = t.paths[leaf][:j]
            assert t.paths[node] == p
    leaves = {u for u in range(N) if not any(t.parent[c] == u for c in range(N))}
    assert {int(r[r >= 0][-1]) for r in t.retrieve} == leaves


def test_root_only_template():
    t = tree.compile_template([], topk=4)
    assert t.n_rows == 1 and t.n_paths == 1 and list(t.retrieve[0]) == [0]


@pytest.mark.parametrize("bad", [
    [(0, 1)],                  # missing (0,)
    [(0,), (0,)],              # duplicate
    [(0,), (5,)],              # rank >= topk
    [(0,), (0, 0), (0, 0, 0)], # deeper than n_heads=2
])
def test_template_rejects(bad):
    with pytest.raises(tree.TemplateError):
        tree.compile_template(bad, topk=4, n_heads=2)


# ----------------------------------------------------------------------------- greedy tree search

def test_greedy_toy_order():
    g = gold("greedy_toy.json")
    acc = np.array(g["accuracy"])
    for key, w in g["weights"].items():
        p = tuple(int(x) for x in key.split(","))
        assert tree.path_weight(p, acc) == pytest.approx(w, rel=1e-12)
    got = tree.greedy_tree(acc, budget=len(g["order"]))
    assert [list(p) for p in got] == g["order"]


def _brute_force_top(acc, budget, depth):
    """Every path up to `depth`, ordered by weight (ties: shorter, then lexicographic)."""
    K, R = acc.shape
    allp = [p for L in range(1, depth + 1) for p in itertools.product(range(R), repeat=L)]
    w = {p: float(np.prod([acc[j, r] for j, r in enumerate(p)])) for p in allp}
    # group weights that agree to 1e-12 relative, as the greedy tie rule does
    key = {p: (round(np.log(w[p]) * 1e9), len(p), p) for p in allp}
    return sorted(allp, key=lambda p: (-key[p][0], key[p][1], key[p][2]))[:budget]


@pytest.mark.parametrize("K,R,budget", [(3, 4, 10), (4, 10, 63), (3, 6, 40), (2, 5, 20)])
def test_greedy_equals_global_order(K, R, budget):
    """With accuracies <= 1 a path never outweighs its parent, so the greedy frontier
    admits exactly the `budget` heaviest paths."""
    rng = np.random.default_rng(K * 100 + R)
    acc = np.sort(rng.uniform(0.01, 0.9, size=(K, R)), axis=1)[:, ::-1]
    got = tree.greedy_tree(acc, budget)
    want = _brute_force_top(acc, budget, K)
    assert set(got) == set(want)
    assert got == want


def test_greedy_page_toy_three_heads():
    """[M7.2] §0x04C toy calibration (budget 10); checked against the brute-force order."""
    acc = np.array([[0.55, 0.25, 0.10, 0.05], [0.50, 0.20, 0.10, 0.05], [0.45, 0.20, 0.10, 0.05]])
    got = tree.greedy_tree(acc, 10)
    assert set(got) == set(_brute_force_top(acc, 10, 3))
    t = tree.compile_template(got, topk=4)                      # prefix-closed by construction
    assert t.n_rows == 11
    assert tree.expected_accept_length(got, acc) == pytest.approx(
        sum(tree.path_weight(p, acc) for p in got))


def test_expected_accept_length_identity():
    """E[A] = sum of node weights equals the sum over depths of the survival
    probability P(A >= t) computed from all accepted-prefix events."""
    acc = np.array([[0.6, 0.2], [0.5, 0.1]])
    paths = tree.greedy_tree(acc, 5)
    # P(A >= t) = sum over depth-t nodes of the probability that exactly that rank path matches
    surv = [sum(tree.path_weight(p, acc) for p in paths if len(p) == t) for t in (1, 2)]
    assert tree.expected_accept_length(paths, acc) == pytest.approx(sum(surv))
    assert tree.expected_accept_length(paths, acc) == pytest.approx(0.6 + 0.2 + 0.3 + 0.1 + 0.06)


@pytest.mark.parametrize("name", ["vicuna7b-64", "llama3-8b-256"])
def test_workload_greedy_templates(name):
    w = synth.WORKLOADS[name]
    acc = synth.rank_accuracy(w.n_heads, 10)
    t = template_for(w.template, w.topk, w.n_heads, acc)
    budget = w.template[1]
    assert t.n_rows == budget + 1
    assert t.max_depth <= w.n_heads
    assert t.retrieve.shape[1] == t.max_depth + 1
    counts = np.bincount(t.depth, minlength=w.n_heads + 1)
    assert counts[0] == 1
    # with these accuracies the heaviest paths are prefix-closed and the top-ranked
    # depth-1 children receive the most descendants
    kids = [int((t.parent == u).sum()) for u in range(1, 1 + counts[1])]
    assert kids == sorted(kids, reverse=True)


@pytest.mark.parametrize("name,depths,leaves", [
    ("vicuna7b-64", [7, 21, 30, 5], 41),
    ("llama3-8b-256", [10, 55, 120, 70], 174),
])
def test_workload_greedy_tree_shapes(name, depths, leaves):
    """The greedy workloads' trees (budget 63 or 255 over ranks <= 10 of the synthetic
    accuracies a_k^(i) = 0.7 * 0.6^(k-1) * 0.45^(i-1), 1e-12 tie rule): nodes per depth and
    leaf count.  The 63-node cut falls inside a 15-way exact weight tie, so a different
    tie rule changes the first shape."""
    from oracle.round import template_for
    w = synth.WORKLOADS[name]
    t = template_for(w.template, w.topk, w.n_heads, synth.rank_accuracy(w.n_heads, 10))
    assert t.n_rows == 1 + sum(depths)
    assert np.bincount(t.depth)[1:].tolist() == depths
    assert t.n_paths == leaves
