"""Pins for acceptance and compaction of the oracle.

The pages describe the nine-row fixture's winners but do not print its target
distributions, so two distributions are constructed here to satisfy that
description; their expected outcomes are derived by hand in the comments.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import accept, compact, tree
from oracle.round import tree_fill

GOLD = os.path.join(os.path.dirname(__file__), "golden")
EPS, DELTA = 0.09, 0.3
V = 64


def gold():
    with open(os.path.join(GOLD, "a31_nine_row.json")) as f:
        return json.load(f)


def a31():
    g = gold()
    t = tree.compile_template(g["paths"], g["topk"])
    pool = np.array([g["head0_ranks"], g["head1_ranks"]])
    tokens, _ = tree_fill(t, g["root_token"], pool, g["prefix_len"])
    return g, t, tokens


def dist(mass: dict, rest_over: int = None):
    """log of a distribution over V ids: given masses, the remainder spread uniformly over the others."""
    p = np.zeros(V)
    for tok, m in mass.items():
        p[tok] = m
    others = [i for i in range(V) if i not in mass]
    p[others] = (1.0 - sum(mass.values())) / len(others)
    return np.log(p)


def fixture_one():
    """Row 0 (root 11): p(21)=.40, p(22)=.35.  Row 1 (token 21): p(31)=.30, p(32)=.06, p(33)=.005.
    Row 2 (token 22): p(31)=.90, p(32)=.02, p(33)=.005.  Leaves get uniform logits.

    Thresholds tau = min(.09, .3 e^-H):  H0 = 2.1123 -> tau0 = .03629;
    H1 = 3.4553 -> tau1 = .009471;  H2 = .70214 -> .3 e^-H2 = .14866 -> tau2 = .09.
    Typical lengths per path (0,0),(0,1),(0,2),(1,0),(1,1),(1,2) = 2,2,1,2,1,1;
    log-likelihoods of the length-2 paths: -2.1203, -3.7297, -1.1552 -> winner (1,0)
    = tokens [11,22,31], rows [0,2,6].  Greedy: argmax row0 = 21, rows 1 and 2 -> 31;
    lengths 2,1,1,0,0,0 -> winner path 0 = [11,21,31].
    """
    logits = np.zeros((9, V))
    logits[0] = dist({21: .40, 22: .35})
    logits[1] = dist({31: .30, 32: .06, 33: .005})
    logits[2] = dist({31: .90, 32: .02, 33: .005})
    return logits


def fixture_two():
    """Separates the log-likelihood tie-break from a raw-probability sum.
    Row 0: p(21)=.40, p(22)=.58.  Row 1: p(31)=.50.  Row 2: p(31)=.34, p(40)=.30.
    tau0 = .09, tau1 = .0189, tau2 = .02271; all other candidates fall below their threshold.
    Length-2 paths: (0,0) with log(.4*.5) = -1.6094 and (1,0) with log(.58*.34) = -1.6235,
    so (0,0) wins, although .58+.34 > .40+.50.
    """
    logits = np.zeros((9, V))
    logits[0] = dist({21: .40, 22: .58})
    logits[1] = dist({31: .50})
    logits[2] = dist({31: .34, 40: .30})
    return logits


def test_greedy_winner_a31():
    g, t, tokens = a31()
    r = accept.accept(fixture_one(), tokens, t.retrieve, "greedy")
    assert list(r.per_path_len) == [2, 1, 1, 0, 0, 0]
    assert list(r.out_tokens) == g["greedy_winner_tokens"]
    assert r.accept_len == g["greedy_accept_len"]
    assert r.best_path == 0 and r.frontier_row == 3


def test_typical_winner_a31():
    g, t, tokens = a31()
    r = accept.accept(fixture_one(), tokens, t.retrieve, "typical", epsilon=EPS, delta=DELTA)
    assert list(r.per_path_len) == [2, 2, 1, 2, 1, 1]
    assert list(r.out_tokens) == g["typical_winner_tokens"]
    assert r.accept_len == g["typical_accept_len"]
    assert list(r.out_rows) == g["commit_rows"]
    assert r.frontier_row == 6
    np.testing.assert_allclose(r.per_path_score[[0, 1, 3]],
                               [math.log(.4 * .3), math.log(.4 * .06), math.log(.35 * .9)], rtol=1e-12)


def test_typical_tie_break_uses_log_likelihood():
    g, t, tokens = a31()
    r = accept.accept(fixture_two(), tokens, t.retrieve, "typical", epsilon=EPS, delta=DELTA)
    assert list(r.per_path_len) == [2, 1, 1, 2, 1, 1]
    assert list(r.out_tokens) == [11, 21, 31]


def test_root_only_progress():
    g, t, tokens = a31()
    logits = np.zeros((9, V))
    logits[0] = dist({5: .9})           # target wants a token no head proposed
    for mode in ("greedy", "typical"):
        r = accept.accept(logits, tokens, t.retrieve, mode, epsilon=EPS, delta=DELTA)
        assert r.accept_len == 0 and r.best_path == 0
        assert list(r.out_tokens) == g["root_only_tokens"]
        assert list(r.out_rows) == [0] and r.frontier_row == 0


def test_prefix_only_counting():
    """[PartII] Part 7: raw matches [T, F, T, T] give accepted length 1."""
    t = tree.compile_template(tree.regular_paths((1, 1, 1, 1)), topk=1)
    tokens = np.array([100, 101, 102, 103, 104])
    logits = np.zeros((5, 200))
    wanted = [101, 999 % 200, 103, 104]           # edge 1 fails, later edges would match
    for u, w in enumerate(wanted):
        logits[u, w] = 5.0
    r = accept.accept(logits, tokens, t.retrieve, "greedy")
    assert r.accept_len == 1 and list(r.out_rows) == [0, 1]


def test_argmax_ties_lowest_id():
    t = tree.compile_template([(0,), (1,)], topk=2)
    tokens = np.array([0, 7, 3])
    logits = np.zeros((3, 10))
    logits[0, [3, 7]] = 2.0                        # tie between ids 3 and 7: argmax is 3
    r = accept.accept(logits, tokens, t.retrieve, "greedy")
    assert r.best_path == 1 and list(r.out_tokens) == [0, 3]


def test_entropy_closed_forms():
    """Uniform over n ids: H = ln n; one-hot: H = 0; two-point (p, 1-p): binary entropy."""
    st = accept.row_stats(np.zeros(1000))
    assert st.entropy == pytest.approx(math.log(1000), rel=1e-13)
    one = np.full(50, -1e4)
    one[3] = 0.0
    assert accept.row_stats(one).entropy == pytest.approx(0.0, abs=1e-12)
    p = 0.2
    two = np.full(2, 0.0)
    two[1] = math.log((1 - p) / p)
    assert accept.row_stats(two).entropy == pytest.approx(-(p * math.log(p) + (1 - p) * math.log(1 - p)))
    # temperature scales logits before the softmax: T -> infinity approaches uniform
    x = np.array([0.0, 1.0, 2.0])
    assert accept.row_stats(x, temperature=1e9).entropy == pytest.approx(math.log(3), rel=1e-6)


def test_five_token_entropy():
    """[PartII] Part 8 distribution p = [.35,.25,.18,.12,.10]: H = 1.5073652 nats, e^-H = .221493.
    (The page's printed value was lost; these digits come from the definition.)"""
    p = np.array([.35, .25, .18, .12, .10])
    st = accept.row_stats(np.log(p))
    assert st.entropy == pytest.approx(1.5073652, abs=2e-7)
    assert math.exp(-st.entropy) == pytest.approx(0.221493, abs=1e-6)
    tau = min(EPS, DELTA * math.exp(-st.entropy))
    assert tau == pytest.approx(0.066448, abs=1e-6)
    assert all(x > tau for x in p)                 # every listed token passes at this position


def test_commit_trace():
    """[M7.2] §0x06B: rows [0,2,6], P = 5 -> sources [5,7,11] -> destinations [5,6,7], length 8."""
    g = gold()
    src, dst = compact.compaction_map(g["prefix_len"], g["commit_rows"])
    assert list(src) == g["commit_sources"] and list(dst) == g["commit_destinations"]
    Hkv, dh, cap = 2, 4, 16
    ck = np.arange(Hkv * cap * dh, dtype=np.float64).reshape(Hkv, cap, dh)
    cv = -ck.copy()
    before_k, before_v = ck.copy(), cv.copy()
    new_len = compact.kv_compact(ck, cv, g["prefix_len"], g["commit_rows"])
    assert new_len == g["commit_new_len"] and new_len - g["prefix_len"] == g["commit_published"]
    for s, d in zip(src, dst):
        assert (ck[:, d] == before_k[:, s]).all() and (cv[:, d] == before_v[:, s]).all()
    assert (ck[:, :5] == before_k[:, :5]).all()   # committed prefix untouched


def test_compact_overlap_needs_snapshot():
    """rows [0,2,5] at L = 0: destination 2 is also the source of edge 1."""
    ck = np.arange(8, dtype=np.float64).reshape(1, 8, 1)
    cv = ck.copy()
    compact.kv_compact(ck, cv, 0, [0, 2, 5])
    assert list(ck[0, :3, 0]) == [0.0, 2.0, 5.0]


# ---- the target's vocabulary projection folded into acceptance -----------------------

def _internal(t):
    return [u for u in range(t.n_rows) if (np.asarray(t.parent) == u).any()]


def test_target_logits_identity_projection_reduces_to_accept():
    """W_LM = I (V = d): the projection returns the internal hidden rows themselves
    (leaves stay NaN: acceptance must never read them), so acceptance on hidden rows
    equals acceptance on those rows taken as logits, which the fixtures above pin."""
    rng = np.random.default_rng(5)
    t = tree.compile_template(tree.regular_paths((2, 3)), 3)
    N, d = t.n_rows, 16
    hidden = rng.normal(size=(N, d))
    internal = _internal(t)
    lg = accept.target_logits(hidden, np.eye(d), internal)
    for u in range(N):
        if u in internal:
            assert np.array_equal(lg[u], hidden[u])
        else:
            assert np.isnan(lg[u]).all()
    tokens = rng.integers(0, d, size=N)
    for v in range(1, N):                      # half the candidates are the parent's argmax
        if rng.random() < 0.5:
            tokens[v] = int(np.argmax(hidden[t.parent[v]]))
    for mode in ("greedy", "typical"):
        a = accept.accept_hidden(hidden, np.eye(d), tokens, t.retrieve, internal, mode)
        b = accept.accept(np.where(np.isnan(lg), 0.0, lg), tokens, t.retrieve, mode)
        assert (a.best_path, a.accept_len, a.frontier_row) == (b.best_path, b.accept_len, b.frontier_row)
        assert list(a.out_rows) == list(b.out_rows) and list(a.out_tokens) == list(b.out_tokens)


def test_target_logits_one_hot_closed_form():
    """Orthonormal rows of W_LM (V = 8 < d = 12) and hidden[u] = alpha W_LM[t_u]: the
    logits are alpha at t_u and 0 elsewhere, so argmax = t_u,
    p(t_u) = e^alpha / (e^alpha + V - 1) and
    H = ln(e^alpha + V - 1) - alpha e^alpha / (e^alpha + V - 1).
    With alpha = 5: p(t_u) = .955 > min(.09, .3 e^-H) = .09, while every other token has
    p = .0064 < .09.  Child 0 of each internal row carries t_u, the others a different
    token, so both greedy and typical accept exactly the all-zero-rank path: rows
    [0, row(0), row(0, 0)], a = 2."""
    V_, d, alpha = 8, 12, 5.0
    rng = np.random.default_rng(9)
    q, _ = np.linalg.qr(rng.normal(size=(d, d)))
    W = q[:V_]                                  # orthonormal rows
    t = tree.compile_template(tree.regular_paths((2, 3)), 3)
    N = t.n_rows
    internal = _internal(t)
    target = {u: int(rng.integers(0, V_)) for u in internal}
    hidden = np.zeros((N, d))
    for u in internal:
        hidden[u] = alpha * W[target[u]]
    tokens = np.zeros(N, dtype=np.int64)
    for v in range(1, N):
        p = int(t.parent[v])
        rank = t.paths[v][-1]
        tokens[v] = target[p] if rank == 0 else (target[p] + 1 + rank) % V_
    lg = accept.target_logits(hidden, W, internal)
    ea = math.exp(alpha)
    for u in internal:
        want = np.zeros(V_)
        want[target[u]] = alpha
        assert np.allclose(lg[u], want, atol=1e-12)
        st = accept.row_stats(lg[u])
        assert st.argmax == target[u]
        assert math.isclose(st.entropy, math.log(ea + V_ - 1) - alpha * ea / (ea + V_ - 1), rel_tol=1e-12)
    row = {tuple(p): i for i, p in enumerate(t.paths)}
    for mode in ("greedy", "typical"):
        r = accept.accept_hidden(hidden, W, tokens, t.retrieve, internal, mode, epsilon=EPS, delta=DELTA)
        assert r.accept_len == 2
        assert list(r.out_rows) == [0, row[(0,)], row[(0, 0)]]
        assert list(r.out_tokens) == [tokens[0], target[0], target[row[(0,)]]]


# ---- the guarded entropy and the temperature ----------------------------------------

def test_guarded_entropy_closed_forms():
    """[M7.2] §0x04E's guarded entropy -sum p ln(p + 1e-5) in special cases worked out
    by hand:
      uniform over n = 1000:  every p = 1/n, so H_g = -ln(1/n + 1e-5) = -ln(0.00101)
                              = 6.897804948128969 (the exact entropy is ln 1000 = 6.907755);
      one-hot:                the zero entries contribute 0 * ln(1e-5) = 0, so
                              H_g = -ln(1 + 1e-5) = -9.99995e-6 (negative: the guard, not p,
                              sits in the logarithm);
      two-point (.2, .8):     ln(.20001) = ln .2 + ln 1.00005 = -1.6093879136840586,
                              ln(.80001) = ln .8 + ln 1.0000125 = -0.2231310513923341,
                              H_g = .2 * 1.6093879136840586 + .8 * 0.2231310513923341
                                  = 0.500382423850679 (exact: 0.5004024235381879)."""
    st = accept.row_stats(np.zeros(1000), entropy_guard=True)
    assert st.entropy == pytest.approx(6.897804948128969, rel=1e-13)
    one = np.full(50, -1e4)                      # e^-1e4 underflows to an exact 0
    one[3] = 0.0
    assert accept.row_stats(one, entropy_guard=True).entropy == pytest.approx(-9.999950000398841e-06, rel=1e-9)
    two = np.array([0.0, math.log(4.0)])          # p = (.2, .8)
    assert accept.row_stats(two, entropy_guard=True).entropy == pytest.approx(0.500382423850679, rel=1e-13)
    assert accept.row_stats(two).entropy == pytest.approx(0.5004024235381879, rel=1e-13)


def guard_decision_case():
    """One edge whose typical decision the guard flips.  Row 0 over V = 1000 ids: the
    candidate (token 7) has p = 3.02e-4, the other 999 ids share the rest equally
    (1.0006987e-3 each).  Exact entropy H = 6.9074186283, threshold
    tau = min(.09, .3 e^-H) = 3.0010101e-4 < p: accepted.  Guarded entropy
    H_g = 6.8974683754, tau_g = .3 e^-H_g = 3.0310200e-4 > p: rejected."""
    V_ = 1000
    p = np.full(V_, (1.0 - 3.02e-4) / (V_ - 1))
    p[7] = 3.02e-4
    t = tree.compile_template([(0,)], topk=1)
    logits = np.zeros((2, V_))
    logits[0] = np.log(p)
    tokens = np.array([0, 7])
    return logits, tokens, t


def test_typical_decision_follows_the_guard():
    logits, tokens, t = guard_decision_case()
    exact = accept.accept(logits, tokens, t.retrieve, "typical", epsilon=EPS, delta=DELTA)
    guarded = accept.accept(logits, tokens, t.retrieve, "typical", epsilon=EPS, delta=DELTA, entropy_guard=True)
    assert exact.accept_len == 1 and list(exact.out_tokens) == [0, 7]
    assert guarded.accept_len == 0 and list(guarded.out_tokens) == [0]


def test_temperature_two_closed_form():
    """logits (0, ln 4) at T = 2 are (0, ln 2) after scaling, so p = (1/3, 2/3):
    log p(1) = ln(2/3) = -0.40546510810816444, log p(0) = ln(1/3) = -1.0986122886681098,
    H = ln 3 - (2/3) ln 2 = 0.6365141682948128, argmax 1."""
    x = np.array([0.0, math.log(4.0)])
    st = accept.row_stats(x, temperature=2.0)
    assert st.argmax == 1
    assert accept.log_prob(x, 1, st, 2.0) == pytest.approx(-0.40546510810816444, rel=1e-14)
    assert accept.log_prob(x, 0, st, 2.0) == pytest.approx(-1.0986122886681098, rel=1e-14)
    assert st.entropy == pytest.approx(0.6365141682948128, rel=1e-13)
