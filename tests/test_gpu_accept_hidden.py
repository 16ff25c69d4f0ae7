"""Acceptance with the target's vocabulary projection folded in
(medusa_tree_accept_hidden) against the oracle's projection + acceptance in float64
on the same bf16 inputs: every published decision bit for bit."""
import numpy as np
import pytest
import torch

import synth
from oracle import accept as oacc
from oracle import tree as otree

import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    import medusa_speculative_tree_gb300 as m
    from medusa_speculative_tree_gb300 import build
    build.build()
    return m


def planted_inputs(t_o, B, d, V, seed, alpha=8.0):
    """W_LM ~ N(0, 1/d); each internal row's hidden state is alpha W_LM[t_u] + N(0, 1),
    so its argmax is t_u by a wide margin; the rank-0 child of u carries t_u with
    probability 0.7, every other child a random token."""
    g = torch.Generator().manual_seed(seed)
    W = (torch.randn((V, d), generator=g) / d ** 0.5).to(torch.bfloat16)
    N = t_o.n_rows
    rng = np.random.default_rng(seed)
    internal = [u for u in range(N) if (np.asarray(t_o.parent) == u).any()]
    hidden = torch.randn((B, N, d), generator=g)
    tokens = rng.integers(0, V, size=(B, N)).astype(np.int32)
    for b in range(B):
        for u in internal:
            tu = int(rng.integers(0, V))
            hidden[b, u] += alpha * W[tu].float()
            for v in range(1, N):
                if t_o.parent[v] == u and t_o.paths[v][-1] == 0 and rng.random() < 0.7:
                    tokens[b, v] = tu
    return hidden.to(torch.bfloat16), W, tokens, internal


@pytest.mark.parametrize("B,d,V,mode", [(1, 256, 3001, "greedy"), (1, 256, 3001, "typical"),
                                        (1, 4096, 32000, "typical"), (16, 512, 5000, "greedy"),
                                        (16, 512, 5000, "typical")])
def test_accept_hidden_matches_oracle(m, B, d, V, mode):
    acc = synth.rank_accuracy(4, 10)
    t_o = otree.compile_template(otree.greedy_tree(acc, 63), 10)
    t_g = m.Template(t_o.paths[1:], 10, device="cuda")
    hidden, W, tokens, internal = planted_inputs(t_o, B, d, V, seed=1000 + d + B)
    r = m.medusa_tree_accept_hidden(t_g, hidden.cuda(), W.cuda(), torch.as_tensor(tokens).cuda(), mode)
    torch.cuda.synchronize()
    W64 = gu.to64(W)
    accepted = 0
    for b in range(B):
        o = oacc.accept_hidden(gu.to64(hidden[b]), W64, tokens[b], t_o.retrieve, internal, mode)
        if mode == "typical" and gu.typical_ambiguous(o):
            continue
        G = o.accept_len + 1
        assert int(r["accept_len"][b]) == o.accept_len, b
        assert int(r["best_path"][b]) == o.best_path, b
        assert int(r["frontier_row"][b]) == o.frontier_row, b
        assert list(r["out_rows"][b, :G].cpu().numpy()) == list(o.out_rows), b
        assert list(r["out_tokens"][b, :G].cpu().numpy()) == list(o.out_tokens), b
        assert (r["out_rows"][b, G:].cpu().numpy() == -1).all()
        accepted += o.accept_len
    assert accepted > 0                       # the planted candidates are accepted somewhere


@pytest.mark.parametrize("B,d,V,mode", [(64, 128, 100, "greedy"), (64, 128, 256, "typical"),
                                        (65, 128, 1000, "typical"), (65, 192, 777, "greedy")])
def test_accept_hidden_pass_and_vocabulary_edges(m, B, d, V, mode):
    """Regular (3, 2) tree: 4 internal rows per sequence, so B = 64 fills exactly one
    256-column pass and B = 65 needs a second pass of 4 columns; V = 100 is a single
    partial group of W_LM (most CTAs have no group), V = 256 two whole groups."""
    t_o = otree.compile_template(otree.regular_paths((3, 2)), 3)
    t_g = m.Template(t_o.paths[1:], 3, device="cuda")
    hidden, W, tokens, internal = planted_inputs(t_o, B, d, V, seed=77 + B + V)
    assert len(internal) == 4
    r = m.medusa_tree_accept_hidden(t_g, hidden.cuda(), W.cuda(), torch.as_tensor(tokens).cuda(), mode)
    torch.cuda.synchronize()
    W64 = gu.to64(W)
    checked = 0
    for b in range(B):
        o = oacc.accept_hidden(gu.to64(hidden[b]), W64, tokens[b], t_o.retrieve, internal, mode)
        if mode == "typical" and gu.typical_ambiguous(o):
            continue
        G = o.accept_len + 1
        assert int(r["accept_len"][b]) == o.accept_len, b
        assert int(r["best_path"][b]) == o.best_path, b
        assert list(r["out_rows"][b, :G].cpu().numpy()) == list(o.out_rows), b
        assert list(r["out_tokens"][b, :G].cpu().numpy()) == list(o.out_tokens), b
        checked += 1
    assert checked >= B - 2
