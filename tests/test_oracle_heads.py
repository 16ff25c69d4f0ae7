"""Pins for the Medusa heads and top-k of the oracle."""
import math

import numpy as np
import pytest

from oracle import heads


def test_silu_closed_form():
    x = np.array([0.0, 1.0, -1.0, 40.0, -40.0, 2.5])
    want = [0.0, 1.0 / (1.0 + math.exp(-1.0)), -1.0 / (1.0 + math.exp(1.0)), 40.0, 0.0,
            2.5 / (1.0 + math.exp(-2.5))]
    got = heads.silu(x)
    assert got[0] == 0.0
    assert got[1] == pytest.approx(0.7310585786300049, rel=1e-15)
    assert got[2] == pytest.approx(-0.2689414213699951, rel=1e-15)
    np.testing.assert_allclose(got, want, rtol=1e-14, atol=1e-15)


def test_ranked_ids_against_sorted_tuples():
    rng = np.random.default_rng(3)
    for _ in range(50):
        v = rng.integers(-3, 4, size=40).astype(np.float64)      # many exact ties
        k = int(rng.integers(1, 12))
        want = [i for _, i in sorted((-x, i) for i, x in enumerate(v))][:k]
        assert list(heads.ranked_ids(v, k)) == want


def test_zero_residual_reduces_to_lm_projection():
    """W1 = 0 gives z = h + SiLU(0) = h ([Math] 'The Medusa head': W1 starts near zero so the
    head behaves like the LM head).  With W2 = W_LM the head's top-1 is the root."""
    rng = np.random.default_rng(0)
    T, d, V, K = 3, 32, 50, 1
    h = rng.standard_normal((T, d))
    w_lm = rng.standard_normal((V, d))
    w1 = np.zeros((K, d, d))
    root, pool, logits = heads.medusa_heads(h, w1, w_lm[None], w_lm, topk=5)
    direct = np.stack([[sum(w_lm[v, j] * h[t, j] for j in range(d)) for v in range(V)]
                       for t in range(T)])
    np.testing.assert_allclose(logits[:, 0], direct, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(logits[:, 1], direct, rtol=1e-12, atol=1e-12)
    assert list(pool[:, 0, 0]) == list(root)
    for t in range(T):
        assert root[t] == int(np.argmax(direct[t]))


def test_residual_block_elementwise():
    """z = h + SiLU(W1 h + b1) checked element by element with explicit loops on a tiny case."""
    rng = np.random.default_rng(1)
    d, K = 4, 2
    h = rng.standard_normal((1, d))
    w1 = rng.standard_normal((K, d, d))
    b1 = rng.standard_normal((K, d))
    z = heads.residual(h, w1, b1)
    for k in range(K):
        for i in range(d):
            pre = sum(w1[k, i, j] * h[0, j] for j in range(d)) + b1[k, i]
            assert z[0, k, i] == pytest.approx(h[0, i] + pre / (1 + math.exp(-pre)), rel=1e-12)


def test_shared_projection_contract():
    """A 2-D W2 is one projection reused by every head ([M7.2] §0x02D)."""
    rng = np.random.default_rng(2)
    T, d, V, K = 2, 16, 30, 3
    h = rng.standard_normal((T, d))
    w1 = 0.1 * rng.standard_normal((K, d, d))
    u = rng.standard_normal((V, d))
    _, p_shared, l_shared = heads.medusa_heads(h, w1, u, u, topk=4)
    _, p_stack, l_stack = heads.medusa_heads(h, w1, np.stack([u] * K), u, topk=4)
    np.testing.assert_allclose(l_shared, l_stack, rtol=1e-14)
    assert (p_shared == p_stack).all()


def test_head_logit_rows_matches_full():
    rng = np.random.default_rng(5)
    d, V, K = 16, 40, 2
    h = rng.standard_normal((1, d))
    w1 = 0.2 * rng.standard_normal((K, d, d))
    w2 = rng.standard_normal((K, V, d))
    w_lm = rng.standard_normal((V, d))
    _, _, full = heads.medusa_heads(h, w1, w2, w_lm, topk=3)
    rows = [(0, 3), (1, 7), (2, 39), (2, 0)]
    got = heads.head_logit_rows(h[0], lambda k: w1[k], lambda k, v: w2[k, v], lambda v: w_lm[v], rows)
    np.testing.assert_allclose(got, [full[0, m, v] for m, v in rows], rtol=1e-12)


def test_blocked_heads_helper_equals_medusa_heads():
    """The parity tests' blocked evaluation of the heads (vocabulary rows in blocks) is the
    oracle's medusa_heads: same root, pools and logits on a tiny case with a ragged
    last block."""
    import torch
    from tests import gpu_util as gu
    rng = np.random.default_rng(3)
    T, K, d, V, topk = 3, 2, 16, 37, 4
    h = torch.tensor(rng.normal(size=(T, d)))
    w1 = torch.tensor(rng.normal(size=(K, d, d)) * 0.1)
    w2 = torch.tensor(rng.normal(size=(K, V, d)))
    w_lm = torch.tensor(rng.normal(size=(V, d)))
    r1, p1, l1 = heads.medusa_heads(h.numpy(), w1.numpy(), w2.numpy(), w_lm.numpy(), topk)
    r2, p2, l2 = gu.oracle_heads_blocked(h, w1, w2, w_lm, topk, block=10)
    assert (r1 == r2).all() and (p1 == p2).all()
    assert np.allclose(l1, l2, rtol=1e-13, atol=1e-12)
