"""Pins for tree attention and RoPE of the oracle."""
import math

import numpy as np
import pytest

from oracle import attention, tree


def test_rope_dh2_is_a_plane_rotation():
    """With dh = 2 the single pair rotates by angle pos * base^0 = pos radians."""
    x = np.array([0.3, -1.7])
    for pos in [0, 1, 5, 37]:
        c, s = math.cos(pos), math.sin(pos)
        want = [0.3 * c - (-1.7) * s, -1.7 * c + 0.3 * s]
        np.testing.assert_allclose(attention.rope(x, pos), want, rtol=1e-14, atol=1e-15)


def test_rope_frequency_layout():
    """dh = 4: pair (0, 2) turns at pos * 1, pair (1, 3) at pos * base^(-1/2)."""
    base = 100.0
    x = np.array([1.0, 0.0, 0.0, 0.0])
    y = np.array([0.0, 1.0, 0.0, 0.0])
    p = 3
    np.testing.assert_allclose(attention.rope(x, p, base), [math.cos(p), 0, math.sin(p), 0], atol=1e-15)
    a = p / math.sqrt(base)
    np.testing.assert_allclose(attention.rope(y, p, base), [0, math.cos(a), 0, math.sin(a)], atol=1e-15)


def test_rope_relative_phase():
    rng = np.random.default_rng(0)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    d1 = attention.rope(q, 100) @ attention.rope(k, 97)
    d2 = attention.rope(q, 5003) @ attention.rope(k, 5000)
    assert d1 == pytest.approx(d2, rel=1e-10)
    assert attention.rope(q, 0) == pytest.approx(q)


def test_softmax_weights_by_hand():
    """Two keys with scores 0 and ln 3 (after scaling): weights 1/4 and 3/4."""
    scale = 0.5
    q = np.array([2.0 * math.log(3.0), 0.0])
    keys = np.array([[0.0, 1.0], [1.0, 0.0]])
    vals = np.array([[4.0, 0.0], [0.0, 8.0]])
    out = attention.single_query_attention(q, keys, vals, scale)
    np.testing.assert_allclose(out, [1.0, 6.0], rtol=1e-14)


def _case(seed, widths_or_paths, Hq=4, Hkv=2, dh=16, L=11, topk=3):
    rng = np.random.default_rng(seed)
    if len(widths_or_paths) and isinstance(widths_or_paths[0], int):
        paths = tree.regular_paths(widths_or_paths)
    else:
        paths = widths_or_paths
    t = tree.compile_template(paths, topk)
    N = t.n_rows
    q = rng.standard_normal((N, Hq, dh))
    k = rng.standard_normal((N, Hkv, dh))
    v = rng.standard_normal((N, Hkv, dh))
    pk = rng.standard_normal((Hkv, L + 5, dh))
    pv = rng.standard_normal((Hkv, L + 5, dh))
    return t, q, k, v, pk, pv, L


@pytest.mark.parametrize("seed,shape", [(0, (2, 3)), (1, (3, 2, 2)), (2, (1, 1, 1)),
                                        (3, [(0,), (1,), (0, 0), (0, 1), (1, 0), (0, 0, 0)])])
def test_tree_equals_independent_path_attention(seed, shape):
    """Every node's output equals causal attention over its own root-to-node path
    ([CN] 'Tree Attention'); the brute force uses the parent chain, not the mask."""
    t, q, k, v, pk, pv, L = _case(seed, shape)
    out, lse, kr = attention.tree_attention(q, k, v, pk, pv, L, t.depth, t.mask, base=500.0)
    for u in range(t.n_rows):
        for h in range(q.shape[1]):
            want = attention.path_attention(q, k, v, pk, pv, L, t.parent, u, h, base=500.0)
            np.testing.assert_allclose(out[u, h], want, rtol=1e-11, atol=1e-12)


def test_chain_tree_is_causal_decode():
    """A width-1 chain is ordinary causal decoding of the chain tokens after the prefix."""
    t, q, k, v, pk, pv, L = _case(7, (1, 1, 1), Hq=2, Hkv=2)
    out, _, _ = attention.tree_attention(q, k, v, pk, pv, L, t.depth, t.mask)
    dh = q.shape[-1]
    for h in range(2):
        keys = np.concatenate([pk[h, :L], attention.rope(k[:, h], L + np.arange(4))])
        vals = np.concatenate([pv[h, :L], v[:, h]])
        for u in range(4):
            qv = attention.rope(q[u, h], L + u)
            s = keys[:L + u + 1] @ qv / math.sqrt(dh)
            w = np.exp(s - s.max())
            want = (w / w.sum()) @ vals[:L + u + 1]
            np.testing.assert_allclose(out[u, h], want, rtol=1e-11)


def test_root_only_is_single_query_attention():
    t, q, k, v, pk, pv, L = _case(9, [], Hq=2, Hkv=1)
    out, _, kr = attention.tree_attention(q, k, v, pk, pv, L, t.depth, t.mask)
    for h in range(2):
        keys = np.concatenate([pk[0, :L], kr[:, 0]])
        vals = np.concatenate([pv[0, :L], v[:, 0]])
        want = attention.single_query_attention(attention.rope(q[0, h], L), keys, vals,
                                                1 / math.sqrt(q.shape[-1]))
        np.testing.assert_allclose(out[0, h], want, rtol=1e-12)


def test_zero_query_averages_visible_values():
    """q = 0 makes every visible score equal: the output is the mean of visible values."""
    t, q, k, v, pk, pv, L = _case(4, (2, 2))
    q[:] = 0.0
    out, lse, _ = attention.tree_attention(q, k, v, pk, pv, L, t.depth, t.mask)
    for u in range(t.n_rows):
        vis = np.flatnonzero(t.mask[u])
        for h in range(q.shape[1]):
            kv = h // 2
            want = (pv[kv, :L].sum(0) + v[vis, kv].sum(0)) / (L + len(vis))
            np.testing.assert_allclose(out[u, h], want, rtol=1e-12)
            assert lse[u, h] == pytest.approx(math.log(L + len(vis)))


def test_node_attention_rows_matches_dense():
    t, q, k, v, pk, pv, L = _case(11, (3, 2))
    out, lse, _ = attention.tree_attention(q, k, v, pk, pv, L, t.depth, t.mask)
    for u in [0, 2, t.n_rows - 1]:
        for h in [0, 3]:
            kv = h // 2
            o, l = attention.node_attention_rows(q[u, h], k[:, kv], v[:, kv], pk[kv], pv[kv],
                                                 L, t.depth, t.mask[u], u)
            np.testing.assert_allclose(o, out[u, h], rtol=1e-12)
            assert l == pytest.approx(lse[u, h], rel=1e-12)


def test_bf16_values_in_fp16_range_convert_exactly():
    """The tensor-core attention multiplies bf16 K/V in fp16, and a cache's fp16 mirror
    stores them so: every bf16 value of magnitude in [2^-14, 65504] has an fp16 twin of
    the same value (all 65536 bit patterns checked), zero stays zero, and every larger
    finite value becomes inf (which the attention reports as a range error)."""
    b = np.arange(65536, dtype=np.uint32)
    f32 = (b << 16).view(np.float32)
    with np.errstate(over="ignore"):
        f16 = f32.astype(np.float16)
    back = f16.astype(np.float32)
    fin = np.isfinite(f32)
    mag = np.abs(f32)
    in_range = fin & (mag >= 2.0 ** -14) & (mag <= 65504)
    assert in_range.sum() == 2 * 30 * 128              # sign x 30 exponents x 128 mantissas
    assert (back[in_range] == f32[in_range]).all()
    assert (back[f32 == 0] == 0).all()
    assert np.isinf(f16[fin & (mag > 65504)]).all()
