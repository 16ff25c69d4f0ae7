"""Failure paths of the device calls, made to happen without a GPU fault.

Timeouts.  Every wait inside a kernel is bounded; when one gives up, the kernel takes
its error path: it records MEDUSA_ETIMEOUT for the sequence (attention) or publishes
-1 ids (heads), waits for its own copies and MMAs, frees its tensor memory, still joins
the cluster barriers and returns, so the context stays usable.  The test hook
medusa_test_set_stall_ns makes each CTA first wait on a flag that nothing sets; after
the given time that wait runs out and the error path runs.  The tests check that the
call returns, what it reports, that nothing of the sequence was written, and that the
next call without the hook is correct again.

Range.  The bf16 tensor-core attention multiplies in fp16; a K/V value or a scaled
rotated query outside fp16's range becomes inf, which turns the softmax of the rows
that see it into NaN.  The kernel must then report MEDUSA_ERANGE for that sequence
instead of returning inf/NaN with status 0.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import attention as oatt
from oracle import round as oround
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

STALL_NS = 1_000_000          # 1 ms: the hook's wait gives up quickly


@pytest.fixture(scope="module")
def m():
    import medusa_speculative_tree_gb300 as m
    from medusa_speculative_tree_gb300 import build
    build.build()
    return m


class stall:
    """Turns the test hook on for the calls inside the block."""

    def __init__(self, m, ns):
        self.lib, self.ns = m.api.nat.lib(), ns

    def __enter__(self):
        self.lib.medusa_test_set_stall_ns(self.ns)

    def __exit__(self, *a):
        self.lib.medusa_test_set_stall_ns(0)
        return False


def attn_case(m, name, **kw):
    w = synth.small_variant(synth.WORKLOADS[name], **kw)
    acc = synth.rank_accuracy(w.n_heads, 10)
    t_o = oround.template_for(w.template, w.topk, w.n_heads, acc)
    t_g = m.Template(t_o.paths[1:], w.topk, w.n_heads, device="cuda")
    N = t_o.n_rows
    lengths = synth.prefix_lengths(w)
    q, k, v = synth.tree_qkv(w, N, device="cuda")
    if w.page_size:
        K, V, bt, _, ks, vs = gu.paged_cache(w, lengths, N)
        mk = lambda K_, V_: m.KVCache(K_, V_, block_table=bt)
    else:
        K, V, ks, vs = gu.contiguous_cache(w, lengths, N)
        mk = lambda K_, V_: m.KVCache(K_, V_)
    return w, t_o, t_g, q, k, v, K, V, ks, vs, lengths, mk


# (one query tile per CTA, two query tiles per CTA, paged)
ATTN_CASES = [
    ("vicuna7b-64", dict(prefix_len=300, n_q_heads=4, n_kv_heads=4)),
    ("llama3-8b-256", dict(prefix_len=700, n_q_heads=8, n_kv_heads=2)),
    ("serving-b16-paged", dict(batch=3, n_q_heads=8, n_kv_heads=2, prefix_range=(100, 900))),
]


@pytest.mark.parametrize("name,kw", ATTN_CASES)
def test_attention_timeout_reports_and_writes_nothing(m, name, kw):
    w, t_o, t_g, q, k, v, K, V, ks, vs, lengths, mk = attn_case(m, name, **kw)
    B, N = w.batch, t_o.n_rows
    L = gu.device_tensor(lengths, torch.int32)
    K0, V0 = K.clone(), V.clone()
    out = torch.full((B, N, w.n_q_heads, w.head_dim), 7.0, device="cuda")
    with stall(m, STALL_NS):
        _, _, status = m.medusa_tree_attn_verify(t_g, q, k, v, mk(K, V), L, int(lengths.max()),
                                                 rope_base=w.rope_base, out=out)
        torch.cuda.synchronize()
    assert (status.cpu().numpy() == m.api.nat.ETIMEOUT).all()
    assert (out == 7.0).all()                                  # no output row written
    assert torch.equal(K, K0) and torch.equal(V, V0)          # no staged row, no cache write

    # the context is usable and the next call is correct again
    out2, _, status2 = m.medusa_tree_attn_verify(t_g, q, k, v, mk(K, V), L, int(lengths.max()),
                                                 rope_base=w.rope_base)
    torch.cuda.synchronize()
    assert (status2.cpu().numpy() == 0).all()
    for b in range(B):
        Lb = int(lengths[b])
        ck = np.zeros((w.n_kv_heads, Lb, w.head_dim))
        cv = np.zeros_like(ck)
        ck[:], cv[:] = gu.to64(ks[b]), gu.to64(vs[b])
        o, _, _ = oatt.tree_attention(gu.to64(q[b]), gu.to64(k[b]), gu.to64(v[b]), ck, cv, Lb, t_o.depth,
                                      t_o.mask, w.rope_base)
        gu.float_parity(out2[b], o, False, f"{name} attention after a timeout, sequence {b}")


def test_heads_timeout_reports_and_writes_nothing(m):
    w = synth.small_variant(synth.WORKLOADS["vicuna7b-64"], hidden=512, vocab=2000, n_heads=2)
    h, w1, w2, w_lm = synth.head_weights(w, device="cuda")
    logits = torch.full((1, w.n_heads + 1, w.vocab), 5.0, device="cuda")
    with stall(m, STALL_NS):
        root, pool = m.medusa_heads_topk(h, w1, w2, w_lm, w.topk, logits_out=logits)
        torch.cuda.synchronize()
    assert (root.cpu().numpy() == -1).all() and (pool.cpu().numpy() == -1).all()
    assert (logits == 5.0).all()
    root2, pool2 = m.medusa_heads_topk(h, w1, w2, w_lm, w.topk, logits_out=logits)
    torch.cuda.synchronize()
    gl = logits[0].cpu().numpy().astype(np.float64)
    assert int(root2[0]) == int(np.lexsort((np.arange(w.vocab), -gl[0]))[0])
    for k in range(w.n_heads):
        assert list(pool2[0, k].cpu().numpy()) == list(np.lexsort((np.arange(w.vocab), -gl[1 + k]))[:w.topk])


@pytest.mark.parametrize("where", ["prefix_k", "prefix_v", "tree_k", "tree_v", "query"])
def test_attention_reports_fp16_range(m, where):
    """One value beyond fp16's range in one sequence: that sequence reports MEDUSA_ERANGE,
    the other keeps status 0 and its parity."""
    w, t_o, t_g, q, k, v, K, V, ks, vs, lengths, mk = attn_case(m, "vicuna7b-64", batch=2, prefix_len=300,
                                                                 n_q_heads=4, n_kv_heads=4)
    B, N = w.batch, t_o.n_rows
    bad = 1
    if where == "prefix_k":
        K[bad, 2, 17, 5] = 1e5
    elif where == "prefix_v":
        V[bad, 1, 200, 64] = 7e4
    elif where == "tree_k":
        k[bad, 0, 0, 9] = 2e5                 # the root's key: every row sees it
    elif where == "tree_v":
        v[bad, 5, 2, 100] = -7e4
    else:
        q[bad, 4, 1, 3] = 1e6                 # times scale * log2 e: about 1.3e5
    L = gu.device_tensor(lengths, torch.int32)
    out, _, status = m.medusa_tree_attn_verify(t_g, q, k, v, mk(K, V), L, int(lengths.max()),
                                               rope_base=w.rope_base)
    torch.cuda.synchronize()
    st = status.cpu().numpy()
    assert st[bad] == m.api.nat.ERANGE
    assert st[0] == 0
    Lb = int(lengths[0])
    o, _, _ = oatt.tree_attention(gu.to64(q[0]), gu.to64(k[0]), gu.to64(v[0]), gu.to64(ks[0]), gu.to64(vs[0]),
                                  Lb, t_o.depth, t_o.mask, w.rope_base)
    gu.float_parity(out[0], o, False, "the sequence without an out-of-range value")
