"""medusa_tree_attn_verify_static: tree attention for callers that cannot allocate.

Some callers cannot allocate device memory at the point where they run the
attention, e.g. a plugin or custom-op interface that only receives its input and
output pointers, or a serving loop whose memory is reserved up front.  For them
the library offers an entry point whose scratch lives in a fixed device array
inside the library.  These tests call it through the C ABI and check that it
returns what the workspace-taking entry point returns, on two calls in a row
(the array keeps the previous call's contents), and that shapes too large for
the array are refused before anything is enqueued.

This file is named so that pytest collects it last.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import synth
from oracle import round as oround
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    import medusa_speculative_tree_gb300 as m
    from medusa_speculative_tree_gb300 import build
    build.build()
    return m


def _setup(m, name, **kw):
    w = synth.small_variant(synth.WORKLOADS[name], **kw)
    acc = synth.rank_accuracy(w.n_heads, 10)
    t_o = oround.template_for(w.template, w.topk, w.n_heads, acc)
    t_g = m.Template(t_o.paths[1:], w.topk, w.n_heads, device="cuda")
    N = t_g.n_rows
    lengths = synth.prefix_lengths(w)
    q, k, v = synth.tree_qkv(w, N, device="cuda")
    K, V, _, _ = gu.contiguous_cache(w, lengths, N)
    return w, t_g, q, k, v, K, V, lengths


def _static_call(m, t_g, q, k, v, cache, L, max_prefix, rope_base, out, lse, status):
    nat = m.api.nat
    d = cache.desc()
    scale = 1.0 / float(q.shape[-1]) ** 0.5
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    vp = lambda x: C.c_void_p(x.data_ptr())
    return nat.lib().medusa_tree_attn_verify_static(
        C.byref(t_g.dev), q.shape[0], q.shape[2], vp(q), vp(k), vp(v), C.byref(d), vp(L), max_prefix,
        float(rope_base), float(scale), vp(out), vp(lse), vp(status), stream)


@pytest.mark.parametrize("name,mirror", [("tiny-fp32", False), ("vicuna7b-64", False), ("llama3-8b-256", False),
                                         ("vicuna7b-64", True), ("llama3-8b-256", True)])
def test_static_scratch_matches_workspace_entry(m, name, mirror):
    """With mirror, the static call runs on a cache carrying an fp16 mirror: the mirror
    holds the values the kernel otherwise converts itself, so the output is bit for bit
    that of the cache without one, and the mirror still mirrors the cache afterwards."""
    w, t_g, q, k, v, K, V, lengths = _setup(m, name)
    B, N = w.batch, t_g.n_rows
    L = gu.device_tensor(lengths, torch.int32)
    max_prefix = int(lengths.max())
    nat = m.api.nat

    # reference: the entry point that takes a caller workspace (fresh, zero-filled)
    K_ref, V_ref = K.clone(), V.clone()
    ws = torch.zeros(m.medusa_tree_attn_workspace(t_g, B, w.n_q_heads, m.KVCache(K_ref, V_ref), max_prefix),
                     dtype=torch.uint8, device="cuda")
    ref, ref_lse, ref_st = m.medusa_tree_attn_verify(t_g, q, k, v, m.KVCache(K_ref, V_ref), L, max_prefix,
                                                     rope_base=w.rope_base, want_lse=True, ws=ws)
    torch.cuda.synchronize()
    assert (ref_st.cpu().numpy() == 0).all()

    is_f32 = w.dtype == "f32"
    for call in range(2):                      # the second call sees the first call's leftovers
        K_s, V_s = K.clone(), V.clone()
        out = torch.full((B, N, w.n_q_heads, w.head_dim), float("nan"), device="cuda")
        lse = torch.full((B, N, w.n_q_heads), float("nan"), device="cuda")
        status = torch.full((B,), 99, dtype=torch.int32, device="cuda")
        cache_s = m.KVCache(K_s, V_s)
        if mirror:
            cache_s.add_mirror()
        torch.cuda.synchronize()
        torch_bytes, (free_bytes, _) = torch.cuda.memory_allocated(), torch.cuda.mem_get_info()
        rc = _static_call(m, t_g, q, k, v, cache_s, L, max_prefix, w.rope_base, out, lse, status)
        assert rc == nat.OK, nat.lib().medusa_status_string(rc)
        torch.cuda.synchronize()
        if call == 1:
            # nothing allocated by the call: neither through torch nor from the device
            # (the first call may still load kernels lazily, so the second is measured)
            assert torch.cuda.memory_allocated() == torch_bytes
            assert torch.cuda.mem_get_info()[0] == free_bytes
        assert (status.cpu().numpy() == 0).all()
        gu.float_parity(out, ref, is_f32, f"static entry, call {call}")
        gu.float_parity(lse, ref_lse, True, f"static entry lse, call {call}")
        assert torch.equal(K_s, K_ref) and torch.equal(V_s, V_ref)     # same staged rows
        if mirror:
            assert torch.equal(out, ref) and torch.equal(lse, ref_lse)
            for c16, c in ((cache_s.k_f16, K_s), (cache_s.v_f16, V_s)):
                assert torch.equal(c16, c.to(torch.float16))


def test_static_scratch_refuses_oversized_shapes(m):
    """A batch whose split partials need more than the fixed 32 MiB is refused up front
    (fp32 caches take the CUDA-core path, whose splits merge through this scratch)."""
    w, t_g, q, k, v, K, V, lengths = _setup(m, "longctx-341", batch=4, prefix_len=64, n_q_heads=64,
                                            n_kv_heads=16, dtype="f32")
    nat = m.api.nat
    cache = m.KVCache(K, V)
    need = m.medusa_tree_attn_workspace(t_g, w.batch, w.n_q_heads, cache, 64)
    assert need > nat.ATTN_STATIC_SCRATCH_BYTES
    out = torch.full((w.batch, t_g.n_rows, w.n_q_heads, w.head_dim), 3.0, device="cuda")
    lse = torch.empty((w.batch, t_g.n_rows, w.n_q_heads), device="cuda")
    status = torch.full((w.batch,), 99, dtype=torch.int32, device="cuda")
    K_before = K.clone()
    rc = _static_call(m, t_g, q, k, v, cache, gu.device_tensor(lengths, torch.int32), 64, w.rope_base,
                      out, lse, status)
    torch.cuda.synchronize()
    assert rc == nat.EWORKSPACE
    assert (out == 3.0).all() and (status == 99).all() and torch.equal(K, K_before)
