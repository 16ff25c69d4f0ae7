"""CPU tests of libmedusa_gb300.so: exported symbols and the host-side template
construction, compared bit for bit with the oracle.  No GPU calls."""
import ctypes as C
import os
import re

import numpy as np
import pytest

import synth
from oracle import tree as otree
from oracle.round import template_for

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="session")
def native():
    from medusa_speculative_tree_gb300 import build, _native
    build.build()
    return _native


def header_functions():
    src = open(os.path.join(ROOT, "include", "medusa_gb300.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(medusa_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(native):
    names = header_functions()
    assert len(names) >= 15
    lib = C.CDLL(native.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(native.EXPORTED)
    assert native.lib().medusa_abi_version() == 5
    assert native.lib().medusa_status_string(-2).decode() == "cache capacity exceeded"


def compare(t_nat, t_ora):
    assert t_nat.n_rows == t_ora.n_rows
    assert t_nat.max_depth == t_ora.max_depth
    assert t_nat.n_paths == t_ora.n_paths
    assert (t_nat.slot == t_ora.slot).all()
    assert (t_nat.depth == t_ora.depth).all()
    assert (t_nat.parent == t_ora.parent).all()
    assert (t_nat.retrieve == t_ora.retrieve).all()
    N = t_ora.n_rows
    anc = t_nat.anc
    for u in range(N):
        bits = [(int(anc[u, v // 64]) >> (v % 64)) & 1 for v in range(N)]
        assert bits == list(t_ora.mask[u].astype(int))
    kids = np.zeros(N, dtype=int)
    for u in range(1, N):
        kids[t_ora.parent[u]] += 1
    assert list(t_nat.internal) == [u for u in range(N) if kids[u] > 0]


@pytest.mark.parametrize("name", synth.WORKLOAD_ORDER)
def test_workload_templates_match_oracle(native, name):
    from medusa_speculative_tree_gb300.api import Template, medusa_tree_greedy, medusa_tree_regular
    w = synth.WORKLOADS[name]
    acc = synth.rank_accuracy(w.n_heads, 10)
    t_ora = template_for(w.template, w.topk, w.n_heads, acc)
    if w.template[0] == "regular":
        paths = medusa_tree_regular(w.template[1])
        assert paths == otree.regular_paths(w.template[1])
    else:
        paths = medusa_tree_greedy(acc[:, :w.template[2]], w.template[1])
        assert paths == otree.greedy_tree(acc[:, :w.template[2]], w.template[1])
    compare(Template(paths, w.topk, w.n_heads), t_ora)


@pytest.mark.parametrize("seed", range(8))
def test_random_templates_match_oracle(native, seed):
    from medusa_speculative_tree_gb300.api import Template
    rng = np.random.default_rng(100 + seed)
    topk = int(rng.integers(1, 8))
    paths = set()
    for _ in range(int(rng.integers(0, 120))):
        L = int(rng.integers(1, 6))
        p = tuple(int(x) for x in rng.integers(0, topk, size=L))
        for t in range(1, L + 1):
            paths.add(p[:t])
    paths = list(paths)
    rng.shuffle(paths)
    compare(Template(paths, topk), otree.compile_template(paths, topk))


@pytest.mark.parametrize("K,R,budget", [(3, 4, 10), (4, 10, 63), (4, 10, 255), (2, 3, 50)])
def test_greedy_matches_oracle(native, K, R, budget):
    from medusa_speculative_tree_gb300.api import medusa_tree_greedy
    rng = np.random.default_rng(K * 31 + R)
    acc = np.sort(rng.uniform(0.0, 1.0, size=(K, R)), axis=1)[:, ::-1].copy()
    assert medusa_tree_greedy(acc, budget) == otree.greedy_tree(acc, budget)
    acc2 = synth.rank_accuracy(K, R)             # many mathematically tied weights
    assert medusa_tree_greedy(acc2, budget) == otree.greedy_tree(acc2, budget)


@pytest.mark.parametrize("widths", [(1,), (3,), (2, 3), (4, 4, 4, 4), (10, 1, 2), (1, 1, 1, 1, 1, 1, 1, 1)])
def test_regular_size_query_and_paths(native, widths):
    """The size query gives sum_k prod_{i<=k} s_i (the oracle's count of non-root
    nodes), the paths equal the oracle's, and a buffer one path short is refused."""
    lib = native.lib()
    K = len(widths)
    w = np.ascontiguousarray(widths, dtype=np.int32)
    n = C.c_int32(-1)
    assert lib.medusa_tree_regular(w.ctypes.data, K, None, 0, C.byref(n)) == native.OK
    assert n.value == otree.regular_node_count(widths) == len(otree.regular_paths(widths))
    out = np.full((n.value, K), -1, dtype=np.int32)
    assert lib.medusa_tree_regular(w.ctypes.data, K, out.ctypes.data, n.value, C.byref(n)) == native.OK
    assert [tuple(int(x) for x in row if x >= 0) for row in out] == otree.regular_paths(widths)
    short = np.full((max(n.value - 1, 1), K), -1, dtype=np.int32)
    assert lib.medusa_tree_regular(w.ctypes.data, K, short.ctypes.data, n.value - 1, C.byref(n)) == native.EWORKSPACE


@pytest.mark.parametrize("bad", [[(0, 1)], [(0,), (0,)], [(0,), (9,)], [(0,), (0, 0), (0, 0, 0)]])
def test_compile_rejects(native, bad):
    from medusa_speculative_tree_gb300.api import Template
    with pytest.raises(native.MedusaError) as e:
        Template(bad, topk=4, n_heads=2)
    assert e.value.status == native.ETEMPLATE


def test_root_only_and_limits(native):
    from medusa_speculative_tree_gb300.api import Template
    t = Template([], topk=3)
    assert t.n_rows == 1 and t.n_paths == 1 and list(t.retrieve[0]) == [0]
    lib = native.lib()
    assert lib.medusa_tree_greedy(None, 1, 1, 1, None, None) == native.EINVAL
    out = native.MedusaTree()
    assert lib.medusa_tree_compile(None, 1, 1, 4, 0, None, 0, C.byref(out)) == native.EINVAL


def test_round_desc_layout_matches_header(native, tmp_path):
    """The ctypes medusa_round_desc (and the structs inside it) has the C layout:
    size and every field offset, from a program compiled against the header."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    structs = [("medusa_round_desc", native.MedusaRoundDesc), ("medusa_tree_t", native.MedusaTree),
               ("medusa_kv_t", native.MedusaKV)]
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "medusa_gb300.h"', "int main(void) {"]
    for cname, py in structs:
        lines.append('printf("%s size %%zu\\n", sizeof(%s));' % (cname, cname))
        for f, _ in py._fields_:
            lines.append('printf("%s %s %%zu\\n", offsetof(%s, %s));' % (cname, f, cname, f))
    lines += ["return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.check_call([cc, "-std=c99", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)])
    out = subprocess.check_output([str(exe)]).decode().split("\n")
    got = {}
    for ln in out:
        if ln.strip():
            a, b, c = ln.split()
            got[(a, b)] = int(c)
    for cname, py in structs:
        assert got[(cname, "size")] == C.sizeof(py), cname
        for f, _ in py._fields_:
            assert got[(cname, f)] == getattr(py, f).offset, (cname, f)


def test_round_create_rejects_bad_arguments_without_a_gpu(native):
    """Host-visible checks come before any CUDA call: a missing descriptor, output
    handle or workspace is refused with MEDUSA_EINVAL and no round."""
    lib = native.lib()
    handle = C.c_void_p(1234)
    assert lib.medusa_round_create(None, None, 0, None, C.byref(handle)) == native.EINVAL
    assert handle.value is None
    desc = native.MedusaRoundDesc()
    assert lib.medusa_round_workspace(C.byref(desc)) == 0
    assert lib.medusa_round_workspace(None) == 0
    assert lib.medusa_round_create(C.byref(desc), None, 0, None, None) == native.EINVAL
    assert lib.medusa_round_create(C.byref(desc), None, 0, None, C.byref(handle)) == native.EINVAL
    assert lib.medusa_round_launch(None, None) == native.EINVAL
    assert lib.medusa_round_destroy(None) == native.EINVAL


def test_kv_compact_layers_checks_layers_without_a_gpu(native):
    """Host-visible checks of medusa_kv_compact_layers come before any CUDA call:
    layers that differ in anything but k and v, no layers, or L_out aliasing L are
    refused with MEDUSA_EINVAL."""
    from medusa_speculative_tree_gb300.api import Template
    lib = native.lib()
    t = Template([(0,), (1,), (0, 0)], 2)
    fake = lambda i: C.c_void_p(4096 * (i + 1))       # never dereferenced: the checks fail first
    def layer(i, head_dim=64):
        c = native.MedusaKV()
        c.k, c.v, c.dtype, c.n_kv_heads, c.head_dim, c.capacity = fake(2 * i).value, fake(2 * i + 1).value, 0, 2, head_dim, 64
        c.page_size, c.block_table, c.max_blocks, c.n_pages = 0, None, 0, 0
        return c
    L, a, rows, L_out, st = (fake(100 + i) for i in range(5))
    arr = (native.MedusaKV * 3)(layer(0), layer(1), layer(2, head_dim=128))
    assert lib.medusa_kv_compact_layers(arr, 3, C.byref(t.host), 2, L, a, rows, L_out, st, None) == native.EINVAL
    arr = (native.MedusaKV * 2)(layer(0), layer(1))
    assert lib.medusa_kv_compact_layers(arr, 0, C.byref(t.host), 2, L, a, rows, L_out, st, None) == native.EINVAL
    assert lib.medusa_kv_compact_layers(arr, 2, C.byref(t.host), 2, L, a, rows, L, st, None) == native.EINVAL
    assert lib.medusa_kv_compact_layers(None, 2, C.byref(t.host), 2, L, a, rows, L_out, st, None) == native.EINVAL


def test_fp16_mirror_checks_without_a_gpu(native):
    """A cache's fp16 mirror is checked before any CUDA call: half a mirror, a mirror
    of an fp32 cache, a misaligned mirror, medusa_kv_mirror_sync without a mirror or
    with B < 1 for a contiguous cache, and layers of which only some have a mirror, are
    refused with MEDUSA_EINVAL."""
    from medusa_speculative_tree_gb300.api import Template
    lib = native.lib()
    t = Template([(0,), (1,), (0, 0)], 2)
    fake = lambda i: C.c_void_p(4096 * (i + 1))       # never dereferenced: the checks fail first
    def cache(i, dtype=native.BF16, k16=True, v16=True, k16_off=0):
        c = native.MedusaKV()
        c.k, c.v, c.dtype, c.n_kv_heads, c.head_dim, c.capacity = fake(4 * i).value, fake(4 * i + 1).value, dtype, 2, 128, 64
        c.page_size, c.block_table, c.max_blocks, c.n_pages = 0, None, 0, 0
        c.k_f16 = fake(4 * i + 2).value + k16_off if k16 else None
        c.v_f16 = fake(4 * i + 3).value if v16 else None
        return c
    L, a, rows, L_out, st = (fake(100 + i) for i in range(5))
    for bad in (cache(0, v16=False), cache(0, k16=False), cache(0, dtype=native.F32), cache(0, k16_off=8)):
        assert lib.medusa_kv_compact(C.byref(bad), C.byref(t.host), 2, L, a, rows, L_out, st, None) == native.EINVAL
        assert lib.medusa_kv_mirror_sync(C.byref(bad), 2, None) == native.EINVAL
    assert lib.medusa_kv_mirror_sync(C.byref(cache(0, k16=False, v16=False)), 2, None) == native.EINVAL
    assert lib.medusa_kv_mirror_sync(C.byref(cache(0)), 0, None) == native.EINVAL
    assert lib.medusa_kv_mirror_sync(None, 2, None) == native.EINVAL
    arr = (native.MedusaKV * 2)(cache(0), cache(1, k16=False, v16=False))
    assert lib.medusa_kv_compact_layers(arr, 2, C.byref(t.host), 2, L, a, rows, L_out, st, None) == native.EINVAL


def test_commit_and_hidden_acceptance_checks_without_a_gpu(native):
    """Host-visible checks that return before any CUDA call: compaction and the fused
    commit refuse L_out aliasing L (the kv-head CTAs of a sequence would race on it);
    acceptance from hidden states refuses a hidden size that is not a multiple of 64."""
    from medusa_speculative_tree_gb300.api import Template
    lib = native.lib()
    t = Template([(0,), (1,), (0, 0)], 2)
    fake = lambda i: C.c_void_p(4096 * (i + 1))       # never dereferenced: the checks fail first
    c = native.MedusaKV()
    c.k, c.v, c.dtype, c.n_kv_heads, c.head_dim, c.capacity = fake(0).value, fake(1).value, 0, 2, 64, 64
    c.page_size, c.block_table, c.max_blocks, c.n_pages = 0, None, 0, 0
    L, a, rows, st = fake(10), fake(11), fake(12), fake(13)
    assert lib.medusa_kv_compact(C.byref(c), C.byref(t.host), 2, L, a, rows, L, st, None) == native.EINVAL
    outs = [fake(20 + i) for i in range(5)]
    ws = fake(30)
    assert lib.medusa_tree_accept_commit(C.byref(t.host), 2, 100, fake(31), native.F32, fake(32), native.GREEDY,
                                         1.0, 0.09, 0.3, 0, C.byref(c), L, *outs, L, st, ws, 1 << 20,
                                         None) == native.EINVAL
    assert lib.medusa_tree_accept_hidden(C.byref(t.host), 2, 100, 100, fake(40), fake(41), fake(42), native.GREEDY,
                                         1.0, 0.09, 0.3, *outs, ws, 1 << 20, None) == native.EUNSUPPORTED
    assert lib.medusa_tree_accept_hidden(C.byref(t.host), 2, 100, 128, None, fake(41), fake(42), native.GREEDY,
                                         1.0, 0.09, 0.3, *outs, ws, 1 << 20, None) == native.EINVAL


def test_template_batches_check_arguments_without_a_gpu(native):
    """Host-visible checks of the per-sequence template calls come before any CUDA call:
    medusa_tree_greedy_device refuses bad shapes (MEDUSA_EINVAL), a search larger than
    its shared-memory frontier (MEDUSA_EUNSUPPORTED) and a short buffer
    (MEDUSA_EWORKSPACE); medusa_tree_batch refuses mixed topk and nested batches;
    medusa_tree_upload refuses a batch descriptor."""
    lib = native.lib()
    fake = C.c_void_p(1 << 20)                  # never dereferenced: every call below fails its checks
    out = native.MedusaTree()
    K, R, budget = 4, 10, 63
    need = lib.medusa_tree_greedy_device_bytes(2, K, R, budget)
    assert need > 0
    assert lib.medusa_tree_greedy_device_bytes(2, 0, R, budget) == 0
    g = lambda B, K_, R_, bud, topk, nbytes: lib.medusa_tree_greedy_device(fake, B, K_, R_, bud, topk, fake, nbytes,
                                                                          fake, None, C.byref(out), None)
    assert g(2, K, R, budget, 10, need - 1) == native.EWORKSPACE
    assert g(2, K, 11, budget, 10, need) == native.EINVAL          # ranks beyond topk
    assert g(0, K, R, budget, 10, need) == native.EINVAL
    assert g(2, K, 32, 255, 32, 1 << 30) == native.EUNSUPPORTED     # 32 x 256 entries > 6144
    host = m_tree(native, [(0,), (1,)], 2)
    other = m_tree(native, [(0,)], 3)
    arr = (native.MedusaTree * 2)(host, other)
    assert lib.medusa_tree_batch(arr, 2, fake, 2 * C.sizeof(native.MedusaTree), C.byref(out), None) == native.EINVAL
    nested = native.MedusaTree.from_buffer_copy(bytes(host))
    nested.per_seq = fake.value
    arr2 = (native.MedusaTree * 1)(nested)
    assert lib.medusa_tree_batch(arr2, 1, fake, C.sizeof(native.MedusaTree), C.byref(out), None) == native.EINVAL
    assert lib.medusa_tree_upload(C.byref(nested), fake, fake, 1 << 20, C.byref(out), None) == native.EINVAL


_KEEP = []


def m_tree(native, paths, topk):
    """A host-compiled template (its blob kept alive for the test)."""
    lib = native.lib()
    n, L = len(paths), max(len(p) for p in paths)
    arr = np.full((n, L), -1, dtype=np.int32)
    for i, p in enumerate(paths):
        arr[i, :len(p)] = p
    blob = np.zeros(lib.medusa_tree_bytes(n, L) // 8 + 2, dtype=np.uint64)
    t = native.MedusaTree()
    assert lib.medusa_tree_compile(arr.ctypes.data, n, L, topk, 0, blob.ctypes.data, blob.nbytes, C.byref(t)) == 0
    _KEEP.append(blob)
    return t
