"""Benchmark of one Medusa verify round on GB300.

A step is one whole round of the hot path on one batch of synthetic input:
medusa_heads_topk -> medusa_tree_fill -> medusa_tree_attn_verify ->
medusa_tree_accept -> medusa_kv_compact.  The headline workload is the
long-context round, the largest configuration (bf16, batch 1, the full 341-row
Cartesian tree (4,4,4,4), GQA 64/8 heads, L = 32768, K = 4 heads over d = 8192 and
V = 128256); the line also carries the other four workloads under `per_workload`.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl native|reference]

Prints one JSON line (rank 0).  `value` is microseconds per verify round for the
whole job (N replicas run one round each per step, so value = step time / N).
--impl reference times the fp64 CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np
import torch

import synth

METRIC = "µs per Medusa verify round; tree nodes/s; tree-attn HBM GB/s as % of GB300 peak"
UNIT = "us/round"


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), "measured"
    return 6800.0, 1900.0, "fallback"


# ----------------------------------------------------------------------------- distributed

def dist_setup(backend):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group(backend=backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, ws: int, device) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", str(self.index)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.15)
        return self

    def __exit__(self, *a):
        self.rows = []
        if self.proc is None:
            return False
        time.sleep(0.15)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) >= 9:
                self.rows.append(f)
        return False

    def summary(self):
        if not getattr(self, "rows", None):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in self.rows:
            for i, n in enumerate(names):
                if r[5 + i].lower() == "active":
                    reasons.add(n)
        load = [s for s in sm if s > 0.5 * max(sm)] if sm else []
        return {"sm_mhz": statistics.median(load) if load else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(self.rows)}


# ----------------------------------------------------------------------------- workload

class Round:
    """Device-resident inputs and outputs of one verify round for a workload.  A bf16
    cache carries an fp16 mirror (filled once here, as a prefill would; every round's
    cache writes keep it in step) unless mirror=False."""

    def __init__(self, m, w: synth.Workload, dev, mirror=None):
        self.m, self.w, self.dev = m, w, dev
        acc = synth.rank_accuracy(w.n_heads, 10)
        if w.template[0] == "regular":
            paths = m.medusa_tree_regular(w.template[1])
        else:
            paths = m.medusa_tree_greedy(acc[:, :w.template[2]], w.template[1])
        self.tmpl = m.Template(paths, w.topk, w.n_heads, device=dev)
        N = self.N = self.tmpl.n_rows
        self.h, self.w1, self.w2, self.w_lm = synth.head_weights(w, device=dev)
        self.q, self.k, self.v = synth.tree_qkv(w, N, device=dev)
        lengths = synth.prefix_lengths(w)
        self.lengths = lengths
        self.L = torch.tensor(lengths, dtype=torch.int32, device=dev)
        self.max_L = int(lengths.max())
        dt = w.torch_dtype
        if w.page_size:
            lay = synth.paged_layout(w, lengths, N)
            self.K = torch.zeros((lay.n_pages, w.n_kv_heads, lay.page_size, w.head_dim), dtype=dt, device=dev)
            self.V = torch.zeros_like(self.K)
            ks, vs = synth.prefix_kv(w, lengths, device=dev)
            bt = torch.tensor(lay.block_table, dtype=torch.int32, device=dev)
            for b, L in enumerate(lengths):
                L = int(L)
                nb = (L + 15) // 16
                pages = bt[b, :nb].long()
                kp = torch.zeros((nb * 16, w.n_kv_heads, w.head_dim), dtype=dt, device=dev)
                vp = torch.zeros_like(kp)
                kp[:L] = ks[b].transpose(0, 1)
                vp[:L] = vs[b].transpose(0, 1)
                self.K[pages] = kp.view(nb, 16, w.n_kv_heads, w.head_dim).transpose(1, 2)
                self.V[pages] = vp.view(nb, 16, w.n_kv_heads, w.head_dim).transpose(1, 2)
            self.cache = m.KVCache(self.K, self.V, block_table=bt)
        else:
            cap = self.max_L + N + 16
            self.K = torch.zeros((w.batch, w.n_kv_heads, cap, w.head_dim), dtype=dt, device=dev)
            self.V = torch.zeros_like(self.K)
            ks, vs = synth.prefix_kv(w, lengths, device=dev)
            for b, L in enumerate(lengths):
                self.K[b, :, :int(L)] = ks[b]
                self.V[b, :, :int(L)] = vs[b]
            self.cache = m.KVCache(self.K, self.V)
        if mirror if mirror is not None else w.dtype == "bf16":
            self.cache.add_mirror()
        # target logits, argmax planted on the candidates the heads actually propose
        root, pool = m.medusa_heads_topk(self.h, self.w1, self.w2, self.w_lm, w.topk)
        logits = synth.target_logits(w, N)
        if w.plant:
            synth.plant_argmax(logits, pool.cpu().numpy(), self.tmpl.depth, acc, synth.plant_uniforms(w, N))
        self.logits = logits.to(dev)
        self.mode = w.accept[0]
        self.out = torch.empty((w.batch, N, w.n_q_heads, w.head_dim), dtype=torch.float32, device=dev)
        nb = m.medusa_tree_attn_workspace(self.tmpl, w.batch, w.n_q_heads, self.cache, self.max_L)
        self.attn_ws = torch.zeros(nb, dtype=torch.uint8, device=dev)
        torch.cuda.synchronize(dev)

    # the five calls of one round; returns the accept dict and L_out
    def heads(self):
        return self.m.medusa_heads_topk(self.h, self.w1, self.w2, self.w_lm, self.w.topk)

    def fill(self, root, pool):
        return self.m.medusa_tree_fill(self.tmpl, root, pool, self.L)

    def attn(self):
        return self.m.medusa_tree_attn_verify(self.tmpl, self.q, self.k, self.v, self.cache, self.L, self.max_L,
                                              rope_base=self.w.rope_base, out=self.out, ws=self.attn_ws)

    def accept(self, tokens, logits=None, mode=None):
        return self.m.medusa_tree_accept(self.tmpl, self.logits if logits is None else logits, tokens,
                                         mode or self.mode, epsilon=self.w.epsilon, delta=self.w.delta)

    def compact(self, r):
        return self.m.medusa_kv_compact(self.cache, self.tmpl, self.L, r["accept_len"], r["out_rows"])

    def step(self):
        root, pool = self.heads()
        tokens, _ = self.fill(root, pool)
        self.attn()
        r = self.accept(tokens)
        L_out, _ = self.compact(r)
        return r, L_out

    # algorithmic bytes / flops
    def head_bytes(self):
        w = self.w
        eb = 4 if w.dtype == "f32" else 2
        weights = (w.n_heads * w.hidden * w.hidden + (w.n_heads + 1) * w.vocab * w.hidden) * eb
        return weights + w.batch * w.hidden * eb

    def attn_bytes(self):
        w = self.w
        eb = 4 if w.dtype == "f32" else 2
        prefix = 2 * int(self.lengths.sum()) * w.n_kv_heads * w.head_dim * eb
        tree_in = w.batch * self.N * (w.n_q_heads + 2 * w.n_kv_heads) * w.head_dim * eb
        staged = 2 * w.batch * self.N * w.n_kv_heads * w.head_dim * eb
        outb = w.batch * self.N * w.n_q_heads * w.head_dim * 4
        return prefix + tree_in + staged + outb

    def round_bytes(self, accept_len):
        """Algorithmic HBM bytes of the whole round: the head weights and hidden rows,
        the template fill, the attention call, the logits of the internal rows that
        acceptance reads, and the K/V rows that compaction reads and writes (a + 1 rows
        per sequence, all KV heads)."""
        w = self.w
        eb = 4 if w.dtype == "f32" else 2
        fill = w.batch * (self.N * 8 + (1 + w.n_heads * w.topk) * 4 + 4)
        accept = w.batch * (self.tmpl.n_internal * w.vocab * eb + self.N * 4)
        published = int((accept_len.to(torch.int64) + 1).sum())
        compact = published * 2 * w.n_kv_heads * w.head_dim * eb * 2
        return self.head_bytes() + fill + self.attn_bytes() + accept + compact

    def attn_flops(self):
        w = self.w
        return 4.0 * w.head_dim * float(self.lengths.sum()) * self.N * w.n_q_heads

    def launches_per_step(self):
        """Kernels of this library launched by one step (memsets not counted)."""
        w = self.w
        bf16 = w.dtype == "bf16"
        T = w.batch
        stream_d = (w.hidden <= 4096 and w.hidden % 256 == 0) or (w.hidden <= 8192 and w.hidden % 512 == 0)
        if bf16 and T == 1 and stream_d and w.n_heads >= 1:
            heads = 1                                   # one persistent weight stream with top-k
        elif bf16 and T >= 2 and w.hidden % 64 == 0 and w.n_heads >= 1:
            per_pass = 128 if T <= 128 else 256        # pair passes, else wide passes
            heads = math.ceil(T / per_pass) + 1        # one tensor-core stream per pass; then top-k
        else:
            tpp = 1
            fit = max(1, min(16, (160 * 1024) // (w.hidden * 4)))
            while tpp * 2 <= min(T, fit):
                tpp *= 2
            heads = 2 * math.ceil(T / tpp) + 1         # two GEMV kernels per pass, then top-k
        accept = 2 if self.tmpl.n_internal > 0 else 1
        return heads + 1 + 1 + accept + 1


# DRAM bytes (read + write) of one heads launch, from an ncu capture of the current
# kernel on that workload; absent for workloads not captured.
HEADS_TRAFFIC = {"longctx-341": 11_044_705_792 + 7_362_560}
# the same for the attention launch (dram__bytes_read.sum + dram__bytes_write.sum)
ATTN_TRAFFIC = {"vicuna7b-64": 35_210_752 + 0}


def heads_all_rows(rd, stream, peak_tflops):
    """medusa_heads_topk with every tree row as a hidden row (T = B N), the variant in which
    the heads are a tensor-core contraction.  `frac` is the method's useful rate, 2 T
    flops per weight element, over the bf16 peak.  bf16 with 2 <= T <= 128 runs on the
    tensor cores with W1 h and W_LM h on the rows of h and W2 z on z as bf16 pairs (hi,
    lo), so the W2 MMAs execute twice the useful flops; more rows run wide passes of up
    to 256 single rows (z in fp16), which execute the useful flops.  The executed rate is
    reported beside the useful one."""
    w = rd.w
    T = w.batch * rd.N                                  # every tree row of every sequence
    h = synth.normal((T, w.hidden), 1.0, w.seed, "h", rd.dev, w.torch_dtype, sub=1)
    call = lambda: rd.m.medusa_heads_topk(h, rd.w1, rd.w2, rd.w_lm, w.topk)
    for _ in range(3):
        call()
    torch.cuda.synchronize(rd.dev)
    n = 5
    us = 1e3 * time_loop(call, n, stream) / n
    elems = rd.w1.numel() + rd.w2.numel() + rd.w_lm.numel()
    useful = 2.0 * T * elems / (us * 1e-6) / 1e12
    mma = w.dtype == "bf16" and T >= 2
    wide = mma and T > 128
    w2_share = rd.w2.numel() / elems
    executed = useful * ((1.0 + w2_share) if mma and not wide else 1.0)
    passes = (math.ceil(T / 256) if wide else math.ceil(T / 128)) if mma else 1
    return {"T": T, "us": us, "useful_tflops": useful, "executed_tflops": executed,
            "peak_tflops": peak_tflops, "frac": useful / peak_tflops, "executed_frac": executed / peak_tflops,
            "weight_passes": passes, "hbm_gbs": passes * rd.head_bytes() / (us * 1e-6) / 1e9}


def compact_all_layers(rd, results, stream, flush, n_layers=32):
    """The winning rows committed in n_layers caches of this workload's layout: one
    medusa_kv_compact_layers call against n_layers medusa_kv_compact calls, each side a
    CUDA graph replayed after an L2 flush."""
    m = rd.m
    caches = [m.KVCache(torch.empty_like(rd.K), torch.empty_like(rd.V), block_table=rd.cache.block_table)
              for _ in range(n_layers)]
    a, rows = results.accept_len, results.out_rows
    one = lambda: m.medusa_kv_compact_layers(caches, rd.tmpl, rd.L, a, rows)
    each = lambda: [m.medusa_kv_compact(c, rd.tmpl, rd.L, a, rows) for c in caches]
    one()
    each()
    torch.cuda.synchronize(rd.dev)
    graphs = {}
    for name, fn in (("one", one), ("each", each)):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        graphs[name] = g
    us = {}
    for name, g in graphs.items():
        tot = 0.0
        for _ in range(10):
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            e1.synchronize()
            tot += e0.elapsed_time(e1) * 1e3
        us[name] = tot / 10
    w = rd.w
    eb = 4 if w.dtype == "f32" else 2
    moved = int((a.to(torch.int64) + 1).sum()) * 2 * w.n_kv_heads * w.head_dim * eb * 2 * n_layers
    del caches, graphs
    torch.cuda.empty_cache()
    return {"layers": n_layers, "one_call_us": us["one"], "per_layer_calls_us": us["each"],
            "bytes_read_and_written": moved}


def accept_hidden(rd, results, stream, flush, hbm_peak):
    """Acceptance with the target's vocabulary projection folded in (hidden states of
    every tree row, bf16, seeded N(0, 1)) on this workload's W_LM and tree tokens: a
    CUDA graph replayed after an L2 flush.  Algorithmic bytes: W_LM once (passes of
    256 internal rows run as interleaved CTA sets that share each group through L2)."""
    w = rd.w
    if w.dtype != "bf16":
        return None
    m = rd.m
    hidden = synth.normal((w.batch, rd.N, w.hidden), 1.0, w.seed, "h", rd.dev, w.torch_dtype, sub=2)
    tokens = results.tokens
    call = lambda: m.medusa_tree_accept_hidden(rd.tmpl, hidden, rd.w_lm, tokens, rd.mode, epsilon=w.epsilon,
                                               delta=w.delta)
    call()
    torch.cuda.synchronize(rd.dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    tot = 0.0
    reps = 10
    for _ in range(reps):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        e1.synchronize()
        tot += e0.elapsed_time(e1) * 1e3
    us = tot / reps
    rows = w.batch * rd.tmpl.n_internal
    passes = math.ceil(rows / 256)
    wbytes = rd.w_lm.numel() * rd.w_lm.element_size()
    gbs = wbytes / (us * 1e-6) / 1e9
    del g
    return {"internal_rows": rows, "us": us, "w_lm_passes": passes, "bytes": wbytes, "hbm_gbs": gbs,
            "frac": gbs / hbm_peak, "tflops": 2.0 * rows * w.hidden * w.vocab / (us * 1e-6) / 1e12}


def time_loop(fn, steps, stream):
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        fn()
    end.record(stream)
    end.synchronize()
    return start.elapsed_time(end)            # ms


class RoundGraphs:
    """The timed step is the library's own round graph (medusa_round_create records
    the five calls; each step is one medusa_round_launch).  For the per-stage split
    each call is also captured alone in a torch CUDA graph: the library's calls are
    stream-ordered and neither allocate nor synchronise, so they capture as they are;
    workspaces and outputs are created by the warm-up calls before capture."""

    NAMES = ["heads", "fill", "attn", "accept", "compact"]

    def __init__(self, rd: Round, dev, fuse_commit: bool = False):
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            for _ in range(3):
                rd.step()
        torch.cuda.current_stream(dev).wait_stream(side)
        torch.cuda.synchronize(dev)
        w = rd.w
        self.native = rd.m.MedusaRound(rd.tmpl, rd.h, rd.w1, rd.w2, rd.w_lm, w.topk, rd.L, rd.q, rd.k, rd.v,
                                       rd.cache, rd.max_L, rd.logits, mode=rd.mode, rope_base=w.rope_base,
                                       epsilon=w.epsilon, delta=w.delta, fuse_commit=fuse_commit)
        self.stage = {n: torch.cuda.CUDAGraph() for n in self.NAMES}
        with torch.cuda.graph(self.stage["heads"]):
            root, pool = rd.heads()
        with torch.cuda.graph(self.stage["fill"]):
            tokens, _ = rd.fill(root, pool)
        with torch.cuda.graph(self.stage["attn"]):
            rd.attn()
        with torch.cuda.graph(self.stage["accept"]):
            r = rd.accept(tokens)
        with torch.cuda.graph(self.stage["compact"]):
            rd.compact(r)
        self._stage_keep = (root, pool, tokens, r)
        torch.cuda.synchronize(dev)

    def step(self):
        self.native.launch()

    def stage_times(self, reps: int, stream, flush):
        """Per-stage device time (µs, mean), CUDA events on the replay stream, with the
        L2 flushed before every stage so that each streams its inputs from HBM."""
        tot = {n: 0.0 for n in self.NAMES}
        for _ in range(reps):
            ev = []
            for n in self.NAMES:
                flush()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                self.stage[n].replay()
                b.record(stream)
                ev.append((n, a, b))
            ev[-1][2].synchronize()
            for n, a, b in ev:
                tot[n] += a.elapsed_time(b) * 1e3
        return {n: tot[n] / reps for n in self.NAMES}


def e2e_loop(rd: Round, steps: int, stream):
    """Same round through the public API with per-step inputs copied from pinned host
    memory and the published result read back (both inside the timed region).  Two
    rounds (medusa_round_create, as the timed step) are bound to two sets of input
    buffers and take the steps in turn.  On a second stream, once the round two steps
    back has finished, its published tokens and L_out are copied to the host and this
    step's inputs into its set, which overlaps the previous step's round; the step's
    round waits for those copies.  The last two rounds' results are read back before
    the timed region closes."""
    w = rd.w
    hosts = [x.cpu().pin_memory() for x in (rd.h, rd.L, rd.q, rd.k, rd.v, rd.logits)]
    sets = [[torch.empty_like(x, device=rd.dev) for x in hosts] for _ in range(2)]
    for st in sets:
        for dst, src in zip(st, hosts):
            dst.copy_(src)
    rounds = [rd.m.MedusaRound(rd.tmpl, st[0], rd.w1, rd.w2, rd.w_lm, w.topk, st[1], st[2], st[3], st[4], rd.cache,
                               rd.max_L, st[5], mode=rd.mode, rope_base=w.rope_base, epsilon=w.epsilon,
                               delta=w.delta) for st in sets]
    tok_host = [torch.empty_like(r.out_tokens, device="cpu").pin_memory() for r in rounds]
    L_host = [torch.empty_like(r.L_out, device="cpu").pin_memory() for r in rounds]
    h2d = sum(x.numel() * x.element_size() for x in hosts)
    d2h = sum(x.numel() * x.element_size() for x in (tok_host[0], L_host[0]))
    side = torch.cuda.Stream(rd.dev)
    ready = [torch.cuda.Event(), torch.cuda.Event()]
    done = [torch.cuda.Event(), torch.cuda.Event()]
    launched = [False, False]
    step = [0]

    def read_back(s):
        # copies only (no kernel on this stream: the heads kernel holds every SM)
        tok_host[s].copy_(rounds[s].out_tokens, non_blocking=True)
        L_host[s].copy_(rounds[s].L_out, non_blocking=True)

    def one():
        s = step[0] & 1
        step[0] += 1
        main = torch.cuda.current_stream(rd.dev)
        with torch.cuda.stream(side):
            side.wait_event(done[s])                 # the round two steps back has finished
            if launched[s]:
                read_back(s)
            for dst, src in zip(sets[s], hosts):
                dst.copy_(src, non_blocking=True)
            ready[s].record(side)
        main.wait_event(ready[s])
        rounds[s].launch(main)
        launched[s] = True
        done[s].record(main)

    def finish():
        main = torch.cuda.current_stream(rd.dev)
        for s in (step[0] & 1, (step[0] + 1) & 1):
            if launched[s]:
                with torch.cuda.stream(side):
                    side.wait_event(done[s])
                    read_back(s)
                launched[s] = False
        main.wait_stream(side)

    for _ in range(3):
        one()
    finish()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        one()
    finish()
    end.record(stream)
    end.synchronize()
    ms = start.elapsed_time(end)
    for r in rounds:
        r.close()
    return ms / steps, h2d, d2h


# ----------------------------------------------------------------------------- CPU oracle

def _blas_threads():
    """Threads of the BLAS that NumPy loaded, asked from the library itself where it
    exports a query (OpenBLAS builds do), else the environment's setting, else None."""
    import ctypes
    names = ["openblas_get_num_threads", "openblas_get_num_threads64_", "scipy_openblas_get_num_threads64_",
             "scipy_openblas_get_num_threads"]
    libs = set()
    try:
        with open("/proc/self/maps") as f:
            for ln in f:
                path = ln.split()[-1]
                base = os.path.basename(path).lower()
                if "blas" in base and ".so" in base:
                    libs.add(path)
    except OSError:
        pass
    libs = sorted(libs)
    for path in libs:
        if not os.path.exists(path):
            continue
        try:
            lib = ctypes.CDLL(path)
        except OSError:
            continue
        for n in names:
            fn = getattr(lib, n, None)
            if fn is not None:
                fn.restype = ctypes.c_int
                return int(fn())
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var):
            return int(os.environ[var])
    return None


class OracleSample:
    """A bounded sample of one verify round of a workload for the fp64 oracle (as it
    stands), and the per-stage times it gives, each scaled to the whole round by the
    stage's share of work that the sample covers:

      heads      medusa_heads on every frontier row with head 0 only and the first
                 `v_rows` rows of W2_0 and W_LM (W1_0 whole): scaled by the weight
                 elements of the round over those of the sample;
      fill       every sequence, whole;
      attention  tree_attention of every sequence for the query heads of KV head 0:
                 scaled by the number of KV heads;
      accept     every sequence, whole (unplanted N(0, 1) target logits);
      compact    every sequence, whole, on the KV head 0 cache.

    The inputs come from the workload's own seeded generators on the host (the leading
    rows of a seeded draw are the rows of the full draw), converted to float64 before
    the clock starts."""

    def __init__(self, w: synth.Workload, v_rows: int):
        from oracle import round as oround
        self.w = w
        acc = synth.rank_accuracy(w.n_heads, 10)
        self.t = oround.template_for(w.template, w.topk, w.n_heads, acc)
        N = self.N = self.t.n_rows
        d, V, K = w.hidden, w.vocab, w.n_heads
        self.v_rows = vr = max(w.topk, min(V, v_rows))
        f64 = lambda x: x.detach().double().numpy()
        self.h = f64(synth.normal((w.batch, d), 1.0, w.seed, "h", "cpu", w.torch_dtype))
        self.w1 = f64(synth.normal((1, d, d), 0.02, w.seed, "w1", "cpu", w.torch_dtype))
        self.w2 = f64(synth.normal((vr, d), 1.0 / math.sqrt(d), w.seed, "w2", "cpu", w.torch_dtype, sub=0))[None]
        self.w_lm = f64(synth.normal((vr, d), 1.0 / math.sqrt(d), w.seed, "w_lm", "cpu", w.torch_dtype))
        self.head_scale = (K * d * d + (K + 1) * V * d) / float(d * d + 2 * vr * d)
        g = w.group
        q, k, v = synth.tree_qkv(w, N)
        self.q, self.k, self.v = f64(q[:, :, :g]), f64(k[:, :, :1]), f64(v[:, :, :1])
        self.lengths = synth.prefix_lengths(w)
        self.ck, self.cv = [], []
        for b, L in enumerate(self.lengths):
            L = int(L)
            cap = L + N + 1
            ck = np.zeros((1, cap, w.head_dim))
            cv = np.zeros_like(ck)
            ck[:, :L] = f64(synth.normal((1, L, w.head_dim), 1.0, w.seed, "cache_k", "cpu", w.torch_dtype, sub=b))
            cv[:, :L] = f64(synth.normal((1, L, w.head_dim), 1.0, w.seed, "cache_v", "cpu", w.torch_dtype, sub=b))
            self.ck.append(ck)
            self.cv.append(cv)
        self.logits = f64(synth.target_logits(w, N))
        self.attn_scale = float(w.n_kv_heads)

    def run(self):
        """Per-stage µs of one round (scaled), the oracle called as it stands."""
        from oracle import accept as oacc
        from oracle import attention as oatt
        from oracle import compact as ocomp
        from oracle import heads as oheads
        from oracle import round as oround
        w, t = self.w, self.t
        clock = time.perf_counter
        t0 = clock()
        root, pool, _ = oheads.medusa_heads(self.h, self.w1, self.w2, self.w_lm, w.topk)
        t1 = clock()
        pool_full = np.tile(pool, (1, w.n_heads, 1))          # the sample's pool stands in for every head
        tokens = [oround.tree_fill(t, root[b], pool_full[b], int(self.lengths[b])) for b in range(w.batch)]
        t2 = clock()
        for b in range(w.batch):
            oatt.tree_attention(self.q[b], self.k[b], self.v[b], self.ck[b], self.cv[b], int(self.lengths[b]),
                                t.depth, t.mask, w.rope_base)
        t3 = clock()
        res = [oacc.accept(self.logits[b], tokens[b][0], t.retrieve, w.accept[0], 1.0, w.epsilon, w.delta)
               for b in range(w.batch)]
        t4 = clock()
        for b in range(w.batch):
            ocomp.kv_compact(self.ck[b], self.cv[b], int(self.lengths[b]), res[b].out_rows)
        t5 = clock()
        us = lambda a, b_: 1e6 * (b_ - a)
        return {"heads": us(t0, t1) * self.head_scale, "fill": us(t1, t2), "attn": us(t2, t3) * self.attn_scale,
                "accept": us(t3, t4), "compact": us(t4, t5)}

    def describe(self):
        w = self.w
        return (f"{w.name}: heads on head 0 with W1_0 and the first {self.v_rows} of {w.vocab} rows of W2_0 and "
                f"W_LM (x{self.head_scale:.1f}), attention for KV head 0's {w.group} query heads of every sequence "
                f"(x{int(self.attn_scale)}), fill, acceptance and compaction whole; fp64 NumPy")


def oracle_stages(w: synth.Workload, v_rows: int, reps: int = 1):
    """Best of `reps` sampled oracle rounds: (per-stage µs, description)."""
    smp = OracleSample(w, v_rows)
    best = None
    for _ in range(reps):
        st = smp.run()
        if best is None or sum(st.values()) < sum(best.values()):
            best = st
    return best, smp.describe()


def cpu_baseline_of(w: synth.Workload, v_rows: int, one_thread: bool):
    """The sampled oracle round on all host cores, and (one_thread) again in a child
    process whose BLAS and torch use one thread (set before NumPy loads)."""
    stages, desc = oracle_stages(w, v_rows)
    out = {"value": sum(stages.values()), "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
           "sample": desc, "all_cores": {"us": sum(stages.values()), "stages_us": stages,
                                         "blas_threads": _blas_threads(), "torch_threads": torch.get_num_threads()},
           "cpu_count": os.cpu_count()}
    if one_thread:
        env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-sample", w.name,
                            "--oracle-v-rows", str(v_rows)], env=env, capture_output=True, text=True, timeout=900)
        if r.returncode == 0 and r.stdout.strip():
            one = json.loads(r.stdout.strip().splitlines()[-1])
            out["one_thread"] = {"us": sum(one["stages_us"].values()), "stages_us": one["stages_us"],
                                 "blas_threads": one["blas_threads"], "torch_threads": one["torch_threads"]}
        else:
            out["one_thread"] = {"error": (r.stderr or "no output").strip().splitlines()[-1:]}
    return out


def run_oracle_sample(args):
    """Child process of the one-thread baseline: prints the sampled stage times."""
    torch.set_num_threads(1)
    w = synth.WORKLOADS[args.oracle_sample]
    stages, desc = oracle_stages(w, args.oracle_v_rows)
    print(json.dumps({"stages_us": stages, "sample": desc, "blas_threads": _blas_threads(),
                      "torch_threads": torch.get_num_threads()}))


# rows of W2_0 / W_LM in the sampled heads stage: the benchmark's CPU baseline, and the
# smaller per-step sample of the reference arm (which repeats it warmup + steps times)
BASELINE_V_ROWS = 8192
REFERENCE_V_ROWS = 4096


def run_reference(args):
    ws, rank, _ = dist_setup("gloo")
    if rank != 0:
        return
    w = synth.WORKLOADS[args.workload]
    smp = OracleSample(w, REFERENCE_V_ROWS)
    rounds = []
    for i in range(args.warmup + args.steps):
        st = smp.run()
        if i >= args.warmup:
            rounds.append(st)
    us = sum(sum(st.values()) for st in rounds) / len(rounds)
    stages = {k: sum(st[k] for st in rounds) / len(rounds) for k in rounds[0]}
    line = {
        "impl": "reference", "metric": METRIC, "value": us, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": us / 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, None),
        "cpu_baseline": {"kind": "oracle", "value": us, "unit": UNIT, "cores": os.cpu_count(),
                         "blas_threads": _blas_threads(), "torch_threads": torch.get_num_threads(),
                         "sample": "each step: " + smp.describe(), "stages_us": stages},
        "e2e": {"value": us, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def config_of(w: synth.Workload, rd):
    c = {"workload": w.name, "batch": w.batch, "template": list(map(str, w.template)),
         "q_heads": w.n_q_heads, "kv_heads": w.n_kv_heads, "head_dim": w.head_dim,
         "prefix_len": w.prefix_len if w.prefix_len else f"U{list(w.prefix_range)}",
         "medusa_heads": w.n_heads, "hidden": w.hidden, "vocab": w.vocab, "accept": w.accept[0],
         "paged": bool(w.page_size), "tree_rows": tree_rows(w),
         "l2": "inputs larger than L2: each step streams the head weights (>= 1.4 GB) before the KV; "
               "stage timings flush L2 with a 512 MB write",
         "launch": "each step is one medusa_round_launch (the library's CUDA graph of the five calls); "
                   "e2e alternates two such rounds bound to two input sets, each step's inputs copied from "
                   "pinned host memory during the previous step's round and its published tokens and L_out "
                   "copied back",
         "kv_cache": "bf16, with the library's fp16 mirror (filled once before timing, as after a prefill; "
                     "every round's cache writes keep it in step)" if w.dtype == "bf16" else w.dtype}
    return c


def tree_rows(w: synth.Workload) -> int:
    """Rows of the workload's template (root included): the regular tree's sum of
    products of widths plus the root, or the greedy budget plus the root."""
    if w.template[0] == "regular":
        n, prod = 1, 1
        for s in w.template[1]:
            prod *= s
            n += prod
        return n
    return 1 + w.template[1]


# ----------------------------------------------------------------------------- measurement

def measure(m, w: synth.Workload, dev, steps: int, warmup: int, flush, ws: int, local: int, rank: int,
            extras: bool):
    """One workload: the timed round-graph steps (clocks sampled meanwhile), then the
    per-stage split, the heads launch, the end-to-end loop and (extras) the variants."""
    hbm, bf16, src = peaks()
    rd = Round(m, w, dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(warmup):
        rd.step()
    graphs = RoundGraphs(rd, dev)
    for _ in range(warmup):
        graphs.step()
    torch.cuda.synchronize(dev)
    barrier(ws)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        ms = time_loop(graphs.step, steps, stream)
        torch.cuda.synchronize(dev)
    barrier(ws)
    ms_step = max_over_ranks(ms / steps, ws, dev)
    us_round = 1e3 * ms_step / ws                      # whole job: ws rounds per step

    stages = graphs.stage_times(20, stream, flush)
    attn_us = stages["attn"]
    round_b = rd.round_bytes(graphs.native.accept_len)
    round_gbs = round_b / (ms_step * 1e-3) / 1e9      # one round per GPU per step
    attn_gbs = rd.attn_bytes() / (attn_us * 1e-6) / 1e9
    attn_tf = rd.attn_flops() / (attn_us * 1e-6) / 1e12
    # the dominant kernel: heads launches back to back (the head weights exceed L2, so
    # every launch streams them from HBM), events on the replay stream
    heads_us = 1e3 * time_loop(graphs.stage["heads"].replay, 20, stream) / 20
    heads_gbs = rd.head_bytes() / (heads_us * 1e-6) / 1e9
    e2e_ms, h2d, d2h = e2e_loop(rd, max(10, steps // 4), stream)
    e2e_ms = max_over_ranks(e2e_ms, ws, dev)
    tensor_bound = w.name in ATTN_TENSOR_BOUND
    res = {
        "value": us_round, "ms_per_step": ms_step, "nodes_per_s": ws * w.batch * rd.N / (ms_step * 1e-3),
        "stages_us": stages,
        "roofline": {"kernel": "medusa_heads_topk (head-weight stream with top-k)",
                     "bound": "hbm", "achieved": heads_gbs, "peak": hbm, "unit": "GB/s",
                     "frac": heads_gbs / hbm, "traffic": HEADS_TRAFFIC.get(w.name), "peak_source": src,
                     "algorithmic_bytes": rd.head_bytes(), "launch_us": heads_us},
        "tree_attn": {"us": attn_us, "hbm_gbs": attn_gbs, "frac_of_hbm_peak": attn_gbs / hbm, "tflops": attn_tf,
                      "frac_of_tensor_peak": attn_tf / bf16},
        "tree_attn_roofline": ({"kernel": "medusa_tree_attn_verify", "bound": "tensor", "achieved": attn_tf,
                                "peak": bf16, "unit": "TFLOP/s", "frac": attn_tf / bf16,
                                "algorithmic_flops": rd.attn_flops(), "peak_source": src,
                                "note": "fp16 operands: the fp16 dense rate equals the bf16 one"}
                               if tensor_bound else
                               {"kernel": "medusa_tree_attn_verify", "bound": "hbm", "achieved": attn_gbs,
                                "peak": hbm, "unit": "GB/s", "frac": attn_gbs / hbm,
                                "traffic": ATTN_TRAFFIC.get(w.name), "peak_source": src,
                                "algorithmic_bytes": rd.attn_bytes()}),
        "round_roofline": {"bound": "hbm", "achieved": round_gbs, "peak": hbm, "unit": "GB/s",
                           "frac": round_gbs / hbm, "peak_source": src, "algorithmic_bytes": round_b,
                           "note": "all five steps' algorithmic bytes over one round's device time"},
        "e2e": {"value": 1e3 * e2e_ms / ws, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": rd.launches_per_step() * steps,
        "clocks": clk.summary(),
        "tree_rows": rd.N,
    }
    if extras and rank == 0:
        res["heads_all_rows"] = heads_all_rows(rd, stream, bf16)
        res["kv_compact_layers"] = compact_all_layers(rd, graphs.native, stream, flush)
        res["accept_hidden"] = accept_hidden(rd, graphs.native, stream, flush, hbm)
    del graphs, rd
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    return res


# workloads whose tree attention is bound by the tensor cores (wide trees: arithmetic
# intensity above the ridge) rather than by the prefix K/V stream
ATTN_TENSOR_BOUND = ("llama3-8b-256", "longctx-341")

HEADLINE = "longctx-341"


# ----------------------------------------------------------------------------- one stage alone

def run_stage(args):
    """One step of the round alone on the workload's inputs (only those inputs are
    built): `heads` (medusa_heads_topk on the frontier rows) or `attn`
    (medusa_tree_attn_verify).  Prints the mean device time of --steps calls after
    --warmup calls; for profiling a single kernel (ncu -k ... -s <warmup> -c 1)."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    from medusa_speculative_tree_gb300 import build
    build.build()
    import medusa_speculative_tree_gb300 as m
    w = synth.WORKLOADS[args.workload]
    if args.stage == "heads":
        h, w1, w2, w_lm = synth.head_weights(w, device=dev)
        call = lambda: m.medusa_heads_topk(h, w1, w2, w_lm, w.topk)
    else:
        acc = synth.rank_accuracy(w.n_heads, 10)
        if w.template[0] == "regular":
            paths = m.medusa_tree_regular(w.template[1])
        else:
            paths = m.medusa_tree_greedy(acc[:, :w.template[2]], w.template[1])
        tmpl = m.Template(paths, w.topk, w.n_heads, device=dev)
        N = tmpl.n_rows
        q, k, v = synth.tree_qkv(w, N, device=dev)
        lengths = synth.prefix_lengths(w)
        L = torch.tensor(lengths, dtype=torch.int32, device=dev)
        gen = torch.Generator(device=dev).manual_seed(w.seed)
        if w.page_size:
            lay = synth.paged_layout(w, lengths, N)
            K = torch.randn((lay.n_pages, w.n_kv_heads, 16, w.head_dim), generator=gen, device=dev).to(w.torch_dtype)
            cache_bt = torch.tensor(lay.block_table, dtype=torch.int32, device=dev)
        else:
            cap = int(lengths.max()) + N + 16
            K = torch.randn((w.batch, w.n_kv_heads, cap, w.head_dim), generator=gen, device=dev).to(w.torch_dtype)
            cache_bt = None
        V = torch.randn(K.shape, generator=gen, device=dev).to(w.torch_dtype)
        cache = m.KVCache(K, V, block_table=cache_bt)
        if w.dtype == "bf16":
            cache.add_mirror()                     # as in the round (Round)
        out = torch.empty((w.batch, N, w.n_q_heads, w.head_dim), dtype=torch.float32, device=dev)
        call = lambda: m.medusa_tree_attn_verify(tmpl, q, k, v, cache, L, int(lengths.max()), rope_base=w.rope_base,
                                                 out=out)
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize(dev)
    ms = time_loop(call, args.steps, torch.cuda.current_stream(dev))
    print(json.dumps({"stage": args.stage, "workload": w.name, "calls": args.steps, "us_per_call": 1e3 * ms / args.steps}))


# ----------------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=HEADLINE, choices=synth.WORKLOAD_ORDER)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-workload", action="store_true", help="measure the headline workload only")
    ap.add_argument("--stage", default="round", choices=["round", "heads", "attn"],
                    help="time one step alone (for single-kernel profiles) instead of the round")
    ap.add_argument("--oracle-sample", default=None, help=argparse.SUPPRESS)
    ap.add_argument("--oracle-v-rows", type=int, default=BASELINE_V_ROWS, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.oracle_sample:
        return run_oracle_sample(args)
    if args.stage != "round":
        return run_stage(args)
    args.warmup = max(args.warmup, 3)
    if args.impl == "reference":
        return run_reference(args)

    ws, rank, local = dist_setup("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from medusa_speculative_tree_gb300 import build
    build.build()
    import medusa_speculative_tree_gb300 as m

    w = synth.WORKLOADS[args.workload]
    flush_buf = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    flush = lambda: flush_buf.fill_(1.0)

    head = measure(m, w, dev, args.steps, args.warmup, flush, ws, local, rank, extras=True)
    per = {}
    if not args.no_per_workload:
        for name in synth.WORKLOAD_ORDER:
            if name == w.name:
                continue
            r = measure(m, synth.WORKLOADS[name], dev, max(args.steps, 20), args.warmup, flush, ws, local, rank,
                        extras=True)
            per[name] = r

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_of(w, BASELINE_V_ROWS, one_thread=True)
        for name, r in per.items():
            st, desc = oracle_stages(synth.WORKLOADS[name], BASELINE_V_ROWS)
            r["cpu_baseline"] = {"value": sum(st.values()), "unit": UNIT, "cores": os.cpu_count(),
                                 "kind": "oracle", "sample": desc, "stages_us": st}

    if rank == 0:
        line = {
            "metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
            "data": "synthetic (seeded generators, random-init weights)",
            "config": config_of(w, None),
            "nodes_per_s": head["nodes_per_s"],
            "tree_attn": head["tree_attn"],
            "stages_us": head["stages_us"],
            "roofline": head["roofline"],
            "heads_all_rows": head.get("heads_all_rows"),
            "kv_compact_layers": head.get("kv_compact_layers"),
            "accept_hidden": head.get("accept_hidden"),
            "round_roofline": head["round_roofline"],
            "tree_attn_roofline": head["tree_attn_roofline"],
            "cpu_baseline": cpu,
            "e2e": head["e2e"],
            "gpu_launches": head["gpu_launches"],
            "clocks": head["clocks"],
            "per_workload": per,
        }
        print(json.dumps(line))
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
