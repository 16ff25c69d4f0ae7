"""Benchmark of one Medusa verify round on GB300.

A step is one whole round of the hot path on one batch of synthetic input:
medusa_heads_topk -> medusa_tree_fill -> medusa_tree_attn_verify ->
medusa_tree_accept -> medusa_kv_compact.  The default workload is the
Vicuna-7B-shaped round (bf16, batch 1, 64-row greedy tree, L = 2048, K = 4
heads over d = 4096 and V = 32000).

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
    """Device-resident inputs and outputs of one verify round for a workload."""

    def __init__(self, m, w: synth.Workload, dev):
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
            heads = 2 * math.ceil(T / 128) + 1         # per pass of <= 128 rows: input pairs and
                                                        # tensor-core stream; then top-k
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
HEADS_TRAFFIC = {"vicuna7b-64": 1_445_265_000 + 4_523_008}
# the same for the attention launch (dram__bytes_read.sum + dram__bytes_write.sum)
ATTN_TRAFFIC = {"vicuna7b-64": 35_210_752 + 0}


def heads_all_rows(rd, stream, peak_tflops):
    """medusa_heads_topk with every tree row as a hidden row (T = B N), the variant in which
    the heads are a tensor-core contraction.  bf16 with T >= 2 runs on the tensor cores
    with each input row as a bf16 pair (hi, lo), so the MMAs execute twice the useful
    2 T flops per weight element; both rates are reported."""
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
    pairs = 2 if (w.dtype == "bf16" and T >= 2) else 1
    passes = math.ceil(T / 128) if pairs == 2 else 1
    return {"T": T, "us": us, "useful_tflops": useful, "tensor_tflops": useful * pairs,
            "peak_tflops": peak_tflops, "frac": useful * pairs / peak_tflops, "weight_passes": passes,
            "hbm_gbs": passes * rd.head_bytes() / (us * 1e-6) / 1e9}


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

    def __init__(self, rd: Round, dev):
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
                                       epsilon=w.epsilon, delta=w.delta)
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
    memory and the published result read back (both inside the timed region).  The
    frontier rows and lengths are copied first, on the round's stream (the heads and
    the fill read them); the attention and acceptance inputs follow on a second stream,
    after the previous step's reads of those buffers, and overlap the heads; the round
    waits for them before the attention call."""
    w = rd.w
    h_host = rd.h.cpu().pin_memory()
    q_host, k_host, v_host = (x.cpu().pin_memory() for x in (rd.q, rd.k, rd.v))
    lg_host = rd.logits.cpu().pin_memory()
    L_host = rd.L.cpu().pin_memory()
    res_host = torch.empty((w.batch, rd.tmpl.max_depth + 2), dtype=torch.int32).pin_memory()
    h_d, q_d, k_d, v_d, lg_d, L_d = (torch.empty_like(x, device=rd.dev) for x in
                                     (h_host, q_host, k_host, v_host, lg_host, L_host))
    h2d = sum(x.numel() * x.element_size() for x in (h_host, q_host, k_host, v_host, lg_host, L_host))
    d2h = res_host.numel() * res_host.element_size()
    m = rd.m

    side = torch.cuda.Stream(rd.dev)
    ready = torch.cuda.Event()

    def one():
        main = torch.cuda.current_stream(rd.dev)
        for dst, src in ((h_d, h_host), (L_d, L_host)):
            dst.copy_(src, non_blocking=True)
        side.wait_stream(main)                       # the previous step has read q, k, v, logits
        with torch.cuda.stream(side):
            for dst, src in ((q_d, q_host), (k_d, k_host), (v_d, v_host), (lg_d, lg_host)):
                dst.copy_(src, non_blocking=True)
            ready.record(side)
        root, pool = m.medusa_heads_topk(h_d, rd.w1, rd.w2, rd.w_lm, w.topk)
        tokens, _ = m.medusa_tree_fill(rd.tmpl, root, pool, L_d)
        main.wait_event(ready)
        m.medusa_tree_attn_verify(rd.tmpl, q_d, k_d, v_d, rd.cache, L_d, rd.max_L, rope_base=w.rope_base,
                                  out=rd.out, ws=rd.attn_ws)
        r = m.medusa_tree_accept(rd.tmpl, lg_d, tokens, rd.mode, epsilon=w.epsilon, delta=w.delta)
        L_out, _ = m.medusa_kv_compact(rd.cache, rd.tmpl, L_d, r["accept_len"], r["out_rows"])
        res = torch.cat([r["out_tokens"], L_out[:, None]], dim=1)
        res_host.copy_(res, non_blocking=True)

    for _ in range(3):
        one()
    torch.cuda.synchronize()
    ms = time_loop(one, steps, stream)
    return ms / steps, h2d, d2h


# ----------------------------------------------------------------------------- CPU oracle

def oracle_round_seconds(w: synth.Workload, reps: int = 1):
    """Time the fp64 oracle (as it stands) on a full round of the workload, host only.
    Returns (seconds per round, threads, description)."""
    from oracle import round as oround
    acc = synth.rank_accuracy(w.n_heads, 10)
    t_o = oround.template_for(w.template, w.topk, w.n_heads, acc)
    N = t_o.n_rows
    h, w1, w2, w_lm = synth.head_weights(w)
    q, k, v = synth.tree_qkv(w, N)
    lengths = synth.prefix_lengths(w)
    ks, vs = synth.prefix_kv(w, lengths)
    logits = synth.target_logits(w, N)
    f64 = lambda t: t.detach().double().numpy()
    times = []
    for _ in range(reps):
        t0 = time.perf_counter()
        for b in range(w.batch):
            L = int(lengths[b])
            cap = L + N + 1
            ck = np.zeros((w.n_kv_heads, cap, w.head_dim))
            cv = np.zeros_like(ck)
            ck[:, :L], cv[:, :L] = f64(ks[b]), f64(vs[b])
            oround.run_sequence(t_o, f64(h[b]), f64(w1), f64(w2), f64(w_lm), f64(q[b]), f64(k[b]), f64(v[b]),
                                ck, cv, L, f64(logits[b]), w.accept[0], w.rope_base, epsilon=w.epsilon,
                                delta=w.delta)
        times.append(time.perf_counter() - t0)
    return min(times), torch.get_num_threads(), f"{reps} full oracle round(s) of {w.name}, best taken"


def run_reference(args):
    ws, rank, _ = dist_setup("gloo")
    if rank != 0:
        return
    w = synth.WORKLOADS[args.workload]
    secs = []
    for i in range(args.warmup + args.steps):
        s, cores, _ = oracle_round_seconds(w, 1)
        if i >= args.warmup:
            secs.append(s)
    us = 1e6 * sum(secs) / len(secs)
    line = {
        "impl": "reference", "metric": METRIC, "value": us, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": us / 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, None),
        "cpu_baseline": {"kind": "oracle", "value": us, "unit": UNIT, "cores": cores,
                         "sample": f"one full fp64 oracle round of {w.name} per step"},
        "e2e": {"value": us, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def config_of(w: synth.Workload, rd):
    c = {"workload": w.name, "batch": w.batch, "template": list(map(str, w.template)),
         "q_heads": w.n_q_heads, "kv_heads": w.n_kv_heads, "head_dim": w.head_dim,
         "prefix_len": w.prefix_len if w.prefix_len else f"U{list(w.prefix_range)}",
         "medusa_heads": w.n_heads, "hidden": w.hidden, "vocab": w.vocab, "accept": w.accept[0],
         "paged": bool(w.page_size),
         "l2": "inputs larger than L2: each step streams the head weights (>= 1.4 GB) before the KV; "
               "stage timings flush L2 with a 512 MB write",
         "launch": "each step is one medusa_round_launch (the library's CUDA graph of the five calls); "
                   "e2e calls the five API functions eagerly"}
    if rd is not None:
        c["tree_rows"] = rd.N
    return c


# ----------------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="vicuna7b-64", choices=synth.WORKLOAD_ORDER)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
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
    rd = Round(m, w, dev)
    stream = torch.cuda.current_stream(dev)
    flush_buf = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    flush = lambda: flush_buf.fill_(1.0)

    for _ in range(args.warmup):
        rd.step()
    graphs = RoundGraphs(rd, dev)
    for _ in range(args.warmup):
        graphs.step()
    torch.cuda.synchronize(dev)
    barrier(ws)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        ms = time_loop(graphs.step, args.steps, stream)
        torch.cuda.synchronize(dev)
    barrier(ws)
    ms_step = max_over_ranks(ms / args.steps, ws, dev)
    us_round = 1e3 * ms_step / ws                      # whole job: ws rounds per step

    stages = graphs.stage_times(20, stream, flush)
    hbm, bf16, src = peaks()
    attn_us = stages["attn"]
    round_b = rd.round_bytes(graphs.native.accept_len)
    round_gbs = round_b / (ms_step * 1e-3) / 1e9      # one round per GPU per step
    attn_gbs = rd.attn_bytes() / (attn_us * 1e-6) / 1e9
    # the dominant kernel: heads launches back to back (the head weights exceed L2, so
    # every launch streams them from HBM), events on the replay stream
    heads_us = 1e3 * time_loop(graphs.stage["heads"].replay, 20, stream) / 20
    heads_gbs = rd.head_bytes() / (heads_us * 1e-6) / 1e9
    e2e_ms, h2d, d2h = e2e_loop(rd, max(10, args.steps // 4), stream)
    e2e_ms = max_over_ranks(e2e_ms, ws, dev)
    all_rows = heads_all_rows(rd, stream, bf16) if rank == 0 else None
    layers = compact_all_layers(rd, graphs.native, stream, flush) if rank == 0 else None
    acc_h = accept_hidden(rd, graphs.native, stream, flush, hbm) if rank == 0 else None

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        s, cores, desc = oracle_round_seconds(w, 1)
        cpu = {"value": 1e6 * s, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc}

    if rank == 0:
        line = {
            "metric": METRIC, "value": us_round, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": w.dtype, "data": "synthetic (seeded generators, random-init weights)",
            "config": config_of(w, rd),
            "nodes_per_s": ws * w.batch * rd.N / (ms_step * 1e-3),
            "tree_attn": {"us": attn_us, "hbm_gbs": attn_gbs, "frac_of_hbm_peak": attn_gbs / hbm,
                          "tflops": rd.attn_flops() / (attn_us * 1e-6) / 1e12},
            "stages_us": stages,
            "roofline": {"kernel": "medusa_heads_topk (head-weight stream with top-k)",
                         "bound": "hbm", "achieved": heads_gbs, "peak": hbm, "unit": "GB/s",
                         "frac": heads_gbs / hbm, "traffic": HEADS_TRAFFIC.get(w.name), "peak_source": src,
                         "algorithmic_bytes": rd.head_bytes(), "launch_us": heads_us},
            "heads_all_rows": all_rows,
            "kv_compact_layers": layers,
            "accept_hidden": acc_h,
            "round_roofline": {"bound": "hbm", "achieved": round_gbs, "peak": hbm, "unit": "GB/s",
                               "frac": round_gbs / hbm, "peak_source": src, "algorithmic_bytes": round_b,
                               "note": "all five steps' algorithmic bytes over one round's device time"},
            "tree_attn_roofline": {"kernel": "medusa_tree_attn_verify", "bound": "hbm", "achieved": attn_gbs,
                                   "peak": hbm, "unit": "GB/s", "frac": attn_gbs / hbm,
                                   "traffic": ATTN_TRAFFIC.get(w.name),
                                   "peak_source": src, "algorithmic_bytes": rd.attn_bytes()},
            "cpu_baseline": cpu,
            "e2e": {"value": 1e3 * e2e_ms / ws, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": rd.launches_per_step() * args.steps,
            "clocks": clk.summary(),
        }
        print(json.dumps(line))
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
