"""Plain fp64 CPU oracle of one Medusa verify round.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import or call anything here.  The CUDA
library never imports it, links it or falls back to it, and it shares no code
with the CUDA library (the seeded input generators in ``synth`` are the only
common module, and they hold none of the method's arithmetic).

Every function is the plain definition of what the pages compute, written for
a reader to check by eye: dense masks, literal prefix tests, full softmaxes in
float64, explicit loops over paths.  Nothing is blocked, fused or reordered.

Pages cited (by title and section):
  [M7.2]   "M7.2 - Medusa: Multi-Head Candidates, Tree Attention, and Verification"
  [CN]     "Medusa 完全拆解：多头树式候选如何用一次验证解码多个 Token"
  [PartII] "Medusa Part II: Candidate Trees, Verification, and Acceptance"
  [Math]   "Medusa — Multi-Head Speculative Decoding Math"

Pinning status (what each function is checked against, in tests/):
  tree.compile_template     worked examples of [M7.2] §0x01A/§0x03F/§0x04A and [CN]
                            "手算一棵两层候选树"; closed-form node counts; mask axioms
  tree.greedy_tree          [PartII] Part 3 toy order; brute-force global sort
  tree.regular_paths        closed form sum_k prod_i s_i ([M7.2] §0x02B, [CN])
  heads.medusa_heads        special case K=1, W1=0 reduces to the LM-head GEMV;
                            SiLU closed form; brute-force top-k on tiny inputs
  attention.tree_attention  brute force: each node equals causal attention over its
                            own root-to-node path; chain tree = causal decode;
                            N=1 = single-query attention; RoPE relative-phase identity
  accept.accept             [M7.2] §0x04G / §0x06B traces; [PartII] Part 7 cumprod
                            example; closed-form entropy of the Part 8 distribution
  accept.row_stats          exact entropy: uniform, one-hot, two-point closed forms;
                            guarded entropy ([M7.2] §0x04E): the same three cases worked
                            by hand, and an edge whose typical decision the guard flips
  accept.log_prob           temperature 2 against a hand-computed softmax
  accept.target_logits      identity and orthonormal projections (closed forms)
  compact.kv_compact        [M7.2] §0x06B trace; overlap case against a snapshot-free copy
  cost                      [M7.2] §0x02E / §0x06 printed parameter and byte counts
  round.tree_fill           [M7.2] §0x04A slot formula worked by hand (widths (2, 2))
  round.run_sequence        a round worked by hand: W1 = 0 heads read by inspection,
                            keys (1, 0) rotated to angle L + depth, planted greedy
                            argmaxes, committed rows and length ([M7.2] §0x06B)
"""
