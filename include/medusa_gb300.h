/*
 * medusa_gb300.h - C ABI of libmedusa_gb300.so: one Medusa verify round on one GPU.
 *
 * A round has five device calls, issued in this order on one stream:
 *   medusa_heads_topk -> medusa_tree_fill -> medusa_tree_attn_verify
 *   -> medusa_tree_accept -> medusa_kv_compact
 * plus host-side template construction (medusa_tree_regular, medusa_tree_greedy,
 * medusa_tree_compile, medusa_tree_upload).
 *
 * Pages that define the operations (cited by title and section):
 *   [M7.2]   "M7.2 - Medusa: Multi-Head Candidates, Tree Attention, and Verification"
 *   [CN]     "Medusa 完全拆解：多头树式候选如何用一次验证解码多个 Token"
 *   [PartII] "Medusa Part II: Candidate Trees, Verification, and Acceptance"
 *   [Math]   "Medusa — Multi-Head Speculative Decoding Math"
 *
 * Conventions shared by every call
 *   - Pointers are device memory unless the comment says [host].  All device
 *     buffers are owned by the caller; no call allocates or frees memory, except
 *     that medusa_round_create allocates its CUDA graph objects (no device buffers)
 *     and medusa_round_destroy frees them.
 *   - Arrays are row-major with the last dimension contiguous.  Float tensors
 *     read with 128-bit loads must be 16-byte aligned (the base pointer and
 *     every row); medusa_tree_attn_verify's bf16 path also needs the KV cache
 *     base 16-byte aligned for its TMA descriptors.
 *   - Token ids, row indices and lengths are int32.  Per-sequence lengths live
 *     in device memory, so a round needs no host synchronisation.
 *   - Device calls are asynchronous on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream).  They return MEDUSA_OK after enqueueing, or a
 *     negative status with nothing enqueued when an argument that the host can
 *     see is invalid.  Conditions only the device can see (a prefix length past
 *     the cache capacity, a corrupt accepted path) are reported per sequence in
 *     `status[b]`, and that sequence is left unmodified.
 *   - No kernel waits on another kernel launch.  Inside one launch, waits are
 *     bounded: the persistent heads kernels (one CTA per SM, cooperative launch,
 *     so every CTA is resident) wait on counters that other CTAs of the same
 *     launch advance, and the pipelined kernels wait on their own mbarriers; a
 *     wait that exceeds about two seconds gives up and the call reports an error
 *     (MEDUSA_ETIMEOUT per sequence, or -1 ids from the heads).  Split-KV
 *     attention merges its splits inside a thread-block cluster (bf16 tensor-core
 *     path) or in the last CTA to finish a unit (an atomic ticket, fp32 path).
 *   - medusa_round_create captures the five device calls of one round into a
 *     CUDA graph; medusa_round_launch replays it with one launch and no host
 *     synchronisation.
 */
#ifndef MEDUSA_GB300_H
#define MEDUSA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t medusa_status;
#define MEDUSA_OK            0
#define MEDUSA_EINVAL       -1   /* bad pointer, size or enum */
#define MEDUSA_ECAPACITY    -2   /* cache too small for L + N rows */
#define MEDUSA_EUNSUPPORTED -3   /* shape outside what the kernels implement */
#define MEDUSA_ETEMPLATE    -4   /* rank paths not prefix-closed, duplicated or out of range */
#define MEDUSA_ECUDA        -5   /* a CUDA runtime call failed */
#define MEDUSA_EWORKSPACE   -6   /* workspace or output buffer too small */
#define MEDUSA_EPATH        -7   /* per-sequence: accepted path is not a valid tree chain */
#define MEDUSA_ETIMEOUT     -8   /* per-sequence: a bounded device wait gave up; the sequence's
                                    outputs are invalid and the workspace must be re-zeroed */
#define MEDUSA_ERANGE       -9   /* per-sequence: an output that is not finite, from an input
                                    outside the range of the kernel's arithmetic (bf16 attention:
                                    fp16 operands, |x| > 65504); the outputs are invalid */

typedef int32_t medusa_dtype;
#define MEDUSA_F32  0
#define MEDUSA_BF16 1

#define MEDUSA_ACCEPT_GREEDY  0
#define MEDUSA_ACCEPT_TYPICAL 1

/* Largest supported sizes. */
#define MEDUSA_MAX_ROWS   4096   /* packed tree rows N, root included */
#define MEDUSA_MAX_DEPTH  16     /* Medusa depth D (paths hold D + 1 rows) */
#define MEDUSA_MAX_TOPK   32     /* candidate pool width TOPK */
#define MEDUSA_MAX_HEAD_ROWS 1024 /* hidden rows T of one medusa_heads_topk call */
#define MEDUSA_MAX_LAYERS 4096   /* layers of one medusa_kv_compact_layers call */

/*
 * Compiled tree template: the four coupled buffers of [M7.2] §0x04A plus the
 * structure derived from them.  Rows are numbered canonically: row 0 is the
 * LM-head root (empty path); non-root rank paths are sorted by (length, path)
 * and row(path) = 1 + index ([M7.2] §0x04A "Canonical row map").
 *
 * The struct is a host value whose array pointers point either into a host
 * buffer (after medusa_tree_compile) or into a device buffer (after
 * medusa_tree_upload).  Device calls take the device form.
 *
 * Per-sequence templates ([M7.2] §0x07D: sequences of a batch may verify different
 * trees; [CN] "局限与适用场景": the best node count moves with the context length): when per_seq
 * is not NULL it points to a device array of B device-form templates, one per
 * sequence (each with per_seq NULL and the batch's topk), and the counts of this
 * struct are bounds over them (n_rows, n_words, max_depth, n_paths and n_internal at
 * least those of every sequence; topk equal); its arrays are not read.  Per-row
 * tensors of the device calls are then laid out with the bound: tokens, pos [B][n_rows],
 * q [B][n_rows][H][dh], logits [B][n_rows][V], out_rows [B][max_depth + 1]; rows past a
 * sequence's own n_rows are not read as tree rows (tokens and pos get -1 there, the
 * attention output is not written there).  medusa_tree_batch builds such a struct;
 * medusa_tree_greedy_device builds a tree per sequence on the GPU.
 */
typedef struct medusa_tree_s {
  int32_t n_rows;       /* N = 1 + number of rank paths */
  int32_t n_words;      /* ceil(N / 64): 64-bit words per ancestor mask row */
  int32_t max_depth;    /* D = longest path */
  int32_t n_paths;      /* maximal root-to-node paths (retrieval rows) */
  int32_t topk;         /* TOPK of the slot formula */
  int32_t n_internal;   /* rows with at least one child */
  const int32_t *slot;           /* [N] tree_indices: 0 for the root, 1 + (t-1)*TOPK + r_t ([M7.2] §0x01B) */
  const int32_t *depth;          /* [N] path length; position = L + depth ([M7.2] §0x03C) */
  const int32_t *parent;         /* [N] parent row, -1 for the root */
  const int32_t *retrieve;       /* [n_paths][D+1] row chains from the root, -1 padded ([M7.2] §0x04A) */
  const int32_t *internal;       /* [n_internal] rows with children, ascending */
  const int32_t *internal_index; /* [N] position of a row in `internal`, -1 for leaves */
  const uint64_t *anc;           /* [N][n_words] bit (v % 64) of word v / 64 set iff path(v) is a prefix of path(u) ([M7.2] §0x04A) */
  const struct medusa_tree_s *per_seq; /* NULL, or [B] device templates, one per sequence (see above) */
} medusa_tree_t;

/* One layer's KV cache, contiguous or paged.
 *
 * A bf16 cache may carry an fp16 mirror: k_f16 and v_f16, buffers of the same layout
 * and size as k and v (caller-owned, device, 16-byte aligned), holding every cache
 * element converted to fp16 (exact for magnitudes in [2^-14, 65504]; smaller ones lose
 * bits, larger ones become inf).  The tensor-core attention multiplies in fp16: with a
 * mirror it reads the prefix tiles from it and converts nothing, instead of converting
 * every prefix row of K and V on every call.  Every call that writes cache rows (the
 * tree rows staged by medusa_tree_attn_verify, the rows moved by the compaction calls
 * and by medusa_tree_accept_commit) writes both copies, so a mirror once filled
 * (medusa_kv_mirror_sync) stays a copy of the cache.  Both NULL: no mirror. */
typedef struct {
  void *k;                /* contiguous: [B][n_kv_heads][capacity][head_dim];
                             paged:      [n_pages][n_kv_heads][page_size][head_dim] */
  void *v;                /* same layout as k */
  medusa_dtype dtype;     /* MEDUSA_F32 or MEDUSA_BF16 */
  int32_t n_kv_heads;
  int32_t head_dim;       /* 64 or 128 */
  int32_t capacity;       /* rows addressable per sequence (paged: max_blocks * page_size) */
  int32_t page_size;      /* 0 = contiguous; otherwise 16 */
  const int32_t *block_table; /* paged: [B][max_blocks] physical page of rows [16j, 16j+16) */
  int32_t max_blocks;
  int32_t n_pages;
  void *k_f16;            /* NULL, or (bf16 caches) the fp16 mirror of k, same layout */
  void *v_f16;            /* NULL, or the fp16 mirror of v; set both or neither */
} medusa_kv_t;

/* ---------------------------------------------------------------------------
 * Host-side template construction (no GPU needed)
 * ------------------------------------------------------------------------- */

/* All rank paths of a regular Cartesian tree with widths s_1..s_K, in canonical
 * order ([M7.2] §0x02B; [CN] "多个 Medusa Head 如何产生候选树"; [Math] "From heads
 * to a candidate tree").  paths_out [host] [max_paths][K], -1 padded.  *n_out gets
 * sum_k prod_{i<=k} s_i.  MEDUSA_EWORKSPACE if max_paths is too small.  With
 * paths_out NULL and max_paths 0 the call is a size query: it sets *n_out only. */
medusa_status medusa_tree_regular(const int32_t *widths /*[host] K*/, int32_t K,
                                  int32_t *paths_out, int32_t max_paths, int32_t *n_out);

/* Greedy frontier search of [M7.2] §0x04C / [PartII] Part 3: starting from the
 * root, repeatedly admit the frontier path of largest weight
 * w(r_1..r_t) = prod_j acc[j][r_j] (computed left to right in double), then open
 * its children, until `budget` paths are chosen.  Weights within 1e-12 relative
 * tie; ties go to the shorter path, then the lexicographically smaller one.
 * acc [host] [K][R] exact-rank accuracies in [0, 1].  paths_out [host] [budget][K],
 * -1 padded, in admission order.  *n_out = paths chosen (< budget only when every
 * path of depth <= K is taken). */
medusa_status medusa_tree_greedy(const double *acc, int32_t K, int32_t R, int32_t budget,
                                 int32_t *paths_out, int32_t *n_out);

/* Greedy trees built on the GPU, one per sequence, from per-sequence rank
 * accuracies ([M7.2] §0x04C; [PartII] Part 3; [CN]: the best tree moves with the
 * context): the search of medusa_tree_greedy (same weights, same tie rule, so the same
 * paths) followed by the compilation of medusa_tree_compile (same arrays, same canonical
 * order), in one kernel with one CTA per sequence, with no host round trip.
 *   acc [B][K][R] device doubles in [0, 1] (a sequence with a value outside gets the
 *   root-only template and status MEDUSA_EINVAL); ranks r < R <= topk; budget >= 0
 *   non-root paths per sequence, R * (budget + 1) <= 6144;
 *   dev_buf: medusa_tree_greedy_device_bytes(B, K, R, budget) bytes (16-byte aligned)
 *   that receive the B template arrays; per_seq [B] device medusa_tree_t (8-byte
 *   aligned), written by the kernel; status [B] device or NULL (0, or MEDUSA_EINVAL);
 *   batch_out [host]: the per-sequence batch to pass to the device calls (counts are
 *   the bounds budget + 1 rows, depth min(K, budget); per_seq set).
 * Returns after enqueueing; MEDUSA_EUNSUPPORTED when R * (budget + 1) > 6144. */
size_t medusa_tree_greedy_device_bytes(int32_t B, int32_t K, int32_t R, int32_t budget);
medusa_status medusa_tree_greedy_device(const double *acc, int32_t B, int32_t K, int32_t R, int32_t budget,
                                        int32_t topk, void *dev_buf, size_t dev_bytes, medusa_tree_t *per_seq,
                                        int32_t *status, medusa_tree_t *batch_out, void *stream);

/* Bytes of the template blob for up to n_paths rank paths of length <= max_len. */
size_t medusa_tree_bytes(int32_t n_paths, int32_t max_len);

/* Compile rank paths into a template ([M7.2] §0x04A).  paths [host]
 * [n_paths][max_len], -1 padded, any order.  Rejects (MEDUSA_ETEMPLATE) duplicate
 * paths, empty paths, ranks outside [0, topk), paths longer than n_heads and
 * families that are not prefix-closed.  The arrays are written into host_buf
 * [host, host_bytes >= medusa_tree_bytes(...), 8-byte aligned]; *out points into it. */
medusa_status medusa_tree_compile(const int32_t *paths, int32_t n_paths, int32_t max_len,
                                  int32_t topk, int32_t n_heads, void *host_buf,
                                  size_t host_bytes, medusa_tree_t *out);

/* Copy a compiled template blob to device memory (one cudaMemcpyAsync on
 * `stream`; host_buf must stay alive until the copy completes) and fill *dev
 * with pointers into dev_buf.  dev_buf 16-byte aligned, dev_bytes >= the blob. */
medusa_status medusa_tree_upload(const medusa_tree_t *host_tree, const void *host_buf,
                                 void *dev_buf, size_t dev_bytes, medusa_tree_t *dev,
                                 void *stream);

/* A per-sequence batch of device templates (see medusa_tree_t): copies the B
 * descriptors seq [host] [B] (device form, per_seq NULL, equal topk) into dev_descs
 * (device, B * sizeof(medusa_tree_t) bytes, 8-byte aligned; one cudaMemcpyAsync on
 * `stream`, seq must stay alive until it completes) and fills *out with the bounds of
 * their counts and out->per_seq = dev_descs.  The same device template may serve
 * several sequences.  MEDUSA_EINVAL on a mismatch of topk or a nested batch. */
medusa_status medusa_tree_batch(const medusa_tree_t *seq, int32_t B, void *dev_descs, size_t dev_bytes,
                                medusa_tree_t *out, void *stream);

/* ---------------------------------------------------------------------------
 * Round step 1: heads + top-k
 * ------------------------------------------------------------------------- */

size_t medusa_heads_topk_workspace(int32_t T, int32_t d, int32_t V, int32_t K, int32_t topk);

/* For each of T frontier rows h[t] ([CN] "Medusa 的核心思路与系统位置"; [Math]
 * "The Medusa head"; [M7.2] §0x02A with one residual block):
 *   root[t]        = argmax_v (W_LM h[t])_v                          ([M7.2] §0x04D)
 *   z_k            = h[t] + SiLU(W1_k h[t] + b1_k)
 *   pool[t][k][:]  = the topk ids of W2_k z_k, by value descending   ([PartII] Part 4)
 * Ties in value go to the lower token id.  Arithmetic: fp32 accumulation of
 * the dtype inputs; z_k is kept in fp32.
 *   h [T][d]; w1 [K][d][d]; b1 [K][d] or NULL; w2: head k's [V][d] matrix starts
 *   at w2 + k * w2_head_stride elements (stride 0 = one projection shared by all
 *   heads, [M7.2] §0x02D); w_lm [V][d].  All in dtype `dt`.
 *   root [T]; pool [T][K][topk]; logits_out [T][K+1][V] fp32 or NULL (slot 0 =
 *   LM head, slot 1+k = head k).
 * T may be every tree row (the all-rows variant, e.g. T = N = 341); bf16 with
 * T >= 2 runs on the tensor cores in passes of up to 128 rows, each reading the
 * weights once.
 * Limits: 1 <= T <= MEDUSA_MAX_HEAD_ROWS, d % 8 == 0, topk <= MEDUSA_MAX_TOPK, topk <= V. */
medusa_status medusa_heads_topk(const void *h, int32_t T, int32_t d, int32_t V, int32_t K,
                                const void *w1, const void *b1, const void *w2,
                                int64_t w2_head_stride, const void *w_lm, int32_t topk,
                                medusa_dtype dt, int32_t *root, int32_t *pool,
                                float *logits_out, void *ws, size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * Round step 2: tree fill
 * ------------------------------------------------------------------------- */

/* tokens[b][u] = cand_b[slot[u]] with cand_b = [root[b], pool[b][0][:], pool[b][1][:], ...]
 * and pos[b][u] = L[b] + depth[u] ([M7.2] §0x01B, §0x04A "Candidate gather",
 * "Visibility and position"; [CN] "手算一棵两层候选树").
 *   t: device template; root [B]; pool [B][K][t->topk] (K >= t->max_depth);
 *   L [B]; tokens, pos [B][N]. */
medusa_status medusa_tree_fill(const medusa_tree_t *t, int32_t B, int32_t K, const int32_t *root,
                               const int32_t *pool, const int32_t *L, int32_t *tokens,
                               int32_t *pos, void *stream);

/* ---------------------------------------------------------------------------
 * Round step 3: tree verification attention
 * ------------------------------------------------------------------------- */

size_t medusa_tree_attn_workspace(const medusa_tree_t *t, int32_t B, int32_t n_q_heads,
                                  const medusa_kv_t *cache, int32_t max_prefix);

/* Tree attention of [M7.2] §0x03C ([CN] "Tree Attention"; [Math] "Tree attention:
 * the mask math").  For sequence b with committed length L = L[b] and each tree
 * row u at logical position L + depth[u]:
 *   q' = RoPE(q[b][u][h], L + depth[u]),  k'_u = RoPE(k_new[b][u][kv], L + depth[u])
 *   (rotate-half pairs (i, i + dh/2), angle pos * rope_base^(-2i/dh));
 *   out[b][u][h] = softmax(scale * q' . K^T) V over keys {cache rows 0..L-1}
 *                  union {tree rows v with anc[u] bit v}, with tree keys k'_v and values v_new[v];
 *   the staged rows L + u of the cache receive k'_u and v_new[b][u] ([M7.2] §0x03E).
 * Query head h reads KV head h / (n_q_heads / n_kv_heads).  The cache prefix K is
 * already rotated.  Rows >= L of the cache are never read as prefix keys.
 *   q [B][N][n_q_heads][head_dim]; k_new, v_new [B][N][n_kv_heads][head_dim] in the
 *   cache dtype; L [B]; max_prefix >= every L[b] (sizes the split-KV grid);
 *   out [B][N][n_q_heads][head_dim] fp32 (the accumulation precision: a bf16 output
 *   would add ~1.6e-3 relative rounding error); lse [B][N][n_q_heads] fp32
 *   natural-log log-sum-exp, or NULL; status [B]: 0, or MEDUSA_ECAPACITY when
 *   L[b] + N > capacity (sequence b is not touched), MEDUSA_ETIMEOUT when a bounded
 *   wait gave up, MEDUSA_ERANGE (bf16 tensor-core path) when an output of b is not
 *   finite: a K/V value or a scaled rotated query outside fp16's range (|x| > 65504)
 *   becomes inf, which makes the softmax of every row whose score of that key is +inf
 *   (or whose value row or query is inf) NaN.  A key that overflows only to scores of
 *   -inf drops out of those rows' softmax without a report.
 *   ws: workspace of medusa_tree_attn_workspace(...) bytes (16-byte aligned),
 *   zero-filled once before its first use.  Its first 256 KiB hold split-KV ticket
 *   counters that every call returns to zero, so one workspace can serve later
 *   calls of any shape without clearing; the rest is scratch.  Calls that share a
 *   workspace must not run concurrently.
 * Arithmetic: fp32 kernels for MEDUSA_F32; for MEDUSA_BF16 with head_dim 128 the
 * prefix and the tree rows run on tcgen05 tensor cores with fp16 operands (q' and P
 * rounded to fp16, bf16 K/V converted exactly for |x| in [2^-14, 65504]) and fp32
 * accumulation and softmax. */
medusa_status medusa_tree_attn_verify(const medusa_tree_t *t, int32_t B, int32_t n_q_heads,
                                      const void *q, const void *k_new, const void *v_new,
                                      const medusa_kv_t *cache, const int32_t *L,
                                      int32_t max_prefix, float rope_base, float scale,
                                      float *out, float *lse, int32_t *status, void *ws,
                                      size_t ws_bytes, void *stream);

/* Size of the fixed device scratch used by medusa_tree_attn_verify_static. */
#define MEDUSA_ATTN_STATIC_SCRATCH_BYTES (32u * 1024u * 1024u)

/* medusa_tree_attn_verify without a workspace argument, for callers that cannot
 * allocate device memory where they call it: for example a plugin or custom-op
 * interface that is handed only its input and output pointers, or a serving loop
 * whose device memory is reserved up front, where a cudaMalloc would fail or would
 * synchronise the device.  The pages describe no such variant; it exists only for
 * these callers.
 *
 * Arguments and results are those of medusa_tree_attn_verify.  The scratch is a
 * file-scope device array of MEDUSA_ATTN_STATIC_SCRATCH_BYTES (32 MiB) that every
 * GPU loading this library holds until the process exits.  A shape whose scratch
 * would exceed it returns MEDUSA_EWORKSPACE with nothing enqueued; use
 * medusa_tree_attn_verify with a caller workspace for such shapes.
 * The call allocates nothing: no cudaMalloc, no cudaFree, no allocating library
 * routine.  The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and caches it for the life of the
 * process; make that first call before any stream capture.  A cudaDeviceReset of that
 * device invalidates the cached address: make no further call of this entry point on
 * a device after resetting it.  Each call clears, with cudaMemsetAsync on `stream`,
 * what must start at zero (the ticket counters it will use, and `status`) and
 * otherwise reuses whatever the previous call left in the array.  All calls share
 * that one array, so calls that can overlap on the GPU (different streams without
 * ordering between them) race and must not be issued. */
medusa_status medusa_tree_attn_verify_static(const medusa_tree_t *t, int32_t B, int32_t n_q_heads,
                                             const void *q, const void *k_new, const void *v_new,
                                             const medusa_kv_t *cache, const int32_t *L,
                                             int32_t max_prefix, float rope_base, float scale,
                                             float *out, float *lse, int32_t *status, void *stream);

/* ---------------------------------------------------------------------------
 * Round step 4: acceptance
 * ------------------------------------------------------------------------- */

size_t medusa_tree_accept_workspace(const medusa_tree_t *t, int32_t B, int32_t V);

/* Greedy or fast-typical acceptance ([M7.2] §0x03D, §0x04D, §0x04E; [PartII] Part 7;
 * [CN] "接受机制").  Target row u scores the token of its child: along retrieval
 * path p = [u_0, u_1, ...] edge j passes when
 *   greedy:  tokens[u_{j+1}] == argmax(logits[u_j])   (lowest id among maxima)
 *   typical: p_j > min(epsilon, delta * exp(-H_j)) with p = softmax(logits[u_j] / T)
 *            evaluated at tokens[u_{j+1}] and H_j its entropy (entropy_guard = 1
 *            uses -sum p log(p + 1e-5) instead of the exact entropy).
 * a_p = edges before the first failure.  Winner: largest a_p; greedy takes the
 * first such path (path 0 when none passes); typical takes the largest
 * sum_{j<a} log p_j, then the lowest path index.  Row statistics are computed
 * once per internal row (rows without children are never read).
 *   logits [B][N][V] in dtype dt; tokens [B][N];
 *   best_path [B]; accept_len [B] (a); out_tokens, out_rows [B][D+1] (G = a + 1
 *   entries, then -1); frontier_row [B] (u_a, [M7.2] §0x06C).
 * ws: medusa_tree_accept_workspace(...) bytes. */
medusa_status medusa_tree_accept(const medusa_tree_t *t, int32_t B, int32_t V, const void *logits,
                                 medusa_dtype dt, const int32_t *tokens, int32_t mode,
                                 float temperature, float epsilon, float delta,
                                 int32_t entropy_guard, int32_t *best_path, int32_t *accept_len,
                                 int32_t *out_tokens, int32_t *out_rows, int32_t *frontier_row,
                                 void *ws, size_t ws_bytes, void *stream);

/* medusa_tree_accept followed by medusa_kv_compact of the winning rows, in the same
 * kernel that picks the winner ([CN] "把 Python 控制流赶出热路径" ranks a fused index
 * and K/V commit among the changes worth most): the acceptance outputs are those of
 * medusa_tree_accept, and cache, L_out and status end as medusa_kv_compact leaves them
 * (same validation; a rejected sequence is untouched).  One launch fewer per round.
 * ws: medusa_tree_accept_workspace(...) bytes.  L_out must not alias L. */
medusa_status medusa_tree_accept_commit(const medusa_tree_t *t, int32_t B, int32_t V, const void *logits,
                                        medusa_dtype dt, const int32_t *tokens, int32_t mode, float temperature,
                                        float epsilon, float delta, int32_t entropy_guard,
                                        const medusa_kv_t *cache, const int32_t *L, int32_t *best_path,
                                        int32_t *accept_len, int32_t *out_tokens, int32_t *out_rows,
                                        int32_t *frontier_row, int32_t *L_out, int32_t *status, void *ws,
                                        size_t ws_bytes, void *stream);

size_t medusa_tree_accept_hidden_workspace(const medusa_tree_t *t, int32_t B, int32_t V, int32_t d);

/* medusa_tree_accept with the target's vocabulary projection folded in ([M7.2] §0x07B:
 * the projection C_LMproj with F_LMproj = 2 N d V and a unique-row posterior; §0x07C:
 * dense target logits hold N V elements).  For each internal row u of sequence b the
 * logits x = W_LM hidden[b][u] are computed on the tensor cores (bf16 operands, fp32
 * accumulation) and reduced at once to what acceptance reads: the argmax, and for
 * typical acceptance the max, partition function and first moment of x / T and x at
 * the token of each child of u.  The [rows x V] logits are never written; leaves are
 * not projected.  Decisions are those of medusa_tree_accept on the same fp32 logits,
 * up to the summation order of the projection.
 *   hidden [B][N][d] bf16: the target's final hidden state of every tree row;
 *   w_lm [V][d] bf16; tokens, mode, temperature, epsilon, delta and the outputs as in
 *   medusa_tree_accept (the guarded entropy is not offered: it needs a second pass
 *   over the logits).  W_LM is streamed once per 256 internal rows of the batch.
 * A bounded device wait that gives up makes every sequence publish nothing:
 * best_path = accept_len = frontier_row = -1 and out_rows, out_tokens all -1 (the
 * following medusa_kv_compact then rejects the sequence).
 * ws: medusa_tree_accept_hidden_workspace(...) bytes, 16-byte aligned.
 * Limits: d a multiple of 64; MEDUSA_EUNSUPPORTED otherwise. */
medusa_status medusa_tree_accept_hidden(const medusa_tree_t *t, int32_t B, int32_t V, int32_t d,
                                        const void *hidden, const void *w_lm, const int32_t *tokens,
                                        int32_t mode, float temperature, float epsilon, float delta,
                                        int32_t *best_path, int32_t *accept_len, int32_t *out_tokens,
                                        int32_t *out_rows, int32_t *frontier_row, void *ws, size_t ws_bytes,
                                        void *stream);

/* ---------------------------------------------------------------------------
 * Round step 5: winning-path K/V compaction
 * ------------------------------------------------------------------------- */

/* Gather-and-compact of [M7.2] §0x06A-§0x06B: with G = accept_len[b] + 1 and
 * rows u_j = out_rows[b][j], cache rows L + u_j are read into a snapshot first
 * and then written to rows L + j, for K and V of every KV head; L_out[b] = L + G.
 * The path is validated first (G <= D + 1, u_0 = 0, each u_j a child of u_{j-1},
 * L + N <= capacity); an invalid sequence gets status[b] = MEDUSA_EPATH or
 * MEDUSA_ECAPACITY, L_out[b] = L[b] and no cache write.
 *   t: device template (its parent array validates the chain); L, accept_len [B];
 *   out_rows [B][D+1]; L_out [B] (must not alias L); status [B]. */
medusa_status medusa_kv_compact(const medusa_kv_t *cache, const medusa_tree_t *t, int32_t B,
                                const int32_t *L, const int32_t *accept_len,
                                const int32_t *out_rows, int32_t *L_out, int32_t *status,
                                void *stream);

/* medusa_kv_compact for every layer of the model at once ([M7.2] §0x06B: the accepted
 * rows are committed in each layer's cache, and uncommitted rows are never
 * published).  caches [host] [n_layers] descriptors that differ only in k and v: the
 * same dtype, head counts, capacity, page size and block table (a paged cache shares
 * its block table across layers).  The path of each sequence is validated once, as in
 * medusa_kv_compact; a rejected sequence is left untouched in every layer.  One
 * kernel launch per 128 layers.  L_out must not alias L.
 * Limits: 1 <= n_layers <= MEDUSA_MAX_LAYERS. */
medusa_status medusa_kv_compact_layers(const medusa_kv_t *caches, int32_t n_layers, const medusa_tree_t *t,
                                       int32_t B, const int32_t *L, const int32_t *accept_len,
                                       const int32_t *out_rows, int32_t *L_out, int32_t *status,
                                       void *stream);

/* Fill a bf16 cache's fp16 mirror (see medusa_kv_t): every element of k and v,
 * converted to fp16 (round to nearest even; beyond 65504 it becomes inf), written to
 * k_f16 and v_f16 over the whole buffers: B * n_kv_heads * capacity * head_dim
 * elements each for a contiguous cache (B: its sequences), n_pages * n_kv_heads * 16 *
 * head_dim for a paged one (B unused).  For a cache filled outside this library (a
 * prefill); after that the library's own writes keep the mirror in step.
 * MEDUSA_EINVAL for a cache without a mirror, not bf16, or B < 1 (contiguous).
 * Stream-ordered. */
medusa_status medusa_kv_mirror_sync(const medusa_kv_t *cache, int32_t B, void *stream);

/* ---------------------------------------------------------------------------
 * Whole round: the five calls as one CUDA graph
 * ------------------------------------------------------------------------- */

/* A replayable round over fixed buffers, with acceptance decided on the device and no
 * host round trip between the steps ([CN] "把 Python 控制流赶出热路径" ranks this above
 * adding heads; [CN] "Mask、位置和 KV 必须一起验证": fixed buffer addresses are what
 * allow a CUDA graph).
 *
 * Every argument of the five calls of one round (steps 1-5 above), with one frontier
 * row per sequence for the heads (T = B).  Pointers are device buffers that the
 * caller keeps alive and fixed while the round exists: the graph records the
 * addresses, so new inputs are written into the same buffers before each launch.
 * `tree` and `cache` are copied at creation (their device arrays are referenced).
 * Fields have the meaning they have in the call they belong to. */
typedef struct {
  medusa_tree_t tree;        /* device template */
  int32_t B;                 /* sequences */
  medusa_dtype dtype;        /* heads weights, hidden rows, logits (the cache has its own) */
  /* step 1: medusa_heads_topk with T = B */
  const void *h;             /* [B][d] */
  int32_t d, V, K, topk;
  const void *w1, *b1, *w2;  /* b1 may be NULL */
  int64_t w2_head_stride;
  const void *w_lm;
  int32_t *root, *pool;      /* [B], [B][K][topk] */
  /* step 2: medusa_tree_fill */
  const int32_t *L;          /* [B] */
  int32_t *tokens, *pos;     /* [B][N] */
  /* step 3: medusa_tree_attn_verify */
  int32_t n_q_heads;
  const void *q, *k_new, *v_new;
  medusa_kv_t cache;
  int32_t max_prefix;
  float rope_base, scale;
  float *out, *lse;          /* lse may be NULL */
  int32_t *attn_status;      /* [B] */
  /* step 4: medusa_tree_accept on logits [B][N][V] in dtype */
  const void *logits;
  int32_t mode;
  float temperature, epsilon, delta;
  int32_t entropy_guard;
  int32_t *best_path, *accept_len, *out_tokens, *out_rows, *frontier_row;
  /* step 5: medusa_kv_compact */
  int32_t *L_out, *compact_status;   /* [B], [B] */
  /* step 4 alternative: when non-NULL, acceptance is medusa_tree_accept_hidden on the
   * target's final hidden states [B][N][d] (bf16, the heads' d) with the same w_lm,
   * and `logits` is not read (it may be NULL) */
  const void *hidden_target;
  /* non-zero: steps 4 and 5 as one (medusa_tree_accept_commit: the winning rows are
   * committed by the acceptance kernel; L_out and compact_status as in step 5) */
  int32_t fuse_commit;
} medusa_round_desc;

typedef struct medusa_round_s *medusa_round_t;

/* Workspace bytes of a round: the heads, attention and acceptance workspaces, each
 * 256-byte aligned, back to back.  0 when the descriptor is invalid. */
size_t medusa_round_workspace(const medusa_round_desc *r);

/* Checks the descriptor as the five calls would, zero-fills the workspace, then
 * records the five calls (on a private stream under thread-local stream capture) and
 * instantiates the graph.  ws: medusa_round_workspace(r) bytes, 16-byte aligned,
 * owned by the caller and used only by this round's launches.  `stream` orders the
 * workspace clearing before the capture; creation returns after that clearing
 * completed.  Creation allocates the graph objects (host memory and driver
 * resources; no device buffers).  Any status of the recorded calls is returned as is,
 * with no round created. */
medusa_status medusa_round_create(const medusa_round_desc *r, void *ws, size_t ws_bytes, void *stream,
                                  medusa_round_t *round_out);

/* Enqueues the whole round on `stream`: one graph launch, no host synchronisation.
 * Launches of one round must not overlap each other (they share the workspace and
 * the output buffers): launch on one stream, or order the streams. */
medusa_status medusa_round_launch(medusa_round_t round, void *stream);

/* Frees the graph objects.  The caller must make sure no launch is still running. */
medusa_status medusa_round_destroy(medusa_round_t round);

/* ---------------------------------------------------------------------------
 * Misc
 * ------------------------------------------------------------------------- */

const char *medusa_status_string(medusa_status s);
int32_t medusa_abi_version(void);

/* Testing only: makes the timeout path of the bounded device waits observable without
 * a fault.  With ns > 0, every later launch of the bf16 tensor-core tree attention and
 * of the one-row heads weight stream first waits on a flag that nothing sets; after ns
 * nanoseconds the wait gives up and the launch takes its error path (attention:
 * status[b] = MEDUSA_ETIMEOUT with no output, staged row or cache write; heads: root
 * and pool -1, no logits written).  ns = 0 (the default) turns it off.  A process-wide
 * setting read when a call is enqueued; not for use while other threads issue calls.
 * The pages have no counterpart: it exists to test this library. */
void medusa_test_set_stall_ns(uint64_t ns);

#ifdef __cplusplus
}
#endif

#endif /* MEDUSA_GB300_H */
