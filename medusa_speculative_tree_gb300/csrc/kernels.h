// Internal launcher declarations shared by the C ABI (medusa_api.cpp) and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "medusa_gb300.h"

#include <atomic>

namespace medusa {

// Test hook of medusa_test_set_stall_ns: when non-zero, the tensor-core attention and
// the heads weight stream first wait this many nanoseconds on a flag that nothing
// sets, then take their error path.  0 (the default) in normal operation.
extern std::atomic<uint64_t> g_test_stall_ns;
uint64_t test_stall_ns();

// ---- heads + top-k ---------------------------------------------------------
struct HeadsPlan {
  int T, d, V, K, topk;
  int tokens_per_pass;   // tokens whose fp32 x rows fit in shared memory at once
  size_t off_z, off_logits, off_scand, off_zhl, off_cand, off_err, bytes;
};
// Weight-stream path (heads_stream.cu): at most this many CTAs, and an error flag plus
// completion counters in the first kHeadsCounterBytes at off_err (zeroed every call).
// Hidden rows per pass of the tensor-core heads stream (more rows run in passes): up to
// 128 rows as bf16 pairs; calls of more rows run "wide" passes of up to 256 single rows
// (z in fp16, W2 re-encoded to fp16 in shared memory).
constexpr int kHeadsMmaMaxRows = 128;
constexpr int kHeadsMmaWideRows = 256;
inline bool heads_mma_wide(int T) { return T > kHeadsMmaMaxRows; }
constexpr int kHeadsStreamMaxGrid = 256;
constexpr size_t kHeadsCounterBytes = 256;
HeadsPlan plan_heads(int T, int d, int V, int K, int topk);
bool heads_stream_supported(int T, int d, int V, int K, int topk, medusa_dtype dt, const void* h, const void* w1,
                            const void* w2, int64_t w2_stride, const void* w_lm, const void* b1);
cudaError_t launch_heads_stream(const HeadsPlan& p, const void* h, const void* w1, const void* b1, const void* w2,
                                int64_t w2_stride, const void* w_lm, int32_t* root, int32_t* pool,
                                float* logits_out, void* ws, cudaStream_t st);
// Tensor-core path for T >= 2 hidden rows (heads_mma.cu), one pass of at most 128 (or,
// wide, 256) rows: writes all logits, the top-k kernels then select.  Input rows of the
// MMA: 2T (pairs) or T (wide) rounded up to 32.
size_t heads_mma_rows(int T, bool wide);
bool heads_mma_supported(int T, int d, int V, int K, medusa_dtype dt, const void* h, const void* w1, const void* w2,
                         int64_t w2_stride, const void* w_lm);
cudaError_t launch_heads_mma(const HeadsPlan& p, bool wide, const void* h, const void* w1, const void* b1,
                             const void* w2, int64_t w2_stride, const void* w_lm, float* logits, void* ws,
                             cudaStream_t st);
cudaError_t launch_heads(const HeadsPlan& p, const void* h, const void* w1, const void* b1,
                         const void* w2, int64_t w2_stride, const void* w_lm, medusa_dtype dt,
                         int32_t* root, int32_t* pool, float* logits_out, void* ws,
                         cudaStream_t st);

// ---- tree templates on the device (tree_build.cu) --------------------------------
// Offsets of the template arrays inside one blob (the layout of medusa_tree_compile).
struct TreeBlobLayout {
  size_t slot, depth, parent, internal, internal_index, retrieve, anc, total;
};
TreeBlobLayout tree_blob_layout(int n_rows, int max_depth, int n_paths);
// Entries (paths created) of one greedy search: R per admitted path plus the first R.
constexpr int kMaxGreedyEntries = 6144;
size_t tree_greedy_smem(int R, int budget);
// One CTA per sequence: greedy frontier search on acc [B][K][R], then the template of the
// chosen paths into blob b of dev_buf (blob_stride bytes each, layout for budget + 1
// rows); per_seq[b] and status[b] (nullable) are written by the kernel.
cudaError_t launch_tree_greedy(const double* acc, int B, int K, int R, int budget, int topk, void* dev_buf,
                               size_t blob_stride, medusa_tree_t* per_seq, int32_t* status, cudaStream_t st);

// ---- tree fill ----------------------------------------------------------------
cudaError_t launch_tree_fill(const medusa_tree_t& t, int B, int K, const int32_t* root,
                             const int32_t* pool, const int32_t* L, int32_t* tokens,
                             int32_t* pos, cudaStream_t st);

// ---- tree attention -------------------------------------------------------------
struct AttnPlan {
  int B, Hq, Hkv, g, dh, N, D, max_prefix;
  int path;              // 0 = CUDA-core kernel, 1 = tcgen05 kernel
  int mt_rows;           // query rows (tree row x group member) per CTA
  int n_mt;              // ceil(N * g / mt_rows)
  int key_tile;          // keys per pipeline stage
  int n_split;           // CTAs along the prefix per (b, kv head, m tile)
  int chunk;             // prefix keys per split (multiple of key_tile)
  int first;             // prefix keys of split 0 (tensor-core path; split 0 also runs the tree rows)
  int qt, stages;        // tensor-core path: 128-row query tiles per CTA, K/V stages in the ring
  size_t off_counter, off_part_o, off_part_ml, off_tmap, bytes;
};
// Bytes reserved for split-KV ticket counters at the start of the attention workspace.
constexpr size_t kAttnCounterBytes = 256 * 1024;
constexpr size_t kAttnMaxUnits = kAttnCounterBytes / sizeof(int);
AttnPlan plan_attn(const medusa_tree_t& t, int B, int Hq, const medusa_kv_t& c, int max_prefix);
size_t attn_units(const AttnPlan& p);
// Device address of the fixed scratch array of medusa_tree_attn_verify_static on the
// current device (looked up once per device, then cached).
cudaError_t attn_static_scratch(void** ptr);
cudaError_t launch_attn(const AttnPlan& p, const medusa_tree_t& t, const void* q,
                        const void* k_new, const void* v_new, const medusa_kv_t& c,
                        const int32_t* L, float rope_base, float scale, float* out, float* lse,
                        int32_t* status, void* ws, cudaStream_t st);

// ---- acceptance -------------------------------------------------------------------
// Statistics of one chunk of one internal row's logits, merged by the select kernel.
struct RowPart {
  float m;      // max of x / T over the chunk
  float z;      // sum exp(x/T - m)
  float s1;     // sum exp(x/T - m) * (x/T - m)
  float amax_v; // largest raw logit (-inf from row_stats_kernel's typical pass, which skips it)
  int amax_i;   // its id (lowest among equal values; INT_MAX when not taken)
  int pad[3];
};

// Fused index + K/V commit ([CN] "把 Python 控制流赶出热路径"): when `on`, the select
// kernel also performs medusa_kv_compact for its sequence, with the same validation
// and status.  Default: off.
struct CommitArgs {
  medusa_kv_t c;
  int on;
  const int32_t* L;
  int32_t* L_out;
  int32_t* status;
};

struct AcceptPlan {
  int B, V, chunk, n_chunks;
  size_t off_part, off_guard, bytes;
};
AcceptPlan plan_accept(const medusa_tree_t& t, int B, int V);
cudaError_t launch_accept(const AcceptPlan& p, const medusa_tree_t& t, const void* logits,
                          medusa_dtype dt, const int32_t* tokens, int mode, float temperature,
                          float epsilon, float delta, int entropy_guard, int32_t* best_path,
                          int32_t* accept_len, int32_t* out_tokens, int32_t* out_rows,
                          int32_t* frontier_row, void* ws, cudaStream_t st, const CommitArgs& cm = CommitArgs{});

// The select step alone, on chunk statistics and per-edge logits written by another
// kernel (edge_x [B][N]: the logit of row v's token at its parent); err (nullable)
// non-zero makes every sequence publish nothing (accept_len = -1).
cudaError_t launch_select_parts(const medusa_tree_t& t, int B, int V, int n_chunks, const RowPart* part,
                                const float* edge_x, const int* err, const int32_t* tokens, int mode,
                                float temperature, float epsilon, float delta, int32_t* best_path,
                                int32_t* accept_len, int32_t* out_tokens, int32_t* out_rows,
                                int32_t* frontier_row, cudaStream_t st, const CommitArgs& cm = CommitArgs{});

// Acceptance with the target's vocabulary projection folded in (lm_accept.cu).
struct LmAcceptPlan {
  int B, V, d, NI, cols, cols_pad, n_chunks;
  size_t off_x, off_etok, off_erow, off_ecnt, off_edge_x, off_part, off_err, bytes;
};
LmAcceptPlan plan_lm_accept(const medusa_tree_t& t, int B, int V, int d);
bool lm_accept_supported(int d, int V);
cudaError_t launch_lm_accept(const LmAcceptPlan& p, const medusa_tree_t& t, const void* hidden, const void* w_lm,
                             const int32_t* tokens, int mode, float temperature, float epsilon, float delta,
                             int32_t* best_path, int32_t* accept_len, int32_t* out_tokens, int32_t* out_rows,
                             int32_t* frontier_row, void* ws, cudaStream_t st, const CommitArgs& cm = CommitArgs{});

// ---- compaction -----------------------------------------------------------------------
cudaError_t launch_kv_compact(const medusa_kv_t& c, const medusa_tree_t& t, int B,
                              const int32_t* L, const int32_t* accept_len,
                              const int32_t* out_rows, int32_t* L_out, int32_t* status,
                              cudaStream_t st);
// All layers' caches in launches of up to kCompactLayersPerLaunch layers (their K/V
// pointers travel in the kernel parameters); the other descriptor fields are those of
// layers[0], which the caller has checked to be common to every layer.
constexpr int kCompactLayersPerLaunch = 128;
cudaError_t launch_kv_compact_layers(const medusa_kv_t* layers, int n_layers, const medusa_tree_t& t, int B,
                                     const int32_t* L, const int32_t* accept_len, const int32_t* out_rows,
                                     int32_t* L_out, int32_t* status, cudaStream_t st);

// The fp16 mirror of a bf16 cache: n elements of k and of v converted (whole buffers).
cudaError_t launch_kv_mirror_sync(const medusa_kv_t& c, int64_t n, cudaStream_t st);

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace medusa
