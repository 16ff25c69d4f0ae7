// C ABI of libmedusa_gb300.so: argument validation, host-side template
// construction and dispatch to the kernel launchers.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <map>
#include <new>
#include <vector>

#include "kernels.h"
#include "medusa_gb300.h"

using medusa::align_up;

namespace medusa {
std::atomic<uint64_t> g_test_stall_ns{0};
uint64_t test_stall_ns() { return g_test_stall_ns.load(std::memory_order_relaxed); }
}  // namespace medusa

namespace {

cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

medusa_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MEDUSA_OK : MEDUSA_ECUDA; }

bool dtype_ok(medusa_dtype d) { return d == MEDUSA_F32 || d == MEDUSA_BF16; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

typedef std::vector<int32_t> Path;

// Canonical order: shorter first, then lexicographic ([M7.2] §0x04A).
bool canon_less(const Path& a, const Path& b) {
  if (a.size() != b.size()) return a.size() < b.size();
  return a < b;
}

// Selection order of the greedy search: larger weight first; weights within
// 1e-12 relative tie and fall back to the canonical order.
bool greedy_before(double wa, const Path& pa, double wb, const Path& pb) {
  const double big = std::max(wa, wb);
  if (std::fabs(wa - wb) <= 1e-12 * big) return canon_less(pa, pb);
  return wa > wb;
}

double path_weight(const Path& p, const double* acc, int R) {
  double w = 1.0;
  for (size_t j = 0; j < p.size(); ++j) w = w * acc[j * R + p[j]];
  return w;
}

using BlobLayout = medusa::TreeBlobLayout;
BlobLayout blob_layout(int n_rows, int max_depth, int n_paths) { return medusa::tree_blob_layout(n_rows, max_depth, n_paths); }

size_t blob_end(const medusa_tree_t* t, const void* base) {
  const char* anc_end = reinterpret_cast<const char*>(t->anc + (size_t)t->n_rows * t->n_words);
  return align_up((size_t)(anc_end - reinterpret_cast<const char*>(base)), 16);
}

// A template, or a per-sequence batch (per_seq set: the counts are bounds, the arrays
// are not read; the per-sequence templates live in device memory, out of the host's view).
bool tree_ok(const medusa_tree_t* t) {
  if (!t || t->n_rows < 1 || t->n_rows > MEDUSA_MAX_ROWS || t->max_depth < 0 || t->max_depth > MEDUSA_MAX_DEPTH ||
      t->n_paths < 1 || t->topk < 1 || t->topk > MEDUSA_MAX_TOPK || t->n_words != (t->n_rows + 63) / 64 ||
      t->n_internal < 0 || t->n_internal > t->n_rows)
    return false;
  if (t->per_seq) return (reinterpret_cast<uintptr_t>(t->per_seq) & 7u) == 0;
  return t->slot && t->depth && t->parent && t->retrieve && t->internal && t->internal_index && t->anc;
}

bool kv_ok(const medusa_kv_t* c) {
  if (!c || !c->k || !c->v || !dtype_ok(c->dtype) || c->n_kv_heads < 1 || c->capacity < 1) return false;
  if (c->head_dim != 64 && c->head_dim != 128) return false;
  if (!aligned16(c->k) || !aligned16(c->v)) return false;
  if (c->page_size != 0) {
    if (c->page_size != 16 || !c->block_table || c->max_blocks < 1 || c->n_pages < 1) return false;
    if (c->capacity > c->max_blocks * c->page_size) return false;
  }
  // an fp16 mirror: both halves, a bf16 cache, aligned like the cache
  if (c->k_f16 || c->v_f16) {
    if (!c->k_f16 || !c->v_f16 || c->dtype != MEDUSA_BF16) return false;
    if (!aligned16(c->k_f16) || !aligned16(c->v_f16)) return false;
  }
  return true;
}

medusa_status accept_logits_impl(const medusa_tree_t* t, int32_t B, int32_t V, const void* logits, medusa_dtype dt,
                                 const int32_t* tokens, int32_t mode, float temperature, float epsilon,
                                 float delta, int32_t entropy_guard, int32_t* best_path, int32_t* accept_len,
                                 int32_t* out_tokens, int32_t* out_rows, int32_t* frontier_row, void* ws,
                                 size_t ws_bytes, void* stream, const medusa::CommitArgs& cm);

}  // namespace

extern "C" {

int32_t medusa_abi_version(void) { return 5; }

void medusa_test_set_stall_ns(uint64_t ns) { medusa::g_test_stall_ns.store(ns, std::memory_order_relaxed); }

const char* medusa_status_string(medusa_status s) {
  switch (s) {
    case MEDUSA_OK: return "ok";
    case MEDUSA_EINVAL: return "invalid argument";
    case MEDUSA_ECAPACITY: return "cache capacity exceeded";
    case MEDUSA_EUNSUPPORTED: return "unsupported shape";
    case MEDUSA_ETEMPLATE: return "invalid tree template";
    case MEDUSA_ECUDA: return "CUDA runtime error";
    case MEDUSA_EWORKSPACE: return "workspace or output buffer too small";
    case MEDUSA_EPATH: return "accepted path is not a valid tree chain";
    case MEDUSA_ETIMEOUT: return "a bounded device wait gave up";
    case MEDUSA_ERANGE: return "a value outside the range of the kernel's fp16 operands";
    default: return "unknown status";
  }
}

medusa_status medusa_tree_regular(const int32_t* widths, int32_t K, int32_t* paths_out,
                                  int32_t max_paths, int32_t* n_out) {
  if (!widths || K < 0 || K > MEDUSA_MAX_DEPTH || !n_out || (max_paths > 0 && !paths_out))
    return MEDUSA_EINVAL;
  std::vector<Path> level(1), all;
  for (int k = 0; k < K; ++k) {
    if (widths[k] < 1 || widths[k] > MEDUSA_MAX_TOPK) return MEDUSA_EINVAL;
    std::vector<Path> next;
    for (const Path& p : level)
      for (int r = 0; r < widths[k]; ++r) {
        Path c = p;
        c.push_back(r);
        next.push_back(c);
        if ((int64_t)all.size() + (int64_t)next.size() > MEDUSA_MAX_ROWS) return MEDUSA_EUNSUPPORTED;
      }
    all.insert(all.end(), next.begin(), next.end());
    level.swap(next);
  }
  *n_out = (int32_t)all.size();
  if (!paths_out && max_paths == 0) return MEDUSA_OK;          // a size query
  if ((int32_t)all.size() > max_paths) return MEDUSA_EWORKSPACE;
  for (size_t i = 0; i < all.size(); ++i)
    for (int j = 0; j < K; ++j) paths_out[i * K + j] = j < (int)all[i].size() ? all[i][j] : -1;
  return MEDUSA_OK;
}

medusa_status medusa_tree_greedy(const double* acc, int32_t K, int32_t R, int32_t budget,
                                 int32_t* paths_out, int32_t* n_out) {
  if (!acc || K < 1 || K > MEDUSA_MAX_DEPTH || R < 1 || R > MEDUSA_MAX_TOPK || budget < 0 ||
      budget >= MEDUSA_MAX_ROWS || !n_out || (budget > 0 && !paths_out))
    return MEDUSA_EINVAL;
  for (int i = 0; i < K * R; ++i)
    if (!(acc[i] >= 0.0 && acc[i] <= 1.0)) return MEDUSA_EINVAL;
  // frontier kept in canonical order so that scans visit it in (len, path) order
  std::map<Path, double, bool (*)(const Path&, const Path&)> frontier(canon_less);
  for (int r = 0; r < R; ++r) {
    Path p{r};
    frontier[p] = path_weight(p, acc, R);
  }
  int n = 0;
  while (n < budget && !frontier.empty()) {
    auto best = frontier.begin();
    for (auto it = std::next(frontier.begin()); it != frontier.end(); ++it)
      if (greedy_before(it->second, it->first, best->second, best->first)) best = it;
    const Path chosen = best->first;
    frontier.erase(best);
    for (int j = 0; j < K; ++j) paths_out[(size_t)n * K + j] = j < (int)chosen.size() ? chosen[j] : -1;
    ++n;
    if ((int)chosen.size() < K) {
      for (int r = 0; r < R; ++r) {
        Path c = chosen;
        c.push_back(r);
        frontier[c] = path_weight(c, acc, R);
      }
    }
  }
  *n_out = n;
  return MEDUSA_OK;
}

size_t medusa_tree_bytes(int32_t n_paths, int32_t max_len) {
  if (n_paths < 0 || max_len < 0) return 0;
  const int n_rows = n_paths + 1;
  return blob_layout(n_rows, max_len, n_rows).total;
}

medusa_status medusa_tree_compile(const int32_t* paths, int32_t n_paths, int32_t max_len,
                                  int32_t topk, int32_t n_heads, void* host_buf,
                                  size_t host_bytes, medusa_tree_t* out) {
  if (n_paths < 0 || max_len < 0 || (n_paths > 0 && (!paths || max_len < 1)) || !host_buf || !out ||
      topk < 1 || topk > MEDUSA_MAX_TOPK || n_heads < 0)
    return MEDUSA_EINVAL;
  if ((reinterpret_cast<uintptr_t>(host_buf) & 7u) != 0) return MEDUSA_EINVAL;
  if (n_paths + 1 > MEDUSA_MAX_ROWS) return MEDUSA_EUNSUPPORTED;
  if (host_bytes < medusa_tree_bytes(n_paths, max_len)) return MEDUSA_EWORKSPACE;

  std::vector<Path> ps;
  ps.reserve(n_paths);
  for (int i = 0; i < n_paths; ++i) {
    Path p;
    bool ended = false;
    for (int j = 0; j < max_len; ++j) {
      const int32_t r = paths[(size_t)i * max_len + j];
      if (r < 0) { ended = true; continue; }
      if (ended) return MEDUSA_ETEMPLATE;          // a rank after the padding
      if (r >= topk) return MEDUSA_ETEMPLATE;
      p.push_back(r);
    }
    if (p.empty()) return MEDUSA_ETEMPLATE;
    if ((int)p.size() > MEDUSA_MAX_DEPTH) return MEDUSA_EUNSUPPORTED;
    if (n_heads > 0 && (int)p.size() > n_heads) return MEDUSA_ETEMPLATE;
    ps.push_back(p);
  }
  std::sort(ps.begin(), ps.end(), canon_less);
  for (size_t i = 1; i < ps.size(); ++i)
    if (ps[i] == ps[i - 1]) return MEDUSA_ETEMPLATE;
  std::map<Path, int> row;
  row[Path()] = 0;
  for (size_t i = 0; i < ps.size(); ++i) row[ps[i]] = (int)i + 1;
  for (const Path& p : ps)
    if (p.size() > 1 && !row.count(Path(p.begin(), p.end() - 1))) return MEDUSA_ETEMPLATE;

  const int N = n_paths + 1;
  std::vector<int32_t> depth(N), parent(N), slot(N), nkids(N, 0);
  depth[0] = 0; parent[0] = -1; slot[0] = 0;
  int D = 0;
  for (int u = 1; u < N; ++u) {
    const Path& p = ps[u - 1];
    depth[u] = (int32_t)p.size();
    parent[u] = p.size() == 1 ? 0 : row[Path(p.begin(), p.end() - 1)];
    slot[u] = 1 + ((int32_t)p.size() - 1) * topk + p.back();
    nkids[parent[u]]++;
    D = std::max(D, depth[u]);
  }
  std::vector<int32_t> leaves, internal, internal_index(N, -1);
  for (int u = 0; u < N; ++u) {
    if (nkids[u] == 0) leaves.push_back(u);
    else { internal_index[u] = (int32_t)internal.size(); internal.push_back(u); }
  }
  const int W = (N + 63) / 64;
  const BlobLayout lay = blob_layout(N, D, (int)leaves.size());
  if (lay.total > host_bytes) return MEDUSA_EWORKSPACE;
  char* base = static_cast<char*>(host_buf);
  std::memset(base, 0, lay.total);
  int32_t* o_slot = reinterpret_cast<int32_t*>(base + lay.slot);
  int32_t* o_depth = reinterpret_cast<int32_t*>(base + lay.depth);
  int32_t* o_parent = reinterpret_cast<int32_t*>(base + lay.parent);
  int32_t* o_internal = reinterpret_cast<int32_t*>(base + lay.internal);
  int32_t* o_iidx = reinterpret_cast<int32_t*>(base + lay.internal_index);
  int32_t* o_ret = reinterpret_cast<int32_t*>(base + lay.retrieve);
  uint64_t* o_anc = reinterpret_cast<uint64_t*>(base + lay.anc);
  for (int u = 0; u < N; ++u) {
    o_slot[u] = slot[u];
    o_depth[u] = depth[u];
    o_parent[u] = parent[u];
    o_iidx[u] = internal_index[u];
    // ancestor-or-self bits by walking the parent chain
    for (int v = u; v >= 0; v = parent[v]) o_anc[(size_t)u * W + v / 64] |= (1ull << (v % 64));
  }
  for (size_t i = 0; i < internal.size(); ++i) o_internal[i] = internal[i];
  // retrieval rows: one per leaf (maximal path), in row order, root first, -1 padded
  for (size_t i = 0; i < leaves.size(); ++i) {
    std::vector<int32_t> chain;
    for (int v = leaves[i]; v >= 0; v = parent[v]) chain.push_back(v);
    std::reverse(chain.begin(), chain.end());
    for (int j = 0; j <= D; ++j) o_ret[i * (D + 1) + j] = j < (int)chain.size() ? chain[j] : -1;
  }
  out->n_rows = N;
  out->n_words = W;
  out->max_depth = D;
  out->n_paths = (int32_t)leaves.size();
  out->topk = topk;
  out->n_internal = (int32_t)internal.size();
  out->slot = o_slot;
  out->depth = o_depth;
  out->parent = o_parent;
  out->retrieve = o_ret;
  out->internal = o_internal;
  out->internal_index = o_iidx;
  out->anc = o_anc;
  out->per_seq = nullptr;
  return MEDUSA_OK;
}

namespace {
bool greedy_args_ok(int32_t B, int32_t K, int32_t R, int32_t budget, int32_t topk) {
  return B >= 1 && K >= 1 && K <= MEDUSA_MAX_DEPTH && R >= 1 && topk >= 1 && topk <= MEDUSA_MAX_TOPK && R <= topk &&
         budget >= 0 && budget < MEDUSA_MAX_ROWS;
}
size_t greedy_blob_stride(int32_t K, int32_t budget) {
  return align_up(blob_layout(budget + 1, K, budget > 0 ? budget : 1).total, 256);
}
}  // namespace

size_t medusa_tree_greedy_device_bytes(int32_t B, int32_t K, int32_t R, int32_t budget) {
  if (!greedy_args_ok(B, K, R, budget, MEDUSA_MAX_TOPK)) return 0;
  return (size_t)B * greedy_blob_stride(K, budget);
}

medusa_status medusa_tree_greedy_device(const double* acc, int32_t B, int32_t K, int32_t R, int32_t budget,
                                        int32_t topk, void* dev_buf, size_t dev_bytes, medusa_tree_t* per_seq,
                                        int32_t* status, medusa_tree_t* batch_out, void* stream) {
  if (!acc || !dev_buf || !per_seq || !batch_out || !greedy_args_ok(B, K, R, budget, topk) || !aligned16(dev_buf) ||
      (reinterpret_cast<uintptr_t>(per_seq) & 7u))
    return MEDUSA_EINVAL;
  if ((int64_t)R * (budget + 1) > medusa::kMaxGreedyEntries) return MEDUSA_EUNSUPPORTED;
  const size_t stride = greedy_blob_stride(K, budget);
  if (dev_bytes < (size_t)B * stride) return MEDUSA_EWORKSPACE;
  if (cuda_status(medusa::launch_tree_greedy(acc, B, K, R, budget, topk, dev_buf, stride, per_seq, status,
                                             as_stream(stream))) != MEDUSA_OK)
    return MEDUSA_ECUDA;
  medusa_tree_t bnd{};
  bnd.n_rows = budget + 1;
  bnd.n_words = (bnd.n_rows + 63) / 64;
  bnd.max_depth = std::min<int32_t>(K, budget);
  bnd.n_paths = budget > 0 ? budget : 1;
  bnd.topk = topk;
  bnd.n_internal = budget;
  bnd.per_seq = per_seq;
  *batch_out = bnd;
  return MEDUSA_OK;
}

medusa_status medusa_tree_batch(const medusa_tree_t* seq, int32_t B, void* dev_descs, size_t dev_bytes,
                                medusa_tree_t* out, void* stream) {
  if (!seq || B < 1 || !dev_descs || !out || (reinterpret_cast<uintptr_t>(dev_descs) & 7u)) return MEDUSA_EINVAL;
  if (dev_bytes < (size_t)B * sizeof(medusa_tree_t)) return MEDUSA_EWORKSPACE;
  medusa_tree_t bnd{};
  for (int b = 0; b < B; ++b) {
    const medusa_tree_t& q = seq[b];
    if (!tree_ok(&q) || q.per_seq || q.topk != seq[0].topk) return MEDUSA_EINVAL;
    bnd.n_rows = std::max(bnd.n_rows, q.n_rows);
    bnd.max_depth = std::max(bnd.max_depth, q.max_depth);
    bnd.n_paths = std::max(bnd.n_paths, q.n_paths);
    bnd.n_internal = std::max(bnd.n_internal, q.n_internal);
  }
  bnd.n_words = (bnd.n_rows + 63) / 64;
  bnd.topk = seq[0].topk;
  bnd.per_seq = static_cast<const medusa_tree_t*>(dev_descs);
  if (cudaMemcpyAsync(dev_descs, seq, (size_t)B * sizeof(medusa_tree_t), cudaMemcpyHostToDevice,
                      as_stream(stream)) != cudaSuccess)
    return MEDUSA_ECUDA;
  *out = bnd;
  return MEDUSA_OK;
}

medusa_status medusa_tree_upload(const medusa_tree_t* host_tree, const void* host_buf,
                                 void* dev_buf, size_t dev_bytes, medusa_tree_t* dev, void* stream) {
  if (!tree_ok(host_tree) || host_tree->per_seq || !host_buf || !dev_buf || !dev || !aligned16(dev_buf))
    return MEDUSA_EINVAL;
  const char* hb = static_cast<const char*>(host_buf);
  if (reinterpret_cast<const char*>(host_tree->slot) < hb) return MEDUSA_EINVAL;
  const size_t bytes = blob_end(host_tree, host_buf);
  if (bytes > dev_bytes) return MEDUSA_EWORKSPACE;
  cudaError_t e = cudaMemcpyAsync(dev_buf, host_buf, bytes, cudaMemcpyHostToDevice, as_stream(stream));
  if (e != cudaSuccess) return MEDUSA_ECUDA;
  char* db = static_cast<char*>(dev_buf);
  auto rebase = [&](const void* p) { return db + (static_cast<const char*>(p) - hb); };
  *dev = *host_tree;
  dev->slot = reinterpret_cast<const int32_t*>(rebase(host_tree->slot));
  dev->depth = reinterpret_cast<const int32_t*>(rebase(host_tree->depth));
  dev->parent = reinterpret_cast<const int32_t*>(rebase(host_tree->parent));
  dev->retrieve = reinterpret_cast<const int32_t*>(rebase(host_tree->retrieve));
  dev->internal = reinterpret_cast<const int32_t*>(rebase(host_tree->internal));
  dev->internal_index = reinterpret_cast<const int32_t*>(rebase(host_tree->internal_index));
  dev->anc = reinterpret_cast<const uint64_t*>(rebase(host_tree->anc));
  return MEDUSA_OK;
}

size_t medusa_heads_topk_workspace(int32_t T, int32_t d, int32_t V, int32_t K, int32_t topk) {
  if (T < 1 || d < 1 || V < 1 || K < 0 || topk < 1) return 0;
  return medusa::plan_heads(T, d, V, K, topk).bytes;
}

medusa_status medusa_heads_topk(const void* h, int32_t T, int32_t d, int32_t V, int32_t K,
                                const void* w1, const void* b1, const void* w2,
                                int64_t w2_head_stride, const void* w_lm, int32_t topk,
                                medusa_dtype dt, int32_t* root, int32_t* pool,
                                float* logits_out, void* ws, size_t ws_bytes, void* stream) {
  if (!h || !w_lm || !root || !ws || !dtype_ok(dt) || T < 1 || T > MEDUSA_MAX_HEAD_ROWS || d < 8 || d % 8 != 0 ||
      V < 1 || K < 0 || K > MEDUSA_MAX_DEPTH || topk < 1 || topk > MEDUSA_MAX_TOPK || topk > V ||
      w2_head_stride < 0)
    return MEDUSA_EINVAL;
  if (K > 0 && (!w1 || !w2 || !pool)) return MEDUSA_EINVAL;
  if (!aligned16(h) || !aligned16(w_lm) || (K > 0 && (!aligned16(w1) || !aligned16(w2))))
    return MEDUSA_EINVAL;
  const size_t esz = dt == MEDUSA_BF16 ? 2 : 4;
  if (((size_t)w2_head_stride * esz) % 16 != 0) return MEDUSA_EINVAL;
  const medusa::HeadsPlan p = medusa::plan_heads(T, d, V, K, topk);
  if (ws_bytes < p.bytes) return MEDUSA_EWORKSPACE;
  return cuda_status(medusa::launch_heads(p, h, w1, b1, w2, w2_head_stride, w_lm, dt, root, pool,
                                          logits_out, ws, as_stream(stream)));
}

medusa_status medusa_tree_fill(const medusa_tree_t* t, int32_t B, int32_t K, const int32_t* root,
                               const int32_t* pool, const int32_t* L, int32_t* tokens,
                               int32_t* pos, void* stream) {
  if (!tree_ok(t) || B < 1 || K < t->max_depth || !root || (t->n_rows > 1 && !pool) || !L ||
      !tokens || !pos)
    return MEDUSA_EINVAL;
  return cuda_status(medusa::launch_tree_fill(*t, B, K, root, pool, L, tokens, pos, as_stream(stream)));
}

size_t medusa_tree_attn_workspace(const medusa_tree_t* t, int32_t B, int32_t n_q_heads,
                                  const medusa_kv_t* cache, int32_t max_prefix) {
  if (!tree_ok(t) || !kv_ok(cache) || B < 1 || n_q_heads < 1 || n_q_heads % cache->n_kv_heads ||
      max_prefix < 0)
    return 0;
  return medusa::plan_attn(*t, B, n_q_heads, *cache, max_prefix).bytes;
}

medusa_status medusa_tree_attn_verify(const medusa_tree_t* t, int32_t B, int32_t n_q_heads,
                                      const void* q, const void* k_new, const void* v_new,
                                      const medusa_kv_t* cache, const int32_t* L,
                                      int32_t max_prefix, float rope_base, float scale,
                                      float* out, float* lse, int32_t* status, void* ws,
                                      size_t ws_bytes, void* stream) {
  if (!tree_ok(t) || !kv_ok(cache) || B < 1 || n_q_heads < 1 || n_q_heads % cache->n_kv_heads ||
      !q || !k_new || !v_new || !L || !out || !status || !ws || max_prefix < 0 ||
      !(rope_base > 1.0f) || !(scale > 0.0f) || !std::isfinite(scale))
    return MEDUSA_EINVAL;
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(out)) return MEDUSA_EINVAL;
  if ((int64_t)max_prefix + t->n_rows > cache->capacity) return MEDUSA_ECAPACITY;
  const medusa::AttnPlan p = medusa::plan_attn(*t, B, n_q_heads, *cache, max_prefix);
  if (medusa::attn_units(p) > medusa::kAttnMaxUnits) return MEDUSA_EUNSUPPORTED;
  if (ws_bytes < p.bytes) return MEDUSA_EWORKSPACE;
  return cuda_status(medusa::launch_attn(p, *t, q, k_new, v_new, *cache, L, rope_base, scale, out,
                                         lse, status, ws, as_stream(stream)));
}

// Same computation as medusa_tree_attn_verify, with the scratch taken from a fixed
// device array instead of a caller workspace, for callers that cannot allocate.
medusa_status medusa_tree_attn_verify_static(const medusa_tree_t* t, int32_t B, int32_t n_q_heads,
                                             const void* q, const void* k_new, const void* v_new,
                                             const medusa_kv_t* cache, const int32_t* L,
                                             int32_t max_prefix, float rope_base, float scale,
                                             float* out, float* lse, int32_t* status, void* stream) {
  if (!tree_ok(t) || !kv_ok(cache) || B < 1 || n_q_heads < 1 || n_q_heads % cache->n_kv_heads ||
      !q || !k_new || !v_new || !L || !out || !status || max_prefix < 0 ||
      !(rope_base > 1.0f) || !(scale > 0.0f) || !std::isfinite(scale))
    return MEDUSA_EINVAL;
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(out)) return MEDUSA_EINVAL;
  if ((int64_t)max_prefix + t->n_rows > cache->capacity) return MEDUSA_ECAPACITY;
  const medusa::AttnPlan p = medusa::plan_attn(*t, B, n_q_heads, *cache, max_prefix);
  if (medusa::attn_units(p) > medusa::kAttnMaxUnits) return MEDUSA_EUNSUPPORTED;
  if (p.bytes > (size_t)MEDUSA_ATTN_STATIC_SCRATCH_BYTES) return MEDUSA_EWORKSPACE;
  void* ws = nullptr;
  if (medusa::attn_static_scratch(&ws) != cudaSuccess) return MEDUSA_ECUDA;
  // the array keeps the previous call's contents: zero the counters this call uses
  const size_t counters = medusa::attn_units(p) * sizeof(int);
  if (cudaMemsetAsync(static_cast<char*>(ws) + p.off_counter, 0, counters, as_stream(stream)) != cudaSuccess)
    return MEDUSA_ECUDA;
  return cuda_status(medusa::launch_attn(p, *t, q, k_new, v_new, *cache, L, rope_base, scale, out,
                                         lse, status, ws, as_stream(stream)));
}

size_t medusa_tree_accept_workspace(const medusa_tree_t* t, int32_t B, int32_t V) {
  if (!tree_ok(t) || B < 1 || V < 1) return 0;
  return medusa::plan_accept(*t, B, V).bytes;
}

medusa_status medusa_tree_accept(const medusa_tree_t* t, int32_t B, int32_t V, const void* logits,
                                 medusa_dtype dt, const int32_t* tokens, int32_t mode,
                                 float temperature, float epsilon, float delta,
                                 int32_t entropy_guard, int32_t* best_path, int32_t* accept_len,
                                 int32_t* out_tokens, int32_t* out_rows, int32_t* frontier_row,
                                 void* ws, size_t ws_bytes, void* stream) {
  return accept_logits_impl(t, B, V, logits, dt, tokens, mode, temperature, epsilon, delta, entropy_guard,
                            best_path, accept_len, out_tokens, out_rows, frontier_row, ws, ws_bytes, stream,
                            medusa::CommitArgs{});
}

size_t medusa_tree_accept_hidden_workspace(const medusa_tree_t* t, int32_t B, int32_t V, int32_t d) {
  if (!tree_ok(t) || B < 1 || V < 1 || d < 1) return 0;
  return medusa::plan_lm_accept(*t, B, V, d).bytes;
}

}  // extern "C"

namespace {

bool commit_ok(const medusa_kv_t* cache, const int32_t* L, const int32_t* L_out, const int32_t* status) {
  return kv_ok(cache) && L && L_out && status && L_out != L;
}

medusa_status accept_hidden_impl(const medusa_tree_t* t, int32_t B, int32_t V, int32_t d, const void* hidden,
                                 const void* w_lm, const int32_t* tokens, int32_t mode, float temperature,
                                 float epsilon, float delta, int32_t* best_path, int32_t* accept_len,
                                 int32_t* out_tokens, int32_t* out_rows, int32_t* frontier_row, void* ws,
                                 size_t ws_bytes, void* stream, const medusa::CommitArgs& cm) {
  if (!tree_ok(t) || B < 1 || V < 1 || d < 1 || !hidden || !w_lm || !tokens || !best_path || !accept_len ||
      !out_tokens || !out_rows || !frontier_row || !ws ||
      (mode != MEDUSA_ACCEPT_GREEDY && mode != MEDUSA_ACCEPT_TYPICAL) || !(temperature > 0.0f) ||
      !std::isfinite(temperature) || !(epsilon >= 0.0f) || !(delta >= 0.0f))
    return MEDUSA_EINVAL;
  if (!aligned16(hidden) || !aligned16(w_lm) || !aligned16(ws)) return MEDUSA_EINVAL;
  if (!medusa::lm_accept_supported(d, V)) return MEDUSA_EUNSUPPORTED;
  const medusa::LmAcceptPlan p = medusa::plan_lm_accept(*t, B, V, d);
  if (ws_bytes < p.bytes) return MEDUSA_EWORKSPACE;
  return cuda_status(medusa::launch_lm_accept(p, *t, hidden, w_lm, tokens, mode, temperature, epsilon, delta,
                                              best_path, accept_len, out_tokens, out_rows, frontier_row, ws,
                                              as_stream(stream), cm));
}

medusa_status accept_logits_impl(const medusa_tree_t* t, int32_t B, int32_t V, const void* logits, medusa_dtype dt,
                                 const int32_t* tokens, int32_t mode, float temperature, float epsilon,
                                 float delta, int32_t entropy_guard, int32_t* best_path, int32_t* accept_len,
                                 int32_t* out_tokens, int32_t* out_rows, int32_t* frontier_row, void* ws,
                                 size_t ws_bytes, void* stream, const medusa::CommitArgs& cm) {
  if (!tree_ok(t) || B < 1 || V < 1 || !logits || !dtype_ok(dt) || !tokens || !best_path ||
      !accept_len || !out_tokens || !out_rows || !frontier_row || !ws ||
      (mode != MEDUSA_ACCEPT_GREEDY && mode != MEDUSA_ACCEPT_TYPICAL) || !(temperature > 0.0f) ||
      !std::isfinite(temperature) || !(epsilon >= 0.0f) || !(delta >= 0.0f))
    return MEDUSA_EINVAL;
  const medusa::AcceptPlan p = medusa::plan_accept(*t, B, V);
  if (ws_bytes < p.bytes) return MEDUSA_EWORKSPACE;
  return cuda_status(medusa::launch_accept(p, *t, logits, dt, tokens, mode, temperature, epsilon,
                                           delta, entropy_guard, best_path, accept_len, out_tokens,
                                           out_rows, frontier_row, ws, as_stream(stream), cm));
}

medusa::CommitArgs commit_args(const medusa_kv_t* cache, const int32_t* L, int32_t* L_out, int32_t* status) {
  medusa::CommitArgs cm{};
  cm.c = *cache;
  cm.on = 1;
  cm.L = L;
  cm.L_out = L_out;
  cm.status = status;
  return cm;
}

}  // namespace

extern "C" {

medusa_status medusa_tree_accept_hidden(const medusa_tree_t* t, int32_t B, int32_t V, int32_t d,
                                        const void* hidden, const void* w_lm, const int32_t* tokens, int32_t mode,
                                        float temperature, float epsilon, float delta, int32_t* best_path,
                                        int32_t* accept_len, int32_t* out_tokens, int32_t* out_rows,
                                        int32_t* frontier_row, void* ws, size_t ws_bytes, void* stream) {
  return accept_hidden_impl(t, B, V, d, hidden, w_lm, tokens, mode, temperature, epsilon, delta, best_path,
                            accept_len, out_tokens, out_rows, frontier_row, ws, ws_bytes, stream,
                            medusa::CommitArgs{});
}

medusa_status medusa_tree_accept_commit(const medusa_tree_t* t, int32_t B, int32_t V, const void* logits,
                                        medusa_dtype dt, const int32_t* tokens, int32_t mode, float temperature,
                                        float epsilon, float delta, int32_t entropy_guard,
                                        const medusa_kv_t* cache, const int32_t* L, int32_t* best_path,
                                        int32_t* accept_len, int32_t* out_tokens, int32_t* out_rows,
                                        int32_t* frontier_row, int32_t* L_out, int32_t* status, void* ws,
                                        size_t ws_bytes, void* stream) {
  if (!commit_ok(cache, L, L_out, status)) return MEDUSA_EINVAL;
  return accept_logits_impl(t, B, V, logits, dt, tokens, mode, temperature, epsilon, delta, entropy_guard,
                            best_path, accept_len, out_tokens, out_rows, frontier_row, ws, ws_bytes, stream,
                            commit_args(cache, L, L_out, status));
}

medusa_status medusa_kv_compact(const medusa_kv_t* cache, const medusa_tree_t* t, int32_t B,
                                const int32_t* L, const int32_t* accept_len,
                                const int32_t* out_rows, int32_t* L_out, int32_t* status,
                                void* stream) {
  if (!kv_ok(cache) || !tree_ok(t) || B < 1 || !L || !accept_len || !out_rows || !L_out || !status || L_out == L)
    return MEDUSA_EINVAL;
  return cuda_status(medusa::launch_kv_compact(*cache, *t, B, L, accept_len, out_rows, L_out, status,
                                               as_stream(stream)));
}

medusa_status medusa_kv_compact_layers(const medusa_kv_t* caches, int32_t n_layers, const medusa_tree_t* t,
                                       int32_t B, const int32_t* L, const int32_t* accept_len,
                                       const int32_t* out_rows, int32_t* L_out, int32_t* status,
                                       void* stream) {
  if (!caches || n_layers < 1 || n_layers > MEDUSA_MAX_LAYERS || !tree_ok(t) || B < 1 || !L || !accept_len ||
      !out_rows || !L_out || !status || L_out == L)
    return MEDUSA_EINVAL;
  const medusa_kv_t& c0 = caches[0];
  for (int32_t i = 0; i < n_layers; ++i) {
    const medusa_kv_t& c = caches[i];
    if (!kv_ok(&c)) return MEDUSA_EINVAL;
    // every layer shares the layout: one row offset serves them all
    if (c.dtype != c0.dtype || c.n_kv_heads != c0.n_kv_heads || c.head_dim != c0.head_dim ||
        c.capacity != c0.capacity || c.page_size != c0.page_size || c.block_table != c0.block_table ||
        c.max_blocks != c0.max_blocks || c.n_pages != c0.n_pages || (c.k_f16 == nullptr) != (c0.k_f16 == nullptr))
      return MEDUSA_EINVAL;
  }
  return cuda_status(medusa::launch_kv_compact_layers(caches, n_layers, *t, B, L, accept_len, out_rows, L_out,
                                                      status, as_stream(stream)));
}

medusa_status medusa_kv_mirror_sync(const medusa_kv_t* cache, int32_t B, void* stream) {
  if (!kv_ok(cache) || !cache->k_f16 || cache->dtype != MEDUSA_BF16) return MEDUSA_EINVAL;
  if (cache->page_size == 0 && B < 1) return MEDUSA_EINVAL;
  const int64_t rows = cache->page_size == 0 ? (int64_t)B * cache->capacity
                                             : (int64_t)cache->n_pages * cache->page_size;
  return cuda_status(medusa::launch_kv_mirror_sync(*cache, rows * cache->n_kv_heads * cache->head_dim,
                                                   as_stream(stream)));
}

// ---- whole round as one CUDA graph ------------------------------------------------

struct medusa_round_s {
  cudaGraph_t graph;
  cudaGraphExec_t exec;
};

namespace {

// Offsets of the three workspaces inside a round's workspace (256-byte aligned).
struct RoundWs {
  size_t attn, accept, total;
};

bool round_ws(const medusa_round_desc* r, RoundWs& w) {
  if (!r || !tree_ok(&r->tree) || !kv_ok(&r->cache) || r->B < 1) return false;
  const size_t h = medusa_heads_topk_workspace(r->B, r->d, r->V, r->K, r->topk);
  const size_t a = medusa_tree_attn_workspace(&r->tree, r->B, r->n_q_heads, &r->cache, r->max_prefix);
  const size_t c = r->hidden_target ? medusa_tree_accept_hidden_workspace(&r->tree, r->B, r->V, r->d)
                                    : medusa_tree_accept_workspace(&r->tree, r->B, r->V);
  if (h == 0 || a == 0 || c == 0) return false;
  w.attn = align_up(h, 256);
  w.accept = w.attn + align_up(a, 256);
  w.total = w.accept + align_up(c, 256);
  return true;
}

// The five calls in round order on `st`; the first failing status is returned.
medusa_status record_round(const medusa_round_desc* r, char* ws, const RoundWs& w, void* st) {
  medusa_status s = medusa_heads_topk(r->h, r->B, r->d, r->V, r->K, r->w1, r->b1, r->w2, r->w2_head_stride,
                                      r->w_lm, r->topk, r->dtype, r->root, r->pool, nullptr, ws, w.attn, st);
  if (s != MEDUSA_OK) return s;
  s = medusa_tree_fill(&r->tree, r->B, r->K, r->root, r->pool, r->L, r->tokens, r->pos, st);
  if (s != MEDUSA_OK) return s;
  s = medusa_tree_attn_verify(&r->tree, r->B, r->n_q_heads, r->q, r->k_new, r->v_new, &r->cache, r->L,
                              r->max_prefix, r->rope_base, r->scale, r->out, r->lse, r->attn_status,
                              ws + w.attn, w.accept - w.attn, st);
  if (s != MEDUSA_OK) return s;
  // steps 4 and 5: acceptance, then compaction, or both in one (the fused commit)
  medusa::CommitArgs cm{};
  if (r->fuse_commit) {
    if (!commit_ok(&r->cache, r->L, r->L_out, r->compact_status)) return MEDUSA_EINVAL;
    cm = commit_args(&r->cache, r->L, r->L_out, r->compact_status);
  }
  if (r->hidden_target)
    s = accept_hidden_impl(&r->tree, r->B, r->V, r->d, r->hidden_target, r->w_lm, r->tokens, r->mode,
                           r->temperature, r->epsilon, r->delta, r->best_path, r->accept_len, r->out_tokens,
                           r->out_rows, r->frontier_row, ws + w.accept, w.total - w.accept, st, cm);
  else
    s = accept_logits_impl(&r->tree, r->B, r->V, r->logits, r->dtype, r->tokens, r->mode, r->temperature,
                           r->epsilon, r->delta, r->entropy_guard, r->best_path, r->accept_len, r->out_tokens,
                           r->out_rows, r->frontier_row, ws + w.accept, w.total - w.accept, st, cm);
  if (s != MEDUSA_OK || r->fuse_commit) return s;
  return medusa_kv_compact(&r->cache, &r->tree, r->B, r->L, r->accept_len, r->out_rows, r->L_out,
                           r->compact_status, st);
}

}  // namespace

size_t medusa_round_workspace(const medusa_round_desc* r) {
  RoundWs w;
  return round_ws(r, w) ? w.total : 0;
}

medusa_status medusa_round_create(const medusa_round_desc* r, void* ws, size_t ws_bytes, void* stream,
                                  medusa_round_t* round_out) {
  if (!round_out) return MEDUSA_EINVAL;
  *round_out = nullptr;
  RoundWs w;
  if (!round_ws(r, w) || !ws || !aligned16(ws)) return MEDUSA_EINVAL;
  if (ws_bytes < w.total) return MEDUSA_EWORKSPACE;
  const cudaStream_t user = as_stream(stream);
  if (cudaMemsetAsync(ws, 0, w.total, user) != cudaSuccess || cudaStreamSynchronize(user) != cudaSuccess)
    return MEDUSA_ECUDA;
  // Record on a private stream: capture needs a stream other than the legacy default,
  // and thread-local mode leaves other threads' CUDA calls alone meanwhile.
  cudaStream_t cs = nullptr;
  if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) return MEDUSA_ECUDA;
  medusa_status s = MEDUSA_OK;
  cudaGraph_t g = nullptr;
  if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    s = MEDUSA_ECUDA;
  } else {
    s = record_round(r, static_cast<char*>(ws), w, cs);
    const cudaError_t e = cudaStreamEndCapture(cs, &g);   // ends the capture on every path
    if (s == MEDUSA_OK && e != cudaSuccess) s = MEDUSA_ECUDA;
  }
  cudaGraphExec_t ex = nullptr;
  if (s == MEDUSA_OK && cudaGraphInstantiate(&ex, g, 0) != cudaSuccess) s = MEDUSA_ECUDA;
  medusa_round_s* rr = nullptr;
  if (s == MEDUSA_OK) {
    rr = new (std::nothrow) medusa_round_s{g, ex};
    if (!rr) s = MEDUSA_ECUDA;
  }
  cudaStreamDestroy(cs);
  if (s != MEDUSA_OK) {
    if (ex) cudaGraphExecDestroy(ex);
    if (g) cudaGraphDestroy(g);
    cudaGetLastError();              // leave no sticky error behind a failed creation
    return s;
  }
  *round_out = rr;
  return MEDUSA_OK;
}

medusa_status medusa_round_launch(medusa_round_t round, void* stream) {
  if (!round) return MEDUSA_EINVAL;
  return cuda_status(cudaGraphLaunch(round->exec, as_stream(stream)));
}

medusa_status medusa_round_destroy(medusa_round_t round) {
  if (!round) return MEDUSA_EINVAL;
  const cudaError_t a = cudaGraphExecDestroy(round->exec);
  const cudaError_t b = cudaGraphDestroy(round->graph);
  delete round;
  return (a == cudaSuccess && b == cudaSuccess) ? MEDUSA_OK : MEDUSA_ECUDA;
}

}  // extern "C"
