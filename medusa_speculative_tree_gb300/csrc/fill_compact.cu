// Tree fill ([M7.2] §0x01B, §0x04A) and winning-path K/V compaction
// ([M7.2] §0x06A-§0x06B).  Both are small integer / data-movement kernels.
#include <vector>

#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"

namespace medusa {

namespace {

// tokens[b][u] = cand_b[slot[u]], cand_b = [root[b], pool[b][0][:], pool[b][1][:], ...]
// pos[b][u]    = L[b] + depth[u]
// With per-sequence templates the rows of sequence b are those of its own template;
// the rows past them (up to the batch bound, the row stride) get -1.
__global__ void tree_fill_kernel(medusa_tree_t t, int K, const int32_t* __restrict__ root,
                                 const int32_t* __restrict__ pool, const int32_t* __restrict__ L,
                                 int32_t* __restrict__ tokens, int32_t* __restrict__ pos) {
  const int b = blockIdx.y;
  const int u = blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= t.n_rows) return;
  const medusa_tree_t tb = seq_tree(t, b);
  int tok = -1, p = -1;
  if (u < tb.n_rows) {
    const int s = tb.slot[u];
    if (s == 0) {
      tok = root[b];
    } else {
      const int head = (s - 1) / tb.topk, rank = (s - 1) % tb.topk;
      tok = (head < K && rank < t.topk) ? pool[((int64_t)b * K + head) * t.topk + rank] : -1;
    }
    p = L[b] + tb.depth[u];
  }
  tokens[(int64_t)b * t.n_rows + u] = tok;
  pos[(int64_t)b * t.n_rows + u] = p;
}

// K and V base pointers of the layers that one launch commits ([M7.2] §0x06B: the
// accepted rows are committed in every layer's cache); blockIdx.z picks the layer.
// The other fields of the cache descriptor are common to all of them.
template <int NL>
struct LayerPtrs {
  void* k[NL];
  void* v[NL];
};

// One CTA per (kv head, sequence, layer).  The whole path is validated first (lane j
// of warp 0 checks row j: 0 for the root, else a child of row j - 1); the G source
// rows of K and V are then read into shared memory before any destination row is
// written, so overlapping source/destination rows are safe.  Rows move as 16-byte
// vectors when their length allows.  status and L_out are written once per sequence
// (kv head 0 of layer 0, in the launch that has write_meta set).
template <typename EL, int NL>
__global__ void kv_compact_kernel(medusa_kv_t c, LayerPtrs<NL> lp, int write_meta, medusa_tree_t t,
                                  const int32_t* __restrict__ L, const int32_t* __restrict__ accept_len,
                                  const int32_t* __restrict__ out_rows, int32_t* __restrict__ L_out,
                                  int32_t* __restrict__ status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  EL* snap = reinterpret_cast<EL*>(smem_raw);       // [2][D+1][dh]
  __shared__ int rows_s[MEDUSA_MAX_DEPTH + 1];
  __shared__ int seq_status;
  const int kvh = blockIdx.x, b = blockIdx.y, layer = blockIdx.z;
  const bool meta = write_meta && kvh == 0 && layer == 0 && threadIdx.x == 0;
  const int dh = c.head_dim, W = t.max_depth + 1;             // row stride of out_rows
  const medusa_tree_t tb = seq_tree(t, b);                     // this sequence's template
  const int Lb = L[b];
  const int a = accept_len[b];
  if (threadIdx.x < 32) {
    const int j = threadIdx.x;
    const int u = j < W ? out_rows[(int64_t)b * W + j] : -1;
    const int prev = (j >= 1 && j < W) ? out_rows[(int64_t)b * W + j - 1] : -1;
    const bool in = a >= 0 && a <= tb.max_depth && j <= a;
    bool bad = false;
    if (in) {
      rows_s[j] = u;
      if (u < 0 || u >= tb.n_rows) bad = true;
      else if (j == 0) bad = u != 0;
      else bad = tb.parent[u] != prev;
    }
    const bool any_bad = __any_sync(0xffffffffu, bad);
    if (j == 0) {
      int v = MEDUSA_OK;
      if (Lb < 0 || !seq_rows_ok(c, b, (int64_t)Lb + tb.n_rows)) v = MEDUSA_ECAPACITY;
      else if (a < 0 || a > tb.max_depth || any_bad) v = MEDUSA_EPATH;
      seq_status = v;
    }
  }
  __syncthreads();
  const int v = seq_status;
  if (v != MEDUSA_OK) {
    if (meta) {
      status[b] = v;
      L_out[b] = Lb;
    }
    return;
  }
  const int G = a + 1;
  EL* ck = (EL*)lp.k[layer];
  EL* cv = (EL*)lp.v[layer];
  if ((dh * (int)sizeof(EL)) % 16 == 0) {
    const int pr = dh * (int)sizeof(EL) / 16;           // 16-byte pieces per row
    uint4* s4 = reinterpret_cast<uint4*>(snap);
    for (int idx = threadIdx.x; idx < G * pr; idx += blockDim.x) {
      const int j = idx / pr, e = idx % pr;
      const int64_t src = cache_row_offset(c, b, kvh, Lb + rows_s[j]);
      s4[j * pr + e] = reinterpret_cast<const uint4*>(ck + src)[e];
      s4[(W + j) * pr + e] = reinterpret_cast<const uint4*>(cv + src)[e];
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < G * pr; idx += blockDim.x) {
      const int j = idx / pr, e = idx % pr;
      const int64_t dst = cache_row_offset(c, b, kvh, Lb + j);
      reinterpret_cast<uint4*>(ck + dst)[e] = s4[j * pr + e];
      reinterpret_cast<uint4*>(cv + dst)[e] = s4[(W + j) * pr + e];
    }
  } else {
    for (int idx = threadIdx.x; idx < G * dh; idx += blockDim.x) {
      const int j = idx / dh, e = idx % dh;
      const int64_t src = cache_row_offset(c, b, kvh, Lb + rows_s[j]) + e;
      snap[j * dh + e] = ck[src];
      snap[(W + j) * dh + e] = cv[src];
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < G * dh; idx += blockDim.x) {
      const int j = idx / dh, e = idx % dh;
      const int64_t dst = cache_row_offset(c, b, kvh, Lb + j) + e;
      ck[dst] = snap[j * dh + e];
      cv[dst] = snap[(W + j) * dh + e];
    }
  }
  if (meta) {
    status[b] = MEDUSA_OK;
    L_out[b] = Lb + G;
  }
}

}  // namespace

cudaError_t launch_tree_fill(const medusa_tree_t& t, int B, int K, const int32_t* root,
                             const int32_t* pool, const int32_t* L, int32_t* tokens,
                             int32_t* pos, cudaStream_t st) {
  const int threads = 128;
  dim3 grid((t.n_rows + threads - 1) / threads, B);
  tree_fill_kernel<<<grid, threads, 0, st>>>(t, K, root, pool, L, tokens, pos);
  return cudaGetLastError();
}

namespace {

// One launch over n caches' (K, V) pointer pairs that share c's layout; the pair at
// z = 0 writes status and L_out when meta is set.
template <int NL>
cudaError_t compact_launch(const medusa_kv_t& c, void* const* ks, void* const* vs, int n, int meta,
                           const medusa_tree_t& t, int B, const int32_t* L, const int32_t* accept_len,
                           const int32_t* out_rows, int32_t* L_out, int32_t* status, cudaStream_t st) {
  const size_t esz = c.dtype == MEDUSA_BF16 ? 2 : 4;
  const size_t smem = 2 * (size_t)(t.max_depth + 1) * c.head_dim * esz;
  LayerPtrs<NL> lp = {};
  for (int i = 0; i < n; ++i) {
    lp.k[i] = ks[i];
    lp.v[i] = vs[i];
  }
  dim3 grid(c.n_kv_heads, B, n);
  if (c.dtype == MEDUSA_BF16)
    kv_compact_kernel<uint16_t, NL><<<grid, 128, smem, st>>>(c, lp, meta, t, L, accept_len, out_rows, L_out, status);
  else
    kv_compact_kernel<float, NL><<<grid, 128, smem, st>>>(c, lp, meta, t, L, accept_len, out_rows, L_out, status);
  return cudaGetLastError();
}

// bf16 -> fp16, eight elements per 16-byte vector (bf16 -> fp32 exactly, then one
// rounding to fp16)
__global__ void kv_mirror_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v, uint4* __restrict__ k16,
                                 uint4* __restrict__ v16, int64_t n_vec) {
  auto conv = [](uint32_t w) {
    const __half2 h = __floats2half2_rn(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
    return *reinterpret_cast<const uint32_t*>(&h);
  };
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n_vec; i += (int64_t)gridDim.x * blockDim.x) {
    const uint4 a = k[i], b = v[i];
    k16[i] = make_uint4(conv(a.x), conv(a.y), conv(a.z), conv(a.w));
    v16[i] = make_uint4(conv(b.x), conv(b.y), conv(b.z), conv(b.w));
  }
}

}  // namespace

// The caches' writes reach their fp16 mirrors too: a mirror is one more (K, V) pair of
// the same layout and element size, whose rows move as raw bits with the cache's.
cudaError_t launch_kv_compact(const medusa_kv_t& c, const medusa_tree_t& t, int B,
                              const int32_t* L, const int32_t* accept_len,
                              const int32_t* out_rows, int32_t* L_out, int32_t* status,
                              cudaStream_t st) {
  void* ks[2] = {c.k, c.k_f16};
  void* vs[2] = {c.v, c.v_f16};
  if (c.k_f16) return compact_launch<2>(c, ks, vs, 2, 1, t, B, L, accept_len, out_rows, L_out, status, st);
  return compact_launch<1>(c, ks, vs, 1, 1, t, B, L, accept_len, out_rows, L_out, status, st);
}

cudaError_t launch_kv_compact_layers(const medusa_kv_t* layers, int n_layers, const medusa_tree_t& t, int B,
                                     const int32_t* L, const int32_t* accept_len, const int32_t* out_rows,
                                     int32_t* L_out, int32_t* status, cudaStream_t st) {
  std::vector<void*> ks, vs;                 // every layer's cache, then its mirror if any
  ks.reserve(2 * (size_t)n_layers);
  vs.reserve(2 * (size_t)n_layers);
  for (int i = 0; i < n_layers; ++i) {
    ks.push_back(layers[i].k);
    vs.push_back(layers[i].v);
    if (layers[i].k_f16) {
      ks.push_back(layers[i].k_f16);
      vs.push_back(layers[i].v_f16);
    }
  }
  const int total = (int)ks.size();
  for (int l0 = 0; l0 < total; l0 += kCompactLayersPerLaunch) {
    const int n = total - l0 < kCompactLayersPerLaunch ? total - l0 : kCompactLayersPerLaunch;
    const cudaError_t e = compact_launch<kCompactLayersPerLaunch>(layers[0], ks.data() + l0, vs.data() + l0, n,
                                                                  l0 == 0 ? 1 : 0, t, B, L, accept_len, out_rows,
                                                                  L_out, status, st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_kv_mirror_sync(const medusa_kv_t& c, int64_t n, cudaStream_t st) {
  const int64_t n_vec = n / 8;                 // head_dim is 64 or 128: whole vectors
  int sms = 148, dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t blocks = (n_vec + 255) / 256;
  if (blocks > 8 * (int64_t)sms) blocks = 8 * (int64_t)sms;
  if (blocks < 1) blocks = 1;
  kv_mirror_kernel<<<(unsigned)blocks, 256, 0, st>>>((const uint4*)c.k, (const uint4*)c.v, (uint4*)c.k_f16,
                                                     (uint4*)c.v_f16, n_vec);
  return cudaGetLastError();
}

}  // namespace medusa
