// Greedy tree templates built on the GPU, one per sequence ([M7.2] §0x04C, [PartII] Part 3
// "grow a prefix-closed tree under a budget"; [CN] "局限与适用场景": the best node count moves
// with the context length, so a serving loop rebuilds trees from per-context rank accuracies).
//
// One CTA per sequence runs the frontier search and then compiles the chosen paths into
// the template arrays of medusa_tree_compile, in the same layout and canonical order:
//   search   every entry is a path with its weight w = prod_j acc[j][r_j] (multiplied
//            left to right in double, so that it is the same double as on the host);
//            the frontier starts with the R depth-1 paths; each step a block reduction
//            picks the frontier entry that ranks first (larger weight; weights within
//            1e-12 relative tie, then the shorter path, then the lexicographically
//            smaller one), marks it chosen and appends its R children (if shorter than
//            K).  Entries live in shared memory: a path is packed one rank per byte,
//            level 0 in the top byte, so that comparing (hi, lo) compares the paths;
//   compile  rows = 1 + rank of each chosen path in (length, path) order; depth, slot
//            (1 + (t - 1) TOPK + r_t), parent, internal rows and their index (a block
//            scan of child counts), retrieval rows (one per leaf, in row order, root
//            first, -1 padded) and the ancestor-or-self bitmask by walking parents.
#include <float.h>

#include "common.cuh"
#include "kernels.h"

namespace medusa {

namespace {

constexpr int kBThreads = 512;

struct BuildArgs {
  const double* acc;          // [B][K][R]
  int K, R, budget, topk;
  char* blobs;                // [B] blobs of blob_stride bytes
  size_t blob_stride;
  TreeBlobLayout lay;         // array offsets inside a blob (bounds: budget + 1 rows)
  medusa_tree_t* per_seq;     // [B] out
  int32_t* status;            // [B] out, or null
};

struct Ent {                  // (for the reductions)
  double w;
  uint64_t hi, lo;
  int len, idx;
};

__device__ __forceinline__ bool ent_before(const Ent& a, const Ent& b) {
  if (a.idx < 0) return false;
  if (b.idx < 0) return true;
  const double big = fmax(a.w, b.w);
  if (fabs(a.w - b.w) <= 1e-12 * big) {
    if (a.len != b.len) return a.len < b.len;
    return a.hi < b.hi || (a.hi == b.hi && a.lo < b.lo);
  }
  return a.w > b.w;
}

__device__ __forceinline__ Ent shfl_ent(const Ent& e, int o) {
  Ent r;
  r.w = __shfl_xor_sync(0xffffffffu, e.w, o);
  r.hi = __shfl_xor_sync(0xffffffffu, e.hi, o);
  r.lo = __shfl_xor_sync(0xffffffffu, e.lo, o);
  r.len = __shfl_xor_sync(0xffffffffu, e.len, o);
  r.idx = __shfl_xor_sync(0xffffffffu, e.idx, o);
  return r;
}

// Rank r at level j of a packed path: byte 7 - j of hi (j < 8) or of lo (j >= 8).
__device__ __forceinline__ void put_rank(uint64_t& hi, uint64_t& lo, int j, int r) {
  if (j < 8) hi |= (uint64_t)r << (8 * (7 - j));
  else lo |= (uint64_t)r << (8 * (15 - j));
}
__device__ __forceinline__ int get_rank(uint64_t hi, uint64_t lo, int j) {
  return (int)((j < 8 ? hi >> (8 * (7 - j)) : lo >> (8 * (15 - j))) & 0xFFu);
}

__global__ void __launch_bounds__(kBThreads) tree_greedy_kernel(BuildArgs a) {
  extern __shared__ __align__(16) unsigned char smem_b[];
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = a.K, R = a.R, E = R * (a.budget + 1);
  double* e_w = reinterpret_cast<double*>(smem_b);
  uint64_t* e_hi = reinterpret_cast<uint64_t*>(e_w + E);
  uint64_t* e_lo = e_hi + E;
  int16_t* e_par = reinterpret_cast<int16_t*>(e_lo + E);
  int16_t* e_row = e_par + E;                          // row of a chosen entry
  uint8_t* e_len = reinterpret_cast<uint8_t*>(e_row + E);
  uint8_t* e_state = e_len + E;                        // 0 frontier, 1 chosen
  __shared__ Ent red[kBThreads / 32];
  __shared__ int s_n, s_best, s_bad, s_chosen, s_D, s_ni, s_nl;
  __shared__ int s_scan[kBThreads / 32];

  const double* acc = a.acc + (size_t)b * K * R;
  char* blob = a.blobs + (size_t)b * a.blob_stride;
  int32_t* slot = reinterpret_cast<int32_t*>(blob + a.lay.slot);
  int32_t* depth = reinterpret_cast<int32_t*>(blob + a.lay.depth);
  int32_t* parent = reinterpret_cast<int32_t*>(blob + a.lay.parent);
  int32_t* internal = reinterpret_cast<int32_t*>(blob + a.lay.internal);
  int32_t* iidx = reinterpret_cast<int32_t*>(blob + a.lay.internal_index);
  int32_t* ret = reinterpret_cast<int32_t*>(blob + a.lay.retrieve);
  uint64_t* anc = reinterpret_cast<uint64_t*>(blob + a.lay.anc);

  if (tid == 0) { s_bad = 0; s_n = 0; s_chosen = 0; s_D = 0; }
  __syncthreads();
  for (int i = tid; i < K * R; i += kBThreads) {
    const double x = acc[i];
    if (!(x >= 0.0 && x <= 1.0)) s_bad = 1;          // also NaN
  }
  __syncthreads();
  const bool bad = s_bad != 0;
  // ---- search ----------------------------------------------------------------------------
  if (!bad && a.budget > 0) {
    for (int r = tid; r < R; r += kBThreads) {
      uint64_t hi = 0, lo = 0;
      put_rank(hi, lo, 0, r);
      e_w[r] = 1.0 * acc[r];
      e_hi[r] = hi;
      e_lo[r] = lo;
      e_par[r] = -1;
      e_len[r] = 1;
      e_state[r] = 0;
    }
    if (tid == 0) s_n = R;
    __syncthreads();
    for (int step = 0; step < a.budget; ++step) {
      const int n = s_n;
      Ent best{0.0, 0, 0, 0, -1};
      for (int i = tid; i < n; i += kBThreads) {
        if (e_state[i] != 0) continue;
        const Ent c{e_w[i], e_hi[i], e_lo[i], (int)e_len[i], i};
        if (ent_before(c, best)) best = c;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const Ent other = shfl_ent(best, o);
        if (ent_before(other, best)) best = other;
      }
      if (lane == 0) red[warp] = best;
      __syncthreads();
      if (warp == 0) {
        best = lane < kBThreads / 32 ? red[lane] : Ent{0.0, 0, 0, 0, -1};
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const Ent other = shfl_ent(best, o);
          if (ent_before(other, best)) best = other;
        }
        if (lane == 0) {
          s_best = best.idx;
          if (best.idx >= 0) {
            e_state[best.idx] = 1;
            s_chosen += 1;
          }
        }
      }
      __syncthreads();
      const int bi = s_best;
      if (bi < 0) break;                               // every path of depth <= K is taken
      const int len = e_len[bi];
      if (len < K) {
        for (int r = tid; r < R; r += kBThreads) {
          const int i = n + r;
          uint64_t hi = e_hi[bi], lo = e_lo[bi];
          put_rank(hi, lo, len, r);
          e_w[i] = e_w[bi] * acc[len * R + r];         // = the left-to-right product of the child
          e_hi[i] = hi;
          e_lo[i] = lo;
          e_par[i] = (int16_t)bi;
          e_len[i] = (uint8_t)(len + 1);
          e_state[i] = 0;
        }
        if (tid == 0) s_n = n + R;
      }
      __syncthreads();
    }
  }
  // ---- compile ---------------------------------------------------------------------------
  const int n_e = bad ? 0 : s_n;
  const int n_rows = (bad ? 0 : s_chosen) + 1;
  // canonical rows: 1 + the number of chosen paths that sort before this one
  for (int i = tid; i < n_e; i += kBThreads) {
    if (e_state[i] != 1) continue;
    const int li = e_len[i];
    const uint64_t hi = e_hi[i], lo = e_lo[i];
    int rank = 0;
    for (int j = 0; j < n_e; ++j) {
      if (e_state[j] != 1) continue;
      const int lj = e_len[j];
      rank += (lj < li || (lj == li && (e_hi[j] < hi || (e_hi[j] == hi && e_lo[j] < lo)))) ? 1 : 0;
    }
    e_row[i] = (int16_t)(1 + rank);
    atomicMax(&s_D, li);
  }
  __syncthreads();
  const int D = s_D;
  const int W = D + 1, n_words = (n_rows + 63) / 64;
  // per row: depth, slot, parent; child counts go to iidx (as a scratch) first
  for (int u = tid; u < n_rows; u += kBThreads) iidx[u] = 0;
  if (tid == 0) {
    depth[0] = 0;
    slot[0] = 0;
    parent[0] = -1;
  }
  __syncthreads();
  for (int i = tid; i < n_e; i += kBThreads) {
    if (e_state[i] != 1) continue;
    const int u = e_row[i], len = e_len[i];
    const int pu = e_par[i] < 0 ? 0 : e_row[e_par[i]];
    depth[u] = len;
    slot[u] = 1 + (len - 1) * a.topk + get_rank(e_hi[i], e_lo[i], len - 1);
    parent[u] = pu;
    atomicAdd(&iidx[pu], 1);
  }
  __syncthreads();
  // internal rows (with children) and leaves, both in row order: a block scan over rows,
  // each thread taking a contiguous run of rows
  const int per = (n_rows + kBThreads - 1) / kBThreads;
  const int r0 = tid * per, r1 = min(n_rows, r0 + per);
  int my_int = 0;
  for (int u = r0; u < r1; ++u) my_int += iidx[u] > 0 ? 1 : 0;
  int incl = my_int;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) s_scan[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int v = lane < kBThreads / 32 ? s_scan[lane] : 0;
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += t;
    }
    if (lane < kBThreads / 32) s_scan[lane] = inc - v;   // exclusive prefix of each warp
    if (lane == kBThreads / 32 - 1) {
      s_ni = inc;
      s_nl = n_rows - inc;
    }
  }
  __syncthreads();
  int ni_before = s_scan[warp] + incl - my_int;          // internal rows before row r0
  int nl_before = r0 - ni_before;                        // leaves before row r0
  for (int u = r0; u < r1; ++u) {
    const bool is_int = iidx[u] > 0;
    if (is_int) {
      internal[ni_before] = u;
      iidx[u] = ni_before++;
    } else {
      iidx[u] = -1;
      int v = u;                                          // retrieval row of this leaf
      for (int j = depth[u]; j >= 0; --j) {
        ret[(size_t)nl_before * W + j] = v;
        v = parent[v];
      }
      for (int j = depth[u] + 1; j < W; ++j) ret[(size_t)nl_before * W + j] = -1;
      ++nl_before;
    }
    // ancestor-or-self bits: walk the parent chain
    uint64_t* arow = anc + (size_t)u * n_words;
    for (int w = 0; w < n_words; ++w) arow[w] = 0ull;
    for (int v = u; v >= 0; v = parent[v]) arow[v / 64] |= 1ull << (v % 64);
  }
  __syncthreads();
  if (tid == 0) {
    medusa_tree_t t{};
    t.n_rows = n_rows;
    t.n_words = n_words;
    t.max_depth = D;
    t.n_paths = s_nl;
    t.topk = a.topk;
    t.n_internal = s_ni;
    t.slot = slot;
    t.depth = depth;
    t.parent = parent;
    t.retrieve = ret;
    t.internal = internal;
    t.internal_index = iidx;
    t.anc = anc;
    t.per_seq = nullptr;
    a.per_seq[b] = t;
    if (a.status) a.status[b] = bad ? MEDUSA_EINVAL : MEDUSA_OK;
  }
}

}  // namespace

TreeBlobLayout tree_blob_layout(int n_rows, int max_depth, int n_paths) {
  TreeBlobLayout l{};
  size_t off = 0;
  const size_t n = (size_t)n_rows * sizeof(int32_t);
  l.slot = off; off += n;
  l.depth = off; off += n;
  l.parent = off; off += n;
  l.internal = off; off += n;
  l.internal_index = off; off += n;
  l.retrieve = off; off += (size_t)n_paths * (max_depth + 1) * sizeof(int32_t);
  off = align_up(off, 16);
  l.anc = off; off += (size_t)n_rows * ((n_rows + 63) / 64) * sizeof(uint64_t);
  l.total = align_up(off, 16);
  return l;
}

size_t tree_greedy_smem(int R, int budget) {
  const size_t E = (size_t)R * (budget + 1);
  return E * (8 + 8 + 8 + 2 + 2 + 1 + 1);
}

cudaError_t launch_tree_greedy(const double* acc, int B, int K, int R, int budget, int topk, void* dev_buf,
                               size_t blob_stride, medusa_tree_t* per_seq, int32_t* status, cudaStream_t st) {
  BuildArgs a{};
  a.acc = acc;
  a.K = K;
  a.R = R;
  a.budget = budget;
  a.topk = topk;
  a.blobs = static_cast<char*>(dev_buf);
  a.blob_stride = blob_stride;
  a.lay = tree_blob_layout(budget + 1, K, budget > 0 ? budget : 1);
  a.per_seq = per_seq;
  a.status = status;
  const size_t smem = tree_greedy_smem(R, budget);
  cudaError_t e = cudaFuncSetAttribute(tree_greedy_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  tree_greedy_kernel<<<B, kBThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace medusa
