// Greedy and fast-typical acceptance on unique packed rows ([M7.2] §0x03D, §0x04D,
// §0x04E, §0x07B; [PartII] Part 7; [CN] "接受机制").
//
// Only internal rows (rows with children) are read: leaves never score a candidate.
//   row_stats_kernel   grid (chunks, internal rows, B): per chunk of V the argmax of x
//                      (greedy) or the max of x/T, sum e^{x/T-m} and sum
//                      e^{x/T-m}(x/T-m) (typical, which reads no argmax).
//   guard_kernel       (entropy_guard only) per chunk sum of -p ln(p + 1e-5) with the
//                      row's merged max and partition function.
//   select_kernel      one CTA per sequence: merge the chunk statistics per row, walk
//                      every retrieval path, pick the winner, publish G = a + 1 rows.
#include <float.h>
#include <limits.h>

#include "common.cuh"
#include "kernels.h"

namespace medusa {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kLoads = 8;          // 16-byte loads in flight per thread in row_stats
constexpr int kSelThreads = 1024;  // select: one warp per internal row, 32 rows at a time
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kCommitPieces = 2;   // 16-byte pieces a select thread holds while moving rows
// The fused commit moves one KV head's K and V rows (2 G rows of head_dim elements, G <=
// D + 1, head_dim <= 128, at most 4 bytes each; a bf16 cache with an fp16 mirror: 4 G
// rows of 2 bytes) in one batch of pieces.
static_assert(2 * (MEDUSA_MAX_DEPTH + 1) * (128 * 4 / 16) <= kSelThreads * kCommitPieces &&
                  4 * (MEDUSA_MAX_DEPTH + 1) * (128 * 2 / 16) <= kSelThreads * kCommitPieces,
              "one head's published K/V rows must fit the select kernel's pieces");


// Merge two partial statistics (log-sum-exp with first moment).
__device__ __forceinline__ void merge_stats(float& m, float& z, float& s1, float m2, float z2, float s12) {
  if (z2 <= 0.f) return;
  if (z <= 0.f) { m = m2; z = z2; s1 = s12; return; }
  const float mn = fmaxf(m, m2);
  const float a = expf(m - mn), b = expf(m2 - mn);
  s1 = a * (s1 + (m - mn) * z) + b * (s12 + (m2 - mn) * z2);
  z = a * z + b * z2;
  m = mn;
}

// 2^x on the MUFU unit (ex2.approx, relative error ~2^-22); 2^-inf = +0.
__device__ __forceinline__ float exp2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
constexpr float kLn2 = 0.6931471805599453f;   // (log2(e): kLog2e of the shared helpers)

// Fold a batch of n values x[] (ids i0..i0+n-1, all above the ids this thread folded
// before) into the running statistics.
//   greedy:  the argmax of x (ties to the lowest id): the batch max first, its first id
//            only when it beats the running max.
//   typical: in base-2 units, y = x * c2 with c2 = log2(e) / T: the max m2 of y,
//            Z = sum 2^(y - m2) (= sum e^{x/T - m} with m = m2 ln 2) and
//            S1 = sum 2^(y - m2) (y - m2) (= the natural-unit sum / ln 2).
template <bool TYP, int NB>
__device__ __forceinline__ void fold(const float* x, int i0, float c2, float& m2, float& z, float& s1,
                                     float& av, int& ai) {
  if (!TYP) {
    float bm = x[0];
#pragma unroll
    for (int e = 1; e < NB; ++e) bm = fmaxf(bm, x[e]);
    // (a NaN never ranks; an equal value folded before keeps its lower id, unless
    // nothing has been folded yet: -inf ranks by id like any value)
    if (bm > av || (bm == av && ai == INT_MAX)) {
      int k = 0;
#pragma unroll
      for (int e = NB - 1; e >= 0; --e)
        if (x[e] == bm) k = e;
      av = bm;
      ai = i0 + k;
    }
  } else {
    float y[NB], mb = -INFINITY;
#pragma unroll
    for (int e = 0; e < NB; ++e) { y[e] = x[e] * c2; mb = fmaxf(mb, y[e]); }
    if (mb == -INFINITY) return;                   // every value -inf: adds nothing
    if (z == 0.f) {
      m2 = mb;
    } else if (mb > m2) {
      const float d0 = m2 - mb;
      const float sc = exp2_approx(d0);
      s1 = sc * (s1 + d0 * z);
      z *= sc;
      m2 = mb;
    }
#pragma unroll
    for (int e = 0; e < NB; ++e) {
      // below -128 the term is 0 either way; the clamp keeps a -inf logit's e d at 0
      // instead of 0 * -inf (a NaN input stays NaN)
      const float d0 = y[e] - m2;
      const float d = d0 < -128.f ? -128.f : d0;
      const float ev = exp2_approx(d);
      z += ev;
      s1 = fmaf(ev, d, s1);
    }
  }
}

// One pass over a chunk of one internal row: argmax (greedy), or max, partition
// function and first moment (typical).  16-byte loads when the chunk is aligned.
template <typename EL, bool TYP>
__global__ void __launch_bounds__(kThreads) row_stats_kernel(medusa_tree_t t, int V, int chunk,
                                                             const EL* __restrict__ logits,
                                                             float inv_temp,
                                                             RowPart* __restrict__ part) {
  constexpr int EPV = Elem<EL>::kPerVec;
  const int c = blockIdx.x, ii = blockIdx.y, b = blockIdx.z;
  const medusa_tree_t tb = seq_tree(t, b);
  if (ii >= tb.n_internal) return;                 // (per-sequence templates: past this one's rows)
  const int u = tb.internal[ii];
  const EL* row = logits + ((int64_t)b * t.n_rows + u) * V;
  const int start = c * chunk, end = min(V, start + chunk);
  const float c2 = inv_temp * kLog2e;
  float m = -INFINITY, z = 0.f, s1 = 0.f, av = -INFINITY;   // (typical: m and s1 in base 2 until the end)
  int ai = INT_MAX;
  const bool vec = (reinterpret_cast<uintptr_t>(row + start) & 15u) == 0;
  int i = start;
  if (vec) {
    // kLoads 16-byte loads per thread are issued before any is folded (a chunk is
    // kLoads vectors per thread), so one memory round trip covers the chunk
    const int nvec = (end - start) / EPV;
    const uint4* rv = reinterpret_cast<const uint4*>(row + start);
    for (int q0 = threadIdx.x; q0 < nvec; q0 += kThreads * kLoads) {
      uint4 raw[kLoads];
#pragma unroll
      for (int l = 0; l < kLoads; ++l) {
        const int q = q0 + l * kThreads;
        raw[l] = q < nvec ? __ldg(rv + q) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int l = 0; l < kLoads; ++l) {
        const int q = q0 + l * kThreads;
        if (q < nvec) {
          float x[EPV];
          Elem<EL>::unpack(raw[l], x);
          fold<TYP, EPV>(x, start + q * EPV, c2, m, z, s1, av, ai);
        }
      }
    }
    i = start + nvec * EPV;
  }
  for (int k = i + threadIdx.x; k < end; k += kThreads) {
    float x[1] = {Elem<EL>::load(row, k)};
    fold<TYP, 1>(x, k, c2, m, z, s1, av, ai);
  }
  // Block reduction.  Typical: the max over the threads, every partial rescaled to it,
  // then plain sums (base 2; natural units in the record).  Greedy: the argmax.
  __shared__ float r_m[kWarps], r_z[kWarps], r_s[kWarps], r_v[kWarps];
  __shared__ int r_i[kWarps];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  auto rescale_sum = [&](float& mm, float& zz, float& ss) {
    float M = mm;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float a = zz > 0.f ? exp2_approx(mm - M) : 0.f;
    float zs = a * zz, s1s = zz > 0.f ? a * (ss + (mm - M) * zz) : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      zs += __shfl_xor_sync(0xffffffffu, zs, o);
      s1s += __shfl_xor_sync(0xffffffffu, s1s, o);
    }
    mm = M;
    zz = zs;
    ss = s1s;
  };
  auto argmax_lanes = [&](float& v, int& i) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, v, o);
      const int oi = __shfl_xor_sync(0xffffffffu, i, o);
      if (ranks_before(ov, oi, v, i)) { v = ov; i = oi; }
    }
  };
  if (TYP) rescale_sum(m, z, s1);
  else argmax_lanes(av, ai);
  if (lane == 0) { r_m[warp] = m; r_z[warp] = z; r_s[warp] = s1; r_v[warp] = av; r_i[warp] = ai; }
  __syncthreads();
  if (warp == 0) {
    const bool w = lane < kWarps;
    m = w ? r_m[lane] : -INFINITY;
    z = w ? r_z[lane] : 0.f;
    s1 = w ? r_s[lane] : 0.f;
    av = w ? r_v[lane] : -INFINITY;
    ai = w ? r_i[lane] : INT_MAX;
    if (TYP) rescale_sum(m, z, s1);
    else argmax_lanes(av, ai);
    if (lane == 0) {
      RowPart p;
      p.m = TYP ? m * kLn2 : -INFINITY;
      p.z = TYP ? z : 0.f;
      p.s1 = TYP ? s1 * kLn2 : 0.f;
      p.amax_v = av; p.amax_i = ai;
      p.pad[0] = p.pad[1] = p.pad[2] = 0;
      part[(((int64_t)b * t.n_internal) + ii) * gridDim.x + c] = p;
    }
  }
}

// Per-row merged (m, log Z) from the chunk partials; used by the guarded entropy.
__device__ __forceinline__ void merged_row(const RowPart* p, int n_chunks, float& m, float& z, float& s1,
                                           float& av, int& ai) {
  m = -INFINITY; z = 0.f; s1 = 0.f; av = -INFINITY; ai = INT_MAX;
  for (int c = 0; c < n_chunks; ++c) {
    merge_stats(m, z, s1, p[c].m, p[c].z, p[c].s1);
    if (ranks_before(p[c].amax_v, p[c].amax_i, av, ai)) { av = p[c].amax_v; ai = p[c].amax_i; }
  }
}

template <typename EL>
__global__ void __launch_bounds__(kThreads) guard_kernel(medusa_tree_t t, int V, int chunk,
                                                         const EL* __restrict__ logits, float inv_temp,
                                                         const RowPart* __restrict__ part,
                                                         float* __restrict__ guard) {
  const int c = blockIdx.x, ii = blockIdx.y, b = blockIdx.z;
  const medusa_tree_t tb = seq_tree(t, b);
  if (ii >= tb.n_internal) return;
  const int u = tb.internal[ii];
  const RowPart* rp = part + (((int64_t)b * t.n_internal) + ii) * gridDim.x;
  float m, z, s1, av;
  int ai;
  merged_row(rp, gridDim.x, m, z, s1, av, ai);
  const float inv_z = 1.f / z;
  const EL* row = logits + ((int64_t)b * t.n_rows + u) * V;
  const int start = c * chunk, end = min(V, start + chunk);
  float acc = 0.f;
  for (int i = start + threadIdx.x; i < end; i += kThreads) {
    const float p = expf(Elem<EL>::load(row, i) * inv_temp - m) * inv_z;
    acc -= p * logf(p + 1e-5f);
  }
  acc = warp_sum(acc);
  __shared__ float red[kWarps];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int w = 0; w < kWarps; ++w) s += red[w];
    guard[(((int64_t)b * t.n_internal) + ii) * gridDim.x + c] = s;
  }
}

// Shared-memory layout of select_kernel: per internal row m, log Z, tau, argmax; per
// node the acceptance of its incoming edge and its log-probability; the retrieval
// table when it fits.
struct SelectSmem {
  size_t off_lp, off_ok, off_ret, off_part, bytes;
  bool ret_staged, part_staged;
};
inline SelectSmem select_smem(const medusa_tree_t& t, int n_chunks, bool guard) {
  SelectSmem L{};
  const size_t ni = t.n_internal > 0 ? t.n_internal : 1;
  L.off_lp = align_up(4 * ni * sizeof(float), 16);
  L.off_ok = align_up(L.off_lp + (size_t)t.n_rows * sizeof(float), 16);
  L.off_ret = align_up(L.off_ok + (size_t)t.n_rows, 16);
  const size_t ret = (size_t)t.n_paths * (t.max_depth + 1) * sizeof(int32_t);
  L.ret_staged = L.off_ret + ret <= 96 * 1024;
  L.off_part = align_up(L.ret_staged ? L.off_ret + ret : L.off_ret, 16);
  // the chunk statistics of every internal row (and their guard terms), when they fit
  const size_t parts = ni * n_chunks * (sizeof(RowPart) + (guard ? sizeof(float) : 0));
  L.part_staged = L.off_part + parts <= 160 * 1024;
  L.bytes = L.part_staged ? L.off_part + parts : L.off_part;
  return L;
}

template <typename EL>
__global__ void __launch_bounds__(kSelThreads) select_kernel(
    medusa_tree_t t, int V, int n_chunks, const EL* __restrict__ logits,
    const int32_t* __restrict__ tokens, int mode, float inv_temp, float epsilon, float delta,
    const RowPart* __restrict__ part, const float* __restrict__ guard, SelectSmem lay,
    const float* __restrict__ edge_x, const int* __restrict__ err, CommitArgs cm,
    int32_t* __restrict__ best_path, int32_t* __restrict__ accept_len,
    int32_t* __restrict__ out_tokens, int32_t* __restrict__ out_rows,
    int32_t* __restrict__ frontier_row) {
  extern __shared__ __align__(16) unsigned char smem_sel[];
  float* s_m = reinterpret_cast<float*>(smem_sel);
  const int b = blockIdx.x;
  // Strides of the per-row tensors and of the chunk statistics come from t (a bound over
  // the batch when templates are per sequence); the tree itself from this sequence's.
  const int NIS = t.n_internal, NS = t.n_rows, WS = t.max_depth + 1;
  const medusa_tree_t tq = seq_tree(t, b);
  const int NI = tq.n_internal, N = tq.n_rows;
  float* s_lz = s_m + NI;                        // [NI] log Z
  float* s_tau = s_m + 2 * NI;                   // [NI] typical threshold
  int* s_am = reinterpret_cast<int*>(s_m + 3 * NI);   // [NI] argmax id
  float* s_lp = reinterpret_cast<float*>(smem_sel + lay.off_lp);   // [N] log p of the edge into v
  uint8_t* s_ok = smem_sel + lay.off_ok;         // [N] edge into v accepted
  int32_t* s_ret = reinterpret_cast<int32_t*>(smem_sel + lay.off_ret);
  const int W = tq.max_depth + 1;                 // retrieval width of this template
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const bool typ = mode != MEDUSA_ACCEPT_GREEDY;
  const int32_t* tok = tokens + (int64_t)b * NS;
  // (the error flag is read now and tested once the loads below are in flight)
  const int err_v = err ? *reinterpret_cast<const volatile int*>(err) : 0;
  // 0. the inputs of every edge parent(v) -> v (a thread's edges are v = 1 + tid +
  //    k kSelThreads, k < kEdges since N <= MEDUSA_MAX_ROWS): parent, its internal row,
  //    the candidate token and (typical) its raw logit, all requested up front so that
  //    their latency overlaps the statistics below.
  constexpr int kEdges = (MEDUSA_MAX_ROWS + kSelThreads - 1) / kSelThreads;
  int e_ii[kEdges], e_ct[kEdges];
  float e_x[kEdges];
  {
    int e_u[kEdges];
#pragma unroll
    for (int k = 0; k < kEdges; ++k) {
      const int v = 1 + threadIdx.x + k * kSelThreads;
      e_u[k] = v < N ? tq.parent[v] : 0;
      e_ct[k] = v < N ? tok[v] : -1;
    }
#pragma unroll
    for (int k = 0; k < kEdges; ++k) {
      const int v = 1 + threadIdx.x + k * kSelThreads;
      e_ii[k] = v < N ? tq.internal_index[e_u[k]] : 0;
      const bool need = typ && v < N && e_ct[k] >= 0 && e_ct[k] < V;
      // the logit of v's token at its parent: from the logits, or (projection folded
      // in) the value the statistics kernel recorded for this edge
      e_x[k] = !need ? 0.f
                     : (edge_x ? edge_x[(int64_t)b * NS + v]
                               : Elem<EL>::load(logits, ((int64_t)b * NS + e_u[k]) * V + e_ct[k])) * inv_temp;
    }
  }
  // 1. merged statistics per internal row (one warp per row, one lane per chunk) and
  //    the retrieval table into shared memory.  The chunk statistics of every row and
  //    the table are staged first, up to two of each per thread in flight, so that the
  //    per-row merges do not wait on global memory one row after another.
  const RowPart* part_b = part + (int64_t)b * NIS * n_chunks;
  const float* guard_b = guard ? guard + (int64_t)b * NIS * n_chunks : nullptr;
  {
    RowPart* sp = reinterpret_cast<RowPart*>(smem_sel + lay.off_part);
    float* sg = reinterpret_cast<float*>(sp + NI * n_chunks);
    const int np = lay.part_staged ? NI * n_chunks : 0;
    const int nr = lay.ret_staged ? tq.n_paths * W : 0;
    for (int i0 = threadIdx.x; i0 < max(np, nr); i0 += 2 * kSelThreads) {
      RowPart q[2];
      float g4[2];
      int rv[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int i = i0 + r * kSelThreads;
        if (i < np) {
          q[r] = part_b[i];
          g4[r] = guard_b ? guard_b[i] : 0.f;
        }
        if (i < nr) rv[r] = tq.retrieve[i];
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int i = i0 + r * kSelThreads;
        if (i < np) {
          sp[i] = q[r];
          if (guard_b) sg[i] = g4[r];
        }
        if (i < nr) s_ret[i] = rv[r];
      }
    }
    if (lay.part_staged) {
      part_b = sp;
      if (guard_b) guard_b = sg;
    }
    __syncthreads();
  }
  if (err_v != 0) {
    // the statistics were not completed (a bounded wait gave up): publish nothing
    if (threadIdx.x == 0) {
      best_path[b] = -1;
      accept_len[b] = -1;
      frontier_row[b] = -1;
      if (cm.on) {                               // nothing to commit: the cache is untouched
        cm.status[b] = MEDUSA_EPATH;
        cm.L_out[b] = cm.L[b];
      }
    }
    for (int j = threadIdx.x; j < WS; j += kSelThreads) {
      out_rows[(int64_t)b * WS + j] = -1;
      out_tokens[(int64_t)b * WS + j] = -1;
    }
    return;
  }
  // A row takes lpr lanes (the smallest power of two >= the chunk count, at most 32), so a
  // warp merges 32 / lpr rows at once; the shuffles stay inside each group of lanes.
  int lpr = 1;
  while (lpr < n_chunks && lpr < 32) lpr <<= 1;
  const int rpw = 32 / lpr, sl = lane & (lpr - 1);
  for (int ii0 = warp * rpw; ii0 < NI; ii0 += kSelWarps * rpw) {
    const int ii = ii0 + lane / lpr;
    const bool row = ii < NI;
    const RowPart* rp = part_b + (int64_t)ii * n_chunks;
    float m = -INFINITY, z = 0.f, s1 = 0.f, av = -INFINITY, g = 0.f;
    int ai = INT_MAX;
    for (int c = sl; row && c < n_chunks; c += lpr) {
      const RowPart q = rp[c];
      if (typ) merge_stats(m, z, s1, q.m, q.z, q.s1);
      if (ranks_before(q.amax_v, q.amax_i, av, ai)) { av = q.amax_v; ai = q.amax_i; }
      if (guard_b) g += guard_b[(int64_t)ii * n_chunks + c];
    }
    if (typ) {
      // the row max over the lanes, every lane's partial rescaled to it, then plain sums
      // (typical needs no argmax)
      float M = m;
      for (int o = lpr >> 1; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      const float a = z > 0.f ? __expf(m - M) : 0.f;
      float zz = a * z, ss = z > 0.f ? a * (s1 + (m - M) * z) : 0.f;
      for (int o = lpr >> 1; o > 0; o >>= 1) {
        zz += __shfl_xor_sync(0xffffffffu, zz, o);
        ss += __shfl_xor_sync(0xffffffffu, ss, o);
      }
      m = M;
      z = zz;
      s1 = ss;
    } else {                                        // greedy needs the argmax only
      for (int o = lpr >> 1; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, av, o);
        const int oi = __shfl_xor_sync(0xffffffffu, ai, o);
        if (ranks_before(ov, oi, av, ai)) { av = ov; ai = oi; }
      }
    }
    if (guard_b)
      for (int o = lpr >> 1; o > 0; o >>= 1) g += __shfl_xor_sync(0xffffffffu, g, o);
    if (row && sl == 0) {
      s_am[ii] = ai;
      if (typ) {
        const float lz = logf(z);
        const float H = guard_b ? g : lz - s1 / z;   // -sum p ln p = ln Z - sum p (x/T - m)
        s_m[ii] = m;
        s_lz[ii] = lz;
        s_tau[ii] = fminf(epsilon, delta * expf(-H));
      }
    }
  }
  __syncthreads();
  // 2. every edge parent(v) -> v at once: accepted? and log p_parent(token of v)
#pragma unroll
  for (int k = 0; k < kEdges; ++k) {
    const int v = 1 + threadIdx.x + k * kSelThreads;
    if (v >= N) break;
    const int ii = e_ii[k], ct = e_ct[k];
    bool ok = false;
    float lp = 0.f;
    if (ct >= 0 && ct < V) {                     // else: not a vocabulary id, never accepted
      if (!typ) {
        ok = ct == s_am[ii];
      } else {
        lp = e_x[k] - s_m[ii] - s_lz[ii];
        ok = expf(lp) > s_tau[ii];
      }
    }
    s_ok[v] = ok ? 1 : 0;
    s_lp[v] = lp;
  }
  __syncthreads();
  // 3. every retrieval path: accepted prefix length and its log-probability
  int best_p = INT_MAX, best_a = -1;
  float best_s = -INFINITY;
  for (int p = threadIdx.x; p < tq.n_paths; p += kSelThreads) {
    const int32_t* r = lay.ret_staged ? s_ret + p * W : tq.retrieve + (int64_t)p * W;
    int a = 0;
    float score = 0.f;
    for (int j = 1; j < W; ++j) {
      const int cnode = r[j];
      if (cnode < 0 || !s_ok[cnode]) break;
      score += s_lp[cnode];
      ++a;
    }
    const bool take = !typ ? (a > best_a || (a == best_a && p < best_p))
                           : (a > best_a || (a == best_a && (score > best_s || (score == best_s && p < best_p))));
    if (take) { best_a = a; best_s = score; best_p = p; }
  }
  // 3. block arg-best over paths
  __shared__ int r_a[kSelWarps], r_p[kSelWarps];
  __shared__ float r_s[kSelWarps];
  auto better = [&](int a1, float s1, int p1, int a2, float s2, int p2) {
    if (a1 != a2) return a1 > a2;
    if (mode != MEDUSA_ACCEPT_GREEDY && s1 != s2) return s1 > s2;
    return p1 < p2;
  };
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const int oa = __shfl_xor_sync(0xffffffffu, best_a, o);
    const float os = __shfl_xor_sync(0xffffffffu, best_s, o);
    const int op = __shfl_xor_sync(0xffffffffu, best_p, o);
    if (better(oa, os, op, best_a, best_s, best_p)) { best_a = oa; best_s = os; best_p = op; }
  }
  if (lane == 0) { r_a[warp] = best_a; r_s[warp] = best_s; r_p[warp] = best_p; }
  __syncthreads();
  static_assert(kSelWarps == 32, "one lane per warp in the final reduction");
  if (warp == 0) {
    // the warps' winners, one per lane, reduced by the same comparison (a total order on
    // (length, score, path id)); then the lanes publish the rows in parallel
    best_a = r_a[lane]; best_s = r_s[lane]; best_p = r_p[lane];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const int oa = __shfl_xor_sync(0xffffffffu, best_a, o);
      const float os = __shfl_xor_sync(0xffffffffu, best_s, o);
      const int op = __shfl_xor_sync(0xffffffffu, best_p, o);
      if (better(oa, os, op, best_a, best_s, best_p)) { best_a = oa; best_s = os; best_p = op; }
    }
    const int32_t* r = lay.ret_staged ? s_ret + best_p * W : tq.retrieve + (int64_t)best_p * W;
    for (int j = lane; j < WS; j += 32) {
      const bool in = j <= best_a;
      const int row = in ? r[j] : -1;
      out_rows[(int64_t)b * WS + j] = row;
      out_tokens[(int64_t)b * WS + j] = in ? tok[row] : -1;
    }
    if (lane == 0) {
      best_path[b] = best_p;
      accept_len[b] = best_a;
      frontier_row[b] = r[best_a];
    }
  }
  if (!cm.on) return;

  // ---- fused commit: medusa_kv_compact of this sequence --------------------------------
  // Thread 0 validates as the compaction kernel does (capacity, then the chain of
  // published rows); then every KV head's G rows of K and V (and of their fp16 mirror,
  // if the cache has one) move as 16-byte pieces, a group of heads at a time: all
  // pieces of the group are read into registers before any is written, so overlapping
  // source and destination rows are safe (rows of different heads never overlap).
  __shared__ int c_rows[MEDUSA_MAX_DEPTH + 1];
  __shared__ int c_status, c_G, c_L;
  if (threadIdx.x == 0) {
    const int a = best_a;
    const int32_t* r = lay.ret_staged ? s_ret + best_p * W : tq.retrieve + (int64_t)best_p * W;
    const int Lb = cm.L[b];
    int v = MEDUSA_OK;
    if (Lb < 0 || !seq_rows_ok(cm.c, b, (int64_t)Lb + N)) {
      v = MEDUSA_ECAPACITY;
    } else if (a < 0 || a > tq.max_depth) {
      v = MEDUSA_EPATH;
    } else {
      for (int j = 0; j <= a; ++j) {
        const int u = r[j];
        c_rows[j] = u;
        if (u < 0 || u >= N || (j == 0 ? u != 0 : tq.parent[u] != r[j - 1])) v = MEDUSA_EPATH;
      }
    }
    c_status = v;
    c_G = a + 1;
    c_L = Lb;
    cm.status[b] = v;
    cm.L_out[b] = v == MEDUSA_OK ? Lb + a + 1 : Lb;
  }
  __syncthreads();
  if (c_status != MEDUSA_OK) return;
  const int G = c_G, Lb = c_L;
  const int esz = cm.c.dtype == MEDUSA_BF16 ? 2 : 4;
  const int pr = cm.c.head_dim * esz / 16;                  // pieces per row
  const int n_arr = cm.c.k_f16 ? 4 : 2;                     // K, V (, K and V mirrors)
  const int per_head = n_arr * G * pr;                      // their rows of one head
  int hg = (kSelThreads * kCommitPieces) / per_head;         // heads per group
  if (hg < 1) hg = 1;
  auto arr = [&](int kv) -> char* {
    return static_cast<char*>(kv == 0 ? cm.c.k : kv == 1 ? cm.c.v : kv == 2 ? cm.c.k_f16 : cm.c.v_f16);
  };
  for (int h0 = 0; h0 < cm.c.n_kv_heads; h0 += hg) {
    const int nh = min(hg, cm.c.n_kv_heads - h0);
    const int n = nh * per_head;
    uint4 piece[kCommitPieces];
#pragma unroll
    for (int k = 0; k < kCommitPieces; ++k) {
      const int i = threadIdx.x + k * kSelThreads;
      if (i < n) {
        const int h = h0 + i / per_head, rem = i % per_head;
        const int kv = rem / (G * pr), j = (rem / pr) % G, e = rem % pr;
        const char* base = arr(kv);
        const int64_t off = cache_row_offset(cm.c, b, h, Lb + c_rows[j]) * esz + 16 * e;
        piece[k] = *reinterpret_cast<const uint4*>(base + off);
      }
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kCommitPieces; ++k) {
      const int i = threadIdx.x + k * kSelThreads;
      if (i < n) {
        const int h = h0 + i / per_head, rem = i % per_head;
        const int kv = rem / (G * pr), j = (rem / pr) % G, e = rem % pr;
        char* base = arr(kv);
        const int64_t off = cache_row_offset(cm.c, b, h, Lb + j) * esz + 16 * e;
        *reinterpret_cast<uint4*>(base + off) = piece[k];
      }
    }
    __syncthreads();
  }
}

}  // namespace

AcceptPlan plan_accept(const medusa_tree_t& t, int B, int V) {
  AcceptPlan p{};
  p.B = B;
  p.V = V;
  int chunk = kThreads * kLoads * 8;                      // bf16: 8 per 16-byte vector
  if (V < chunk) chunk = (V + 255) / 256 * 256;
  p.chunk = chunk;
  p.n_chunks = (V + chunk - 1) / chunk;
  const size_t nparts = (size_t)B * (t.n_internal > 0 ? t.n_internal : 1) * p.n_chunks;
  p.off_part = 0;
  p.off_guard = align_up(nparts * sizeof(RowPart), 256);
  p.bytes = align_up(p.off_guard + nparts * sizeof(float), 256);
  return p;
}

cudaError_t launch_accept(const AcceptPlan& p, const medusa_tree_t& t, const void* logits,
                          medusa_dtype dt, const int32_t* tokens, int mode, float temperature,
                          float epsilon, float delta, int entropy_guard, int32_t* best_path,
                          int32_t* accept_len, int32_t* out_tokens, int32_t* out_rows,
                          int32_t* frontier_row, void* ws, cudaStream_t st, const CommitArgs& cm) {
  RowPart* part = (RowPart*)((char*)ws + p.off_part);
  float* guard = (float*)((char*)ws + p.off_guard);
  const float inv_t = 1.f / temperature;
  const bool bf = dt == MEDUSA_BF16;
  const bool typ = mode == MEDUSA_ACCEPT_TYPICAL;
  if (t.n_internal > 0) {
    dim3 g(p.n_chunks, t.n_internal, p.B);
    if (bf && typ) row_stats_kernel<uint16_t, true><<<g, kThreads, 0, st>>>(t, p.V, p.chunk, (const uint16_t*)logits, inv_t, part);
    else if (bf) row_stats_kernel<uint16_t, false><<<g, kThreads, 0, st>>>(t, p.V, p.chunk, (const uint16_t*)logits, inv_t, part);
    else if (typ) row_stats_kernel<float, true><<<g, kThreads, 0, st>>>(t, p.V, p.chunk, (const float*)logits, inv_t, part);
    else row_stats_kernel<float, false><<<g, kThreads, 0, st>>>(t, p.V, p.chunk, (const float*)logits, inv_t, part);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (entropy_guard && typ) {
      if (bf) guard_kernel<uint16_t><<<g, kThreads, 0, st>>>(t, p.V, p.chunk, (const uint16_t*)logits, inv_t, part, guard);
      else guard_kernel<float><<<g, kThreads, 0, st>>>(t, p.V, p.chunk, (const float*)logits, inv_t, part, guard);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
  }
  const float* gptr = (entropy_guard && typ) ? guard : nullptr;
  const SelectSmem lay = select_smem(t, p.n_chunks, gptr != nullptr);
  cudaError_t e;
  if (bf) {
    e = cudaFuncSetAttribute(select_kernel<uint16_t>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)lay.bytes);
    if (e != cudaSuccess) return e;
    select_kernel<uint16_t><<<p.B, kSelThreads, lay.bytes, st>>>(t, p.V, p.n_chunks, (const uint16_t*)logits, tokens,
                                                              mode, inv_t, epsilon, delta, part, gptr, lay, nullptr,
                                                              nullptr, cm, best_path, accept_len, out_tokens,
                                                              out_rows, frontier_row);
  } else {
    e = cudaFuncSetAttribute(select_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)lay.bytes);
    if (e != cudaSuccess) return e;
    select_kernel<float><<<p.B, kSelThreads, lay.bytes, st>>>(t, p.V, p.n_chunks, (const float*)logits, tokens, mode,
                                                           inv_t, epsilon, delta, part, gptr, lay, nullptr, nullptr,
                                                           cm, best_path, accept_len, out_tokens, out_rows,
                                                           frontier_row);
  }
  return cudaGetLastError();
}

cudaError_t launch_select_parts(const medusa_tree_t& t, int B, int V, int n_chunks, const RowPart* part,
                                const float* edge_x, const int* err, const int32_t* tokens, int mode,
                                float temperature, float epsilon, float delta, int32_t* best_path,
                                int32_t* accept_len, int32_t* out_tokens, int32_t* out_rows,
                                int32_t* frontier_row, cudaStream_t st, const CommitArgs& cm) {
  const SelectSmem lay = select_smem(t, n_chunks, false);
  cudaError_t e = cudaFuncSetAttribute(select_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)lay.bytes);
  if (e != cudaSuccess) return e;
  select_kernel<float><<<B, kSelThreads, lay.bytes, st>>>(t, V, n_chunks, nullptr, tokens, mode, 1.f / temperature,
                                                         epsilon, delta, part, nullptr, lay, edge_x, err, cm,
                                                         best_path, accept_len, out_tokens, out_rows,
                                                         frontier_row);
  return cudaGetLastError();
}

}  // namespace medusa
