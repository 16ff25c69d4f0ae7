// Greedy and fast-typical acceptance on unique packed rows ([M7.2] §0x03D, §0x04D,
// §0x04E, §0x07B; [PartII] Part 7; [CN] "接受机制").
//
// Only internal rows (rows with children) are read: leaves never score a candidate.
//   row_stats_kernel   grid (chunks, internal rows, B): per chunk of V the max of
//                      x/T, sum e^{x/T-m}, sum e^{x/T-m}(x/T-m) and the argmax of x.
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

struct RowPart {
  float m;      // max of x / T over the chunk
  float z;      // sum exp(x/T - m)
  float s1;     // sum exp(x/T - m) * (x/T - m)
  float amax_v; // largest raw logit
  int amax_i;   // its id (lowest among equal values)
  int pad[3];
};

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

template <typename EL>
__global__ void __launch_bounds__(kThreads) row_stats_kernel(medusa_tree_t t, int V, int chunk,
                                                             const EL* __restrict__ logits,
                                                             float inv_temp,
                                                             RowPart* __restrict__ part) {
  const int c = blockIdx.x, ii = blockIdx.y, b = blockIdx.z;
  const int u = t.internal[ii];
  const EL* row = logits + ((int64_t)b * t.n_rows + u) * V;
  const int start = c * chunk, end = min(V, start + chunk);
  // pass 1: max and argmax
  float mx = -INFINITY, av = -INFINITY;
  int ai = INT_MAX;
  for (int i = start + threadIdx.x; i < end; i += kThreads) {
    const float x = Elem<EL>::load(row, i);
    if (ranks_before(x, i, av, ai)) { av = x; ai = i; }
  }
  __shared__ float red_v[kWarps];
  __shared__ int red_i[kWarps];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, av, o);
    const int oi = __shfl_xor_sync(0xffffffffu, ai, o);
    if (ranks_before(ov, oi, av, ai)) { av = ov; ai = oi; }
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) { red_v[warp] = av; red_i[warp] = ai; }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kWarps; ++w)
      if (ranks_before(red_v[w], red_i[w], av, ai)) { av = red_v[w]; ai = red_i[w]; }
    red_v[0] = av; red_i[0] = ai;
  }
  __syncthreads();
  av = red_v[0]; ai = red_i[0];
  mx = av * inv_temp;                         // T > 0: the max of x/T is at the argmax of x
  // pass 2: partition function and first moment relative to mx
  float z = 0.f, s1 = 0.f;
  for (int i = start + threadIdx.x; i < end; i += kThreads) {
    const float y = Elem<EL>::load(row, i) * inv_temp - mx;
    const float e = expf(y);
    z += e;
    s1 = fmaf(e, y, s1);
  }
  z = warp_sum(z);
  s1 = warp_sum(s1);
  __shared__ float red_z[kWarps], red_s[kWarps];
  __syncthreads();
  if (lane == 0) { red_z[warp] = z; red_s[warp] = s1; }
  __syncthreads();
  if (threadIdx.x == 0) {
    z = 0.f; s1 = 0.f;
    for (int w = 0; w < kWarps; ++w) { z += red_z[w]; s1 += red_s[w]; }
    RowPart p;
    p.m = mx; p.z = z; p.s1 = s1; p.amax_v = av; p.amax_i = ai;
    p.pad[0] = p.pad[1] = p.pad[2] = 0;
    part[(((int64_t)b * t.n_internal) + ii) * gridDim.x + c] = p;
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
  const int u = t.internal[ii];
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

template <typename EL>
__global__ void __launch_bounds__(kThreads) select_kernel(
    medusa_tree_t t, int V, int n_chunks, const EL* __restrict__ logits,
    const int32_t* __restrict__ tokens, int mode, float inv_temp, float epsilon, float delta,
    const RowPart* __restrict__ part, const float* __restrict__ guard,
    int32_t* __restrict__ best_path, int32_t* __restrict__ accept_len,
    int32_t* __restrict__ out_tokens, int32_t* __restrict__ out_rows,
    int32_t* __restrict__ frontier_row) {
  extern __shared__ float sm[];
  const int b = blockIdx.x;
  const int NI = t.n_internal;
  float* s_m = sm;             // [NI] max of x/T
  float* s_lz = sm + NI;       // [NI] log Z
  float* s_tau = sm + 2 * NI;  // [NI] typical threshold
  int* s_am = (int*)(sm + 3 * NI);  // [NI] argmax id
  // 1. merged statistics per internal row
  for (int ii = threadIdx.x; ii < NI; ii += kThreads) {
    const RowPart* rp = part + (((int64_t)b * NI) + ii) * n_chunks;
    float m, z, s1, av;
    int ai;
    merged_row(rp, n_chunks, m, z, s1, av, ai);
    const float lz = logf(z);
    float H;
    if (guard) {
      H = 0.f;
      for (int c = 0; c < n_chunks; ++c) H += guard[(((int64_t)b * NI) + ii) * n_chunks + c];
    } else {
      H = lz - s1 / z;          // -sum p ln p = ln Z - sum p (x/T - m)
    }
    s_m[ii] = m;
    s_lz[ii] = lz;
    s_tau[ii] = fminf(epsilon, delta * expf(-H));
    s_am[ii] = ai;
  }
  __syncthreads();
  // 2. every retrieval path
  const int W = t.max_depth + 1;
  const int32_t* tok = tokens + (int64_t)b * t.n_rows;
  int best_p = INT_MAX, best_a = -1;
  float best_s = -INFINITY;
  for (int p = threadIdx.x; p < t.n_paths; p += kThreads) {
    const int32_t* r = t.retrieve + (int64_t)p * W;
    int a = 0;
    float score = 0.f;
    for (int j = 0; j + 1 < W; ++j) {
      const int u = r[j], cnode = r[j + 1];
      if (cnode < 0) break;
      const int ii = t.internal_index[u];
      const int ct = tok[cnode];
      bool ok;
      if (ct < 0 || ct >= V) {
        ok = false;                          // not a vocabulary id: never accepted
      } else if (mode == MEDUSA_ACCEPT_GREEDY) {
        ok = (ct == s_am[ii]);
      } else {
        const float x = Elem<EL>::load(logits, ((int64_t)b * t.n_rows + u) * V + ct) * inv_temp;
        const float lp = x - s_m[ii] - s_lz[ii];
        ok = expf(lp) > s_tau[ii];
        if (ok) score += lp;
      }
      if (!ok) break;
      ++a;
    }
    const bool take = mode == MEDUSA_ACCEPT_GREEDY
                          ? (a > best_a || (a == best_a && p < best_p))
                          : (a > best_a || (a == best_a && (score > best_s || (score == best_s && p < best_p))));
    if (take) { best_a = a; best_s = score; best_p = p; }
  }
  // 3. block arg-best over paths
  __shared__ int r_a[kWarps], r_p[kWarps];
  __shared__ float r_s[kWarps];
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
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) { r_a[warp] = best_a; r_s[warp] = best_s; r_p[warp] = best_p; }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kWarps; ++w)
      if (better(r_a[w], r_s[w], r_p[w], best_a, best_s, best_p)) {
        best_a = r_a[w]; best_s = r_s[w]; best_p = r_p[w];
      }
    const int32_t* r = t.retrieve + (int64_t)best_p * W;
    best_path[b] = best_p;
    accept_len[b] = best_a;
    for (int j = 0; j < W; ++j) {
      const bool in = j <= best_a;
      out_rows[(int64_t)b * W + j] = in ? r[j] : -1;
      out_tokens[(int64_t)b * W + j] = in ? tok[r[j]] : -1;
    }
    frontier_row[b] = r[best_a];
  }
}

}  // namespace

AcceptPlan plan_accept(const medusa_tree_t& t, int B, int V) {
  AcceptPlan p{};
  p.B = B;
  p.V = V;
  int chunk = 8192;
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
                          int32_t* frontier_row, void* ws, cudaStream_t st) {
  RowPart* part = (RowPart*)((char*)ws + p.off_part);
  float* guard = (float*)((char*)ws + p.off_guard);
  const float inv_t = 1.f / temperature;
  const bool bf = dt == MEDUSA_BF16;
  if (t.n_internal > 0) {
    dim3 g(p.n_chunks, t.n_internal, p.B);
    if (bf) row_stats_kernel<uint16_t><<<g, kThreads, 0, st>>>(t, p.V, p.chunk, (const uint16_t*)logits, inv_t, part);
    else row_stats_kernel<float><<<g, kThreads, 0, st>>>(t, p.V, p.chunk, (const float*)logits, inv_t, part);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (entropy_guard && mode == MEDUSA_ACCEPT_TYPICAL) {
      if (bf) guard_kernel<uint16_t><<<g, kThreads, 0, st>>>(t, p.V, p.chunk, (const uint16_t*)logits, inv_t, part, guard);
      else guard_kernel<float><<<g, kThreads, 0, st>>>(t, p.V, p.chunk, (const float*)logits, inv_t, part, guard);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
  }
  const float* gptr = (entropy_guard && mode == MEDUSA_ACCEPT_TYPICAL) ? guard : nullptr;
  const size_t smem = (size_t)4 * (t.n_internal > 0 ? t.n_internal : 1) * sizeof(float);
  if (bf)
    select_kernel<uint16_t><<<p.B, kThreads, smem, st>>>(t, p.V, p.n_chunks, (const uint16_t*)logits, tokens, mode,
                                                         inv_t, epsilon, delta, part, gptr, best_path,
                                                         accept_len, out_tokens, out_rows, frontier_row);
  else
    select_kernel<float><<<p.B, kThreads, smem, st>>>(t, p.V, p.n_chunks, (const float*)logits, tokens, mode,
                                                      inv_t, epsilon, delta, part, gptr, best_path,
                                                      accept_len, out_tokens, out_rows, frontier_row);
  return cudaGetLastError();
}

}  // namespace medusa
