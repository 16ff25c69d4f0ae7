// Medusa heads + top-k ([CN] "Medusa 的核心思路与系统位置"; [Math] "The Medusa head:
// math and shapes"; [M7.2] §0x02A, §0x04D; [PartII] Part 4).
//
// Three phases, all HBM-bound at small T (weights are read exactly once):
//   1. residual GEMV  z_k = h + SiLU(W1_k h + b1_k)      rows: K*d,  x = h
//   2. vocabulary GEMV logits[m] = W_m x_m               rows: (K+1)*V, x_0 = h, x_k = z_{k-1}
//   3. top-k: per-chunk candidates, then one merge per (row t, matrix m).
// The GEMV streams each weight row with 128-bit L1-bypassing loads, keeps the
// fp32 input rows in shared memory and reduces each dot product with warp shuffles.
#include <float.h>
#include <limits.h>

#include "common.cuh"
#include "kernels.h"

namespace medusa {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTopkMaxSpans = 64;     // CTAs per logits row in the top-k

struct GemvArgs {
  const void* w0;           // matrix 0
  const void* w_rest;       // matrix 1 (further matrices at w_rest_stride elements)
  int64_t w_rest_stride;
  int n_rows, d;
  const void* x0;           // input rows of matrix 0 (dtype EL when x0_el, else fp32)
  int x0_el;
  int64_t x0_tok_stride;
  const float* x_rest;      // fp32 input rows of matrix m >= 1, or nullptr to reuse x0
  int64_t x_rest_tok_stride, x_rest_mat_stride;
  int t0, tcount;           // token rows [t0, t0 + tcount)
  float* out;
  int64_t out_tok_stride, out_mat_stride;
  int resid;                // 1: out = hres + SiLU(acc + b1[m]) (residual block epilogue)
  const void* b1;
};

template <typename EL, int TT, int R, int U>
__global__ void __launch_bounds__(kThreads) gemv_kernel(GemvArgs a) {
  extern __shared__ float xs[];               // [TT][d]
  constexpr int EPV = Elem<EL>::kPerVec;
  const int m = blockIdx.y;
  const int d = a.d;
  const EL* W = (const EL*)(m == 0 ? a.w0 : (const void*)((const EL*)a.w_rest +
                                                          (int64_t)(m - 1) * a.w_rest_stride));
  // Stage the fp32 input rows of this matrix.
  for (int tt = 0; tt < TT; ++tt) {
    const int t = a.t0 + tt;
    for (int i = threadIdx.x; i < d; i += kThreads) {
      float v = 0.f;
      if (tt < a.tcount) {
        if (m == 0 || a.x_rest == nullptr) {
          v = a.x0_el ? Elem<EL>::load((const EL*)a.x0, (int64_t)t * a.x0_tok_stride + i)
                      : ((const float*)a.x0)[(int64_t)t * a.x0_tok_stride + i];
        } else {
          v = a.x_rest[(int64_t)t * a.x_rest_tok_stride + (int64_t)(m - 1) * a.x_rest_mat_stride + i];
        }
      }
      xs[tt * d + i] = v;
    }
  }
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nvec = d / EPV;
  const int rows_per_iter = kWarps * R;
  for (int base = blockIdx.x * rows_per_iter; base < a.n_rows; base += gridDim.x * rows_per_iter) {
    const int row0 = base + warp * R;
    float acc[R][TT];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int t = 0; t < TT; ++t) acc[r][t] = 0.f;

    for (int v0 = 0; v0 < nvec; v0 += 32 * U) {
      uint4 w[R][U];
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int j = 0; j < U; ++j) {
          const int vi = v0 + j * 32 + lane;
          const int row = row0 + r;
          if (row < a.n_rows && vi < nvec)
            w[r][j] = ldg_stream(W + (int64_t)row * d + (int64_t)vi * EPV);
          else
            w[r][j] = make_uint4(0, 0, 0, 0);
        }
#pragma unroll
      for (int j = 0; j < U; ++j) {
        const int vi = v0 + j * 32 + lane;
        if (vi >= nvec) break;
        float wf[R][EPV];
#pragma unroll
        for (int r = 0; r < R; ++r) Elem<EL>::unpack(w[r][j], wf[r]);
#pragma unroll
        for (int t = 0; t < TT; ++t) {
          const float4* xp = reinterpret_cast<const float4*>(xs + t * d + vi * EPV);
          float xf[EPV];
#pragma unroll
          for (int e = 0; e < EPV / 4; ++e) {
            float4 q = xp[e];
            xf[4 * e] = q.x; xf[4 * e + 1] = q.y; xf[4 * e + 2] = q.z; xf[4 * e + 3] = q.w;
          }
#pragma unroll
          for (int r = 0; r < R; ++r)
#pragma unroll
            for (int e = 0; e < EPV; ++e) acc[r][t] = fmaf(wf[r][e], xf[e], acc[r][t]);
        }
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int t = 0; t < TT; ++t) acc[r][t] = warp_sum(acc[r][t]);

    if (lane == 0) {
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int row = row0 + r;
        if (row >= a.n_rows) continue;
#pragma unroll
        for (int t = 0; t < TT; ++t) {
          if (t >= a.tcount) continue;
          const int tg = a.t0 + t;
          float v = acc[r][t];
          if (a.resid) {
            if (a.b1) v += Elem<EL>::load((const EL*)a.b1, (int64_t)m * d + row);
            const float s = v / (1.f + expf(-v));                 // SiLU
            v = xs[t * d + row] + s;                              // residual: x0 is h
          }
          a.out[(int64_t)tg * a.out_tok_stride + (int64_t)m * a.out_mat_stride + row] = v;
        }
      }
    }
  }
}

// ---- bulk-copy streaming GEMV (T <= 2) -------------------------------------------
// One CTA per SM and matrix slice.  A producer warp streams groups of 8 weight rows,
// one row segment of up to 8 KiB per consumer warp, with cp.async.bulk into a
// shared-memory ring of NS stages of 64 KiB (three when the input rows leave room,
// so that up to 192 KiB are in flight per SM); 8 consumer warps
// each dot their row segment against the fp32 input rows kept in shared memory.
// Rows longer than one segment are streamed as several column chunks.
constexpr int kBulkConsumers = 8;
constexpr int kBulkThreads = (kBulkConsumers + 1) * 32;
constexpr int kBulkSegBytes = 8192;

inline size_t bulk_smem_bytes(int TT, int d, int stages) {
  return (size_t)((TT * d * 4 + 1023) & ~1023) + (size_t)stages * kBulkConsumers * kBulkSegBytes +
         2 * (size_t)stages * sizeof(uint64_t);
}

template <typename EL, int TT, int kBulkStages>
__global__ void __launch_bounds__(kBulkThreads, 1) gemv_bulk_kernel(GemvArgs a, int* __restrict__ err) {
  extern __shared__ __align__(1024) uint8_t smem_b[];
  constexpr int EPV = Elem<EL>::kPerVec;
  constexpr int CW = kBulkSegBytes / (int)sizeof(EL);            // columns per segment
  const int d = a.d;
  const int m = blockIdx.y;
  float* xs = reinterpret_cast<float*>(smem_b);                    // [TT][d]
  const int x_bytes = ((TT * d * 4) + 1023) & ~1023;
  uint8_t* ring = smem_b + x_bytes;                                 // [stages][8][CW]
  uint64_t* bars = reinterpret_cast<uint64_t*>(ring + kBulkStages * kBulkConsumers * kBulkSegBytes);
  const uint32_t full0 = smem_u32(&bars[0]), empty0 = smem_u32(&bars[kBulkStages]);
  const EL* W = (const EL*)(m == 0 ? a.w0 : (const void*)((const EL*)a.w_rest +
                                                          (int64_t)(m - 1) * a.w_rest_stride));
  for (int tt = 0; tt < TT; ++tt) {
    const int t = a.t0 + tt;
    for (int i = threadIdx.x; i < d; i += kBulkThreads) {
      float v = 0.f;
      if (tt < a.tcount) {
        if (m == 0 || a.x_rest == nullptr)
          v = a.x0_el ? Elem<EL>::load((const EL*)a.x0, (int64_t)t * a.x0_tok_stride + i)
                      : ((const float*)a.x0)[(int64_t)t * a.x0_tok_stride + i];
        else
          v = a.x_rest[(int64_t)t * a.x_rest_tok_stride + (int64_t)(m - 1) * a.x_rest_mat_stride + i];
      }
      xs[tt * d + i] = v;
    }
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kBulkStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, kBulkConsumers);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_chunks = (d + CW - 1) / CW;
  const int n_groups = (a.n_rows + kBulkConsumers - 1) / kBulkConsumers;
  const int my_groups = n_groups > (int)blockIdx.x ? (n_groups - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  const int total = my_groups * n_chunks;

  if (warp == kBulkConsumers) {                      // producer
    if (lane == 0) {
      for (int it = 0; it < total; ++it) {
        const int s = it % kBulkStages, ph = (it / kBulkStages) & 1;
        if (!mbar_wait(empty0 + 8 * s, ph ^ 1)) { atomicExch(err, 1); break; }
        const int g = blockIdx.x + (it / n_chunks) * gridDim.x, c = it % n_chunks;
        const int rows = min(kBulkConsumers, a.n_rows - g * kBulkConsumers);
        const int cols = min(CW, d - c * CW);
        const uint32_t bytes = (uint32_t)cols * sizeof(EL);
        mbar_expect_tx(full0 + 8 * s, bytes * rows);
        for (int r = 0; r < rows; ++r)
          bulk_copy_g2s(smem_u32(ring + (s * kBulkConsumers + r) * kBulkSegBytes),
                        W + (int64_t)(g * kBulkConsumers + r) * d + (int64_t)c * CW, bytes, full0 + 8 * s);
      }
    }
    return;
  }

  float acc[TT];
#pragma unroll
  for (int t = 0; t < TT; ++t) acc[t] = 0.f;
  for (int it = 0; it < total; ++it) {
    const int s = it % kBulkStages, ph = (it / kBulkStages) & 1;
    const bool timed_out = !mbar_wait(full0 + 8 * s, ph);
    if (__any_sync(0xffffffffu, timed_out)) { if (lane == 0) atomicExch(err, 1); break; }
    const int g = blockIdx.x + (it / n_chunks) * gridDim.x, c = it % n_chunks;
    const int row = g * kBulkConsumers + warp;
    if (row < a.n_rows) {
      const int cols = min(CW, d - c * CW);
      const uint8_t* seg = ring + (s * kBulkConsumers + warp) * kBulkSegBytes;
      const float* xc = xs + c * CW;
#pragma unroll 4
      for (int j = lane; j < cols / EPV; j += 32) {
        float wf[EPV];
        Elem<EL>::unpack(*reinterpret_cast<const uint4*>(seg + j * 16), wf);
#pragma unroll
        for (int t = 0; t < TT; ++t) {
          const float4* xp = reinterpret_cast<const float4*>(xc + t * d + j * EPV);
#pragma unroll
          for (int e4 = 0; e4 < EPV / 4; ++e4) {
            const float4 x4 = xp[e4];
            acc[t] = fmaf(wf[4 * e4], x4.x, acc[t]);
            acc[t] = fmaf(wf[4 * e4 + 1], x4.y, acc[t]);
            acc[t] = fmaf(wf[4 * e4 + 2], x4.z, acc[t]);
            acc[t] = fmaf(wf[4 * e4 + 3], x4.w, acc[t]);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * s);      // this warp is done with the stage
    if (c == n_chunks - 1) {
#pragma unroll
      for (int t = 0; t < TT; ++t) acc[t] = warp_sum(acc[t]);
      if (lane == 0 && row < a.n_rows) {
#pragma unroll
        for (int t = 0; t < TT; ++t) {
          if (t >= a.tcount) continue;
          float v = acc[t];
          if (a.resid) {
            if (a.b1) v += Elem<EL>::load((const EL*)a.b1, (int64_t)m * d + row);
            v = xs[t * d + row] + v / (1.f + expf(-v));    // h + SiLU(W1 h + b1)
          }
          a.out[(int64_t)(a.t0 + t) * a.out_tok_stride + (int64_t)m * a.out_mat_stride + row] = v;
        }
      }
#pragma unroll
      for (int t = 0; t < TT; ++t) acc[t] = 0.f;
    }
  }
}

// ---- top-k -------------------------------------------------------------------

struct Cand {
  float v;
  int i;
};

// Top-k of the logits rows (row = t * (K + 1) + m), each row split over gridDim.x CTAs.
// Every warp of a CTA scans a slice of the CTA's span and keeps its own top-k sorted
// across its lanes (lane i holds the i-th best, value desc, id asc); a value enters
// only when it ranks before the current k-th entry (a ballot over 32 values at a time,
// rare after the first few hundred values), so the scan runs at load speed.  The CTA
// merges its warps' lists and publishes them; the last CTA of the row (a ticket it
// resets) merges all spans into root (m = 0, top-1) or pool.
__device__ __forceinline__ void topk_insert(float v, int id, int kk, float& lv, int& li) {
  const int lane = threadIdx.x & 31;
  const bool before = lane < kk && ranks_before(v, id, lv, li);
  const unsigned mask = __ballot_sync(0xffffffffu, before);
  if (mask) {
    const int pos = __ffs(mask) - 1;
    const float uv = __shfl_up_sync(0xffffffffu, lv, 1);
    const int ui = __shfl_up_sync(0xffffffffu, li, 1);
    if (lane == pos) { lv = v; li = id; }
    else if (lane > pos && lane < kk) { lv = uv; li = ui; }
  }
}

// Merge n sorted lists of kk entries (list l at lists[l * stride], l < n <= 64) into
// the first kk entries of the union; warp-wide, every lane gets the result r in round r.
template <typename Load>
__device__ __forceinline__ void merge_lists(int n, int kk, Load load, float* out_v, int* out_i) {
  const int lane = threadIdx.x & 31;
  int hp[2] = {0, 0};
  Cand head[2];
#pragma unroll
  for (int q = 0; q < 2; ++q) head[q] = lane + 32 * q < n ? load(lane + 32 * q, 0) : Cand{-INFINITY, INT_MAX};
  for (int r = 0; r < kk; ++r) {
    int qb = (head[1].i != INT_MAX && (head[0].i == INT_MAX || ranks_before(head[1].v, head[1].i, head[0].v, head[0].i))) ? 1 : 0;
    float bv = head[qb].v;
    int bi = head[qb].i;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ranks_before(ov, oi, bv, bi)) { bv = ov; bi = oi; }
    }
    if (bi != INT_MAX && head[qb].i == bi) {
      ++hp[qb];
      head[qb] = hp[qb] < kk ? load(lane + 32 * qb, hp[qb]) : Cand{-INFINITY, INT_MAX};
    }
    out_v[r] = bv;
    out_i[r] = bi;
  }
}

// Orderable 64-bit key of a candidate: a larger key ranks before (higher value, then
// lower id); -0 counts as +0, as in ranks_before.
__device__ __forceinline__ unsigned long long rank_key(float v, int i) {
  if (v == 0.f) v = 0.f;
  const uint32_t b = __float_as_uint(v);
  const uint32_t ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return ((unsigned long long)ord << 32) | (0xFFFFFFFFu - (uint32_t)i);
}

__global__ void __launch_bounds__(kThreads) topk_rows_kernel(const float* __restrict__ logits, int V, int topk,
                                                             int Kp1, int span, Cand* __restrict__ cand,
                                                             int* __restrict__ tick, int32_t* __restrict__ root,
                                                             int32_t* __restrict__ pool, const int* __restrict__ err) {
  __shared__ Cand lists[kWarps][32];
  __shared__ Cand spans[kTopkMaxSpans * 32];
  __shared__ float mv[32];
  __shared__ int mi[32];
  __shared__ int last;
  // The best k-th entry over the warps' lists: every warp's k-th entry is beaten by k
  // values of the span, so no value that does not beat the best of them is in the
  // span's top k.  Warps publish theirs (atomicMax of rank_key) and filter by it.
  __shared__ unsigned long long s_thr;
  if (threadIdx.x == 0) s_thr = 0ull;
  __syncthreads();
  const int row = blockIdx.y, c = blockIdx.x, ns = gridDim.x;
  const int t = row / Kp1, m = row % Kp1;
  const int kk = m == 0 ? 1 : topk;
  const float* src = logits + (int64_t)row * V;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c_lo = c * span, c_hi = min(V, c_lo + span);
  float lv = -INFINITY;
  int li = INT_MAX;
  // The current k-th entry (the admission threshold) is kept in registers and
  // refreshed only after an insertion.
  float tv = -INFINITY;
  int ti = INT_MAX;
  unsigned long long own = 0ull;  // rank_key of (tv, ti) once the list is full
  bool filled = false;            // warp-uniform: the list has been seeded
  // warp w scans part of [c_lo, c_hi); 128 values per step as one float4 per lane when
  // rows are 16-byte aligned (span is a multiple of 128 then)
  auto offer = [&](float v, int i, bool valid) {
    if (!filled) {
      // the first 32 values seed the list: one bitonic sort across the warp (best
      // first) instead of up to 32 single insertions
      float sv = valid ? v : -INFINITY;
      int si = valid ? i : INT_MAX;
#pragma unroll
      for (int k = 2; k <= 32; k <<= 1)
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, sv, j);
          const int oi = __shfl_xor_sync(0xffffffffu, si, j);
          const bool best_first = (lane & k) == 0 || k == 32;   // direction of this block
          const bool lower = (lane & j) == 0;
          const bool o_better = ranks_before(ov, oi, sv, si);
          if ((lower == best_first) ? o_better : (!o_better && (ov != sv || oi != si))) { sv = ov; si = oi; }
        }
      lv = lane < kk ? sv : -INFINITY;
      li = lane < kk ? si : INT_MAX;
      tv = __shfl_sync(0xffffffffu, lv, kk - 1);
      ti = __shfl_sync(0xffffffffu, li, kk - 1);
      if (ti != INT_MAX) {
        own = rank_key(tv, ti);
        if (lane == 0) atomicMax(&s_thr, own);
      }
      filled = true;
      return;
    }
    const unsigned long long shared_thr = *reinterpret_cast<volatile unsigned long long*>(&s_thr);
    const unsigned long long thr = own > shared_thr ? own : shared_thr;
    unsigned cm = __ballot_sync(0xffffffffu, valid && rank_key(v, i) > thr && ranks_before(v, i, tv, ti));
    if (cm) {
      do {
        const int sl = __ffs(cm) - 1;
        cm &= cm - 1;
        topk_insert(__shfl_sync(0xffffffffu, v, sl), __shfl_sync(0xffffffffu, i, sl), kk, lv, li);
      } while (cm);
      tv = __shfl_sync(0xffffffffu, lv, kk - 1);
      ti = __shfl_sync(0xffffffffu, li, kk - 1);
      if (ti != INT_MAX) {
        own = rank_key(tv, ti);
        if (lane == 0) atomicMax(&s_thr, own);
      }
    }
  };
  if ((V & 3) == 0) {
    // Chunks of 32 values per lane (eight float4, all loaded before any is used).  The
    // k-th largest of the 32 lanes' maxima bounds the chunk's k-th best from below (k
    // distinct values reach it), so only values at or above it can enter the list:
    // about k per chunk instead of every value that beats a fresh list's threshold.
    constexpr int kVec = 8;
    filled = true;                 // the lists start empty: the bound seeds them
    for (int base = c_lo + 128 * warp; base < c_hi; base += 128 * kWarps * kVec) {
      float x[4 * kVec];
#pragma unroll
      for (int u = 0; u < kVec; ++u) {
        const int i0 = base + 128 * kWarps * u + 4 * lane;
        const float4 q = i0 < c_hi ? __ldg(reinterpret_cast<const float4*>(src + i0))
                                   : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        x[4 * u] = q.x; x[4 * u + 1] = q.y; x[4 * u + 2] = q.z; x[4 * u + 3] = q.w;
      }
      float lm = -INFINITY;
#pragma unroll
      for (int e = 0; e < 4 * kVec; ++e) lm = fmaxf(lm, x[e]);
      // k-th largest lane maximum: bitonic sort of the 32 maxima, largest first
#pragma unroll
      for (int k = 2; k <= 32; k <<= 1)
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
          const float o = __shfl_xor_sync(0xffffffffu, lm, j);
          const bool best_first = (lane & k) == 0 || k == 32;
          const bool lower = (lane & j) == 0;
          lm = (lower == best_first) ? fmaxf(lm, o) : fminf(lm, o);
        }
      const float bound = __shfl_sync(0xffffffffu, lm, kk - 1);
#pragma unroll
      for (int e = 0; e < 4 * kVec; ++e) {
        const int id = base + 128 * kWarps * (e >> 2) + 4 * lane + (e & 3);
        unsigned cm = __ballot_sync(0xffffffffu, x[e] >= bound && id < c_hi);
        if (cm) {
          const unsigned long long shared_thr = *reinterpret_cast<volatile unsigned long long*>(&s_thr);
          const unsigned long long thr = own > shared_thr ? own : shared_thr;
          cm = __ballot_sync(0xffffffffu, ((cm >> lane) & 1u) && rank_key(x[e], id) > thr &&
                                              ranks_before(x[e], id, tv, ti));
          if (cm) {
            do {
              const int sl = __ffs(cm) - 1;
              cm &= cm - 1;
              topk_insert(__shfl_sync(0xffffffffu, x[e], sl), __shfl_sync(0xffffffffu, id, sl), kk, lv, li);
            } while (cm);
            tv = __shfl_sync(0xffffffffu, lv, kk - 1);
            ti = __shfl_sync(0xffffffffu, li, kk - 1);
            if (ti != INT_MAX) {
              own = rank_key(tv, ti);
              if (lane == 0) atomicMax(&s_thr, own);
            }
          }
        }
      }
    }
  } else {
    for (int base = c_lo + 32 * warp; base < c_hi; base += 32 * kWarps) {
      const int i = base + lane;
      offer(i < c_hi ? __ldg(src + i) : -INFINITY, i, i < c_hi);
    }
  }
  lists[warp][lane] = Cand{lv, li};
  __syncthreads();
  if (warp == 0) {
    merge_lists(kWarps, kk, [&](int l, int e) { return lists[l][e]; }, mv, mi);
    __syncwarp();
    Cand* out = cand + ((int64_t)row * ns + c) * topk;
    if (lane < kk) out[lane] = Cand{mv[lane], mi[lane]};
    __threadfence();
    __syncwarp();
    int tk = 0;
    if (lane == 0) tk = atomicAdd(&tick[row], 1);
    tk = __shfl_sync(0xffffffffu, tk, 0);
    last = tk == ns - 1;
  }
  __syncthreads();
  if (!last) return;
  // the last CTA of the row: stage every span's list in shared memory (all loads in
  // flight at once), then merge them
  __threadfence();
  const Cand* rl = cand + (int64_t)row * ns * topk;
  for (int e = threadIdx.x; e < ns * kk; e += kThreads) {
    const int l = e / kk, r = e % kk;
    const float2 f = __ldcg(reinterpret_cast<const float2*>(rl + (int64_t)l * topk + r));
    spans[l * kk + r] = Cand{f.x, __float_as_int(f.y)};
  }
  __syncthreads();
  if (warp != 0) return;
  merge_lists(ns, kk, [&](int l, int e) { return spans[l * kk + e]; }, mv, mi);
  __syncwarp();
  if (lane == 0) {
    const bool bad = *reinterpret_cast<const volatile int*>(err) != 0;   // a weight-stream wait gave up
    for (int r = 0; r < kk; ++r) {
      const int id = (bad || mi[r] == INT_MAX) ? -1 : mi[r];
      if (m == 0) root[t] = id;
      else pool[((int64_t)t * (Kp1 - 1) + (m - 1)) * topk + r] = id;
    }
    tick[row] = 0;                                       // ready for the next call
  }
}

template <typename EL, int TT, int R, int U>
cudaError_t run_gemv(const GemvArgs& a, int n_mats, cudaStream_t st) {
  const size_t smem = (size_t)TT * a.d * sizeof(float);
  auto kern = gemv_kernel<EL, TT, R, U>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0, sms = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const int groups = (a.n_rows + kWarps * R - 1) / (kWarps * R);
  int gx = (sms * per_sm + n_mats - 1) / n_mats;
  if (gx > groups) gx = groups;
  if (gx < 1) gx = 1;
  kern<<<dim3(gx, n_mats), kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

template <typename EL>
cudaError_t gemv_dispatch(int TT, const GemvArgs& a, int n_mats, cudaStream_t st) {
  switch (TT) {
    case 1: return run_gemv<EL, 1, 2, 8>(a, n_mats, st);
    case 2: return run_gemv<EL, 2, 2, 8>(a, n_mats, st);
    case 4: return run_gemv<EL, 4, 4, 4>(a, n_mats, st);
    case 8: return run_gemv<EL, 8, 4, 4>(a, n_mats, st);
    default: return run_gemv<EL, 16, 4, 4>(a, n_mats, st);
  }
}

template <typename EL, int TT, int NS>
cudaError_t run_gemv_bulk(const GemvArgs& a, int n_mats, int* err, cudaStream_t st) {
  const size_t smem = bulk_smem_bytes(TT, a.d, NS);
  auto kern = gemv_bulk_kernel<EL, TT, NS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int sms = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int groups = (a.n_rows + kBulkConsumers - 1) / kBulkConsumers;
  int gx = sms / n_mats;
  if (gx < 1) gx = 1;
  if (gx > groups) gx = groups;
  kern<<<dim3(gx, n_mats), kBulkThreads, smem, st>>>(a, err);
  return cudaGetLastError();
}

constexpr size_t kSmemOptin = 227 * 1024;

// T <= 2 and an input row that fits next to the ring: the bulk-copy kernel (three
// stages when they fit); else the register-blocked kernel.
template <typename EL>
cudaError_t gemv_any(int TT, const GemvArgs& a, int n_mats, int* err, cudaStream_t st) {
  if (TT <= 2 && (size_t)TT * a.d * 4 <= 64 * 1024) {
    const bool three = bulk_smem_bytes(TT, a.d, 3) <= kSmemOptin;
    if (TT == 1) return three ? run_gemv_bulk<EL, 1, 3>(a, n_mats, err, st) : run_gemv_bulk<EL, 1, 2>(a, n_mats, err, st);
    return three ? run_gemv_bulk<EL, 2, 3>(a, n_mats, err, st) : run_gemv_bulk<EL, 2, 2>(a, n_mats, err, st);
  }
  return gemv_dispatch<EL>(TT, a, n_mats, st);
}


int pow2_at_least(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

}  // namespace

HeadsPlan plan_heads(int T, int d, int V, int K, int topk) {
  HeadsPlan p{};
  p.T = T; p.d = d; p.V = V; p.K = K; p.topk = topk;
  const size_t smem_budget = 160 * 1024;
  int fit = (int)(smem_budget / ((size_t)d * sizeof(float)));
  if (fit > 16) fit = 16;
  if (fit < 1) fit = 1;
  int tpp = T < fit ? T : fit;
  // round down to a supported tile (1, 2, 4, 8, 16)
  int tile = 1;
  while (tile * 2 <= tpp) tile *= 2;
  p.tokens_per_pass = tile;
  size_t off = 0;
  p.off_z = off;
  off = align_up(off + (size_t)T * K * d * sizeof(float), 256);
  p.off_logits = off;
  off = align_up(off + (size_t)T * (K + 1) * V * sizeof(float), 256);
  p.off_scand = off;                                       // weight-stream path: per-CTA lists
  off = align_up(off + (size_t)(K + 1) * kHeadsStreamMaxGrid * topk * sizeof(Cand), 256);
  // tensor-core path: z of one pass (bf16 pairs of at most kHeadsMmaMaxRows rows, or
  // wide: single fp16 rows, at most kHeadsMmaWideRows); h is read in place
  const bool wide = heads_mma_wide(T);
  const int per_pass = wide ? kHeadsMmaWideRows : kHeadsMmaMaxRows;
  const int Tp = T < per_pass ? T : per_pass;
  p.off_zhl = off;
  off = align_up(off + (T >= 2 ? (size_t)K * heads_mma_rows(Tp, wide) * d * 2 : 0), 256);
  p.off_cand = off;                                        // top-k: per-span sorted lists
  off = align_up(off + (size_t)T * (K + 1) * kTopkMaxSpans * topk * sizeof(Cand), 256);
  p.off_err = off;                                         // error flag and counters, then tickets
  off = align_up(off + kHeadsCounterBytes + (size_t)T * (K + 1) * sizeof(int), 256);
  p.bytes = off;
  (void)pow2_at_least;
  return p;
}

cudaError_t launch_heads(const HeadsPlan& p, const void* h, const void* w1, const void* b1,
                         const void* w2, int64_t w2_stride, const void* w_lm, medusa_dtype dt,
                         int32_t* root, int32_t* pool, float* logits_out, void* ws,
                         cudaStream_t st) {
  char* base = (char*)ws;
  float* z = (float*)(base + p.off_z);
  float* logits = logits_out ? logits_out : (float*)(base + p.off_logits);
  int* err = (int*)(base + p.off_err);
  const int d = p.d, V = p.V, K = p.K, T = p.T;
  // One hidden row in bf16: the persistent weight stream with in-stream top-k.
  if (heads_stream_supported(T, d, V, K, p.topk, dt, h, w1, w2, w2_stride, w_lm, b1))
    return launch_heads_stream(p, h, w1, b1, w2, w2_stride, w_lm, root, pool, logits_out, ws, st);
  const size_t esz = dt == MEDUSA_BF16 ? 2 : 4;
  const int rows = T * (K + 1);
  // error flag, counters and top-k tickets start at zero
  cudaError_t e = cudaMemsetAsync(err, 0, kHeadsCounterBytes + (size_t)rows * sizeof(int), st);
  if (e != cudaSuccess) return e;
  if (heads_mma_supported(T, d, V, K, dt, h, w1, w2, w2_stride, w_lm)) {
    // several bf16 hidden rows: tensor-core weight stream (passes of at most
    // kHeadsMmaMaxRows rows as pairs, or kHeadsMmaWideRows wide, each reading the weights
    // once), then top-k on the logits
    const bool wide = heads_mma_wide(T);
    const int per_pass = wide ? kHeadsMmaWideRows : kHeadsMmaMaxRows;
    for (int t0 = 0; t0 < T; t0 += per_pass) {
      HeadsPlan pp = p;
      pp.T = (T - t0) < per_pass ? (T - t0) : per_pass;
      if (t0 > 0) {                // the pass's work counters start at zero; the error flag stays
        e = cudaMemsetAsync(err + 4, 0, kHeadsCounterBytes - 4 * sizeof(int), st);
        if (e != cudaSuccess) return e;
      }
      e = launch_heads_mma(pp, wide, (const uint16_t*)h + (size_t)t0 * d, w1, b1, w2, w2_stride, w_lm,
                           logits + (size_t)t0 * (K + 1) * V, ws, st);
      if (e != cudaSuccess) return e;
    }
  } else {
  for (int t0 = 0; t0 < T; t0 += p.tokens_per_pass) {
    const int tc = (T - t0) < p.tokens_per_pass ? (T - t0) : p.tokens_per_pass;
    // 1. residual block per head: rows i of W1_k, x = h
    GemvArgs r{};
    r.w0 = w1;
    r.w_rest = (const char*)w1 + (size_t)d * d * esz;
    r.w_rest_stride = (int64_t)d * d;
    r.n_rows = d; r.d = d;
    r.x0 = h; r.x0_el = 1; r.x0_tok_stride = d;
    r.x_rest = nullptr;
    r.t0 = t0; r.tcount = tc;
    r.out = z; r.out_tok_stride = (int64_t)K * d; r.out_mat_stride = d;
    r.resid = 1; r.b1 = b1;
    if (K > 0) {
      e = dt == MEDUSA_BF16 ? gemv_any<uint16_t>(p.tokens_per_pass, r, K, err, st)
                            : gemv_any<float>(p.tokens_per_pass, r, K, err, st);
      if (e != cudaSuccess) return e;
    }
    // 2. vocabulary projections: matrix 0 = LM head on h, matrix 1 + k = W2_k on z_k
    GemvArgs g{};
    g.w0 = w_lm;
    g.w_rest = w2;
    g.w_rest_stride = w2_stride;
    g.n_rows = V; g.d = d;
    g.x0 = h; g.x0_el = 1; g.x0_tok_stride = d;
    g.x_rest = z; g.x_rest_tok_stride = (int64_t)K * d; g.x_rest_mat_stride = d;
    g.t0 = t0; g.tcount = tc;
    g.out = logits; g.out_tok_stride = (int64_t)(K + 1) * V; g.out_mat_stride = V;
    g.resid = 0; g.b1 = nullptr;
    e = dt == MEDUSA_BF16 ? gemv_any<uint16_t>(p.tokens_per_pass, g, K + 1, err, st)
                          : gemv_any<float>(p.tokens_per_pass, g, K + 1, err, st);
    if (e != cudaSuccess) return e;
  }
  }
  // 3. top-k, one CTA per (row t, matrix m)
  int sms = 148, dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int ns = (2 * sms + rows - 1) / rows;                    // spans per row: about two CTAs per SM
  if (ns > kTopkMaxSpans) ns = kTopkMaxSpans;
  if (ns > (V + 1023) / 1024) ns = (V + 1023) / 1024;      // at least ~1024 logits per span
  if (ns < 1) ns = 1;
  const int span = ((V + ns - 1) / ns + 127) / 128 * 128;
  ns = (V + span - 1) / span;
  topk_rows_kernel<<<dim3(ns, rows), kThreads, 0, st>>>(logits, V, p.topk, K + 1, span, (Cand*)(base + p.off_cand),
                                                        err + kHeadsCounterBytes / sizeof(int), root, pool, err);
  return cudaGetLastError();
}

}  // namespace medusa
