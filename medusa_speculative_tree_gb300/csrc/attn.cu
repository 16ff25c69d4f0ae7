// Tree verification attention ([M7.2] §0x03, §0x03C, §0x03E; [CN] "Tree Attention";
// [Math] "Tree attention: the mask math").
//
// Work decomposition shared by both kernels.  For sequence b and KV head kvh the
// M = N * g query rows (tree row u, group member gi; query head kvh * g + gi) share
// one K/V stream.  Rows are cut into m-tiles; the committed prefix [0, L) is cut
// into n_split key ranges.  CTA (split, m-tile, b * Hkv + kvh):
//   - rotates its queries (RoPE at L + depth[u]) and, for split 0, stages the
//     rotated tree keys and the tree values at cache rows L + u;
//   - runs an online-softmax pass over its prefix key range (no mask: every
//     committed key is visible) and writes an unnormalised partial (O, m, l);
//   - takes a ticket; the last CTA of the (b, kvh, m-tile) unit merges all
//     partials, adds the tree block (ancestors from the multiword bitmask, fp32),
//     normalises and writes the output.  It then resets the unit's counter.
// Softmax runs in the log2 domain (scores pre-multiplied by scale * log2 e).
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace medusa {

// Declared in attn_tc.cu.
cudaError_t launch_attn_tc(const AttnPlan& p, const medusa_tree_t& t, const void* q,
                           const void* k_new, const void* v_new, const medusa_kv_t& c,
                           const int32_t* L, const float* th_hi, const float* th_lo,
                           float scale_log2, float* out, float* lse, int32_t* status, void* ws,
                           cudaStream_t st);
bool attn_tc_supported(const medusa_tree_t& t, int Hq, const medusa_kv_t& c);
void attn_tc_plan(AttnPlan& p);

namespace {

constexpr int kSimtThreads = 128;
constexpr int kSimtRows = 16;   // 4 warps x 4 rows
constexpr int kSimtKT = 32;     // keys per tile
constexpr int kAncGroup = 4;    // tree-block ancestors whose rows are loaded together

struct SimtArgs {
  medusa_tree_t t;
  medusa_kv_t c;
  const void* q;
  const void* k_new;
  const void* v_new;
  const int32_t* L;
  float* out;
  float* lse;
  int32_t* status;
  int* counter;
  float* part_o;
  float* part_ml;
  int Hq, Hkv, g, n_mt, n_split, chunk;
  float scale_log2;
  float th_hi[64], th_lo[64];
};

__device__ __forceinline__ int64_t row_off(const medusa_kv_t& c, int b, int kvh, int row) {
  if (c.page_size == 0)
    return (((int64_t)b * c.n_kv_heads + kvh) * c.capacity + row) * c.head_dim;
  const int page = c.block_table[(int64_t)b * c.max_blocks + row / c.page_size];
  return (((int64_t)page * c.n_kv_heads + kvh) * c.page_size + row % c.page_size) * c.head_dim;
}

template <typename EL, int DH>
__global__ void __launch_bounds__(kSimtThreads) attn_simt_kernel(SimtArgs a) {
  constexpr int HALF = DH / 2;
  constexpr int PER_LANE = DH / 32;
  constexpr int EPV = Elem<EL>::kPerVec;
  extern __shared__ __align__(16) float smem[];
  const int D = a.t.max_depth;                        // (a bound over the batch with per-sequence templates)
  float* tab_c = smem;                                // [(D+1)][HALF]
  float* tab_s = tab_c + (D + 1) * HALF;
  float* qs = tab_s + (D + 1) * HALF;                 // [kSimtRows][DH]
  float* kts = qs + kSimtRows * DH;                   // [DH][kSimtKT + 1]
  float* vs = kts + DH * (kSimtKT + 1);               // [kSimtKT][DH]
  __shared__ int last_flag;

  const int s = blockIdx.x, mt = blockIdx.y;
  const int b = blockIdx.z / a.Hkv, kvh = blockIdx.z % a.Hkv;
  // NS: row stride of q, k_new, v_new, out (the batch's bound); N: this sequence's rows
  const medusa_tree_t t = seq_tree(a.t, b);
  const int NS = a.t.n_rows, N = t.n_rows, g = a.g, M = N * g;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const EL* q = (const EL*)a.q;
  const EL* kn = (const EL*)a.k_new;
  const EL* vn = (const EL*)a.v_new;
  // The elements this thread rotates (its query pairs and, in split 0, the pairs of the
  // tree keys and values it stages) are loaded with L, before anything waits on them:
  // one memory round trip for the whole prologue instead of one per loop iteration.
  constexpr int QIT = kSimtRows * HALF / kSimtThreads;
  static_assert(QIT * kSimtThreads == kSimtRows * HALF, "whole (row, pair) items per thread");
  float qx1[QIT], qx2[QIT], kx1[QIT], kx2[QIT];
  EL vx1[QIT], vx2[QIT];
  int rdep[QIT];
#pragma unroll
  for (int it = 0; it < QIT; ++it) {
    const int idx = tid + it * kSimtThreads;
    const int r = idx / HALF, i = idx % HALF;
    const int R = mt * kSimtRows + r;
    qx1[it] = qx2[it] = kx1[it] = kx2[it] = 0.f;
    vx1[it] = vx2[it] = EL(0);
    rdep[it] = 0;
    if (R < M) {
      const int u = R / g, h = kvh * g + R % g;
      const int64_t base = (((int64_t)b * NS + u) * a.Hq + h) * DH;
      qx1[it] = Elem<EL>::load(q, base + i);
      qx2[it] = Elem<EL>::load(q, base + i + HALF);
      rdep[it] = t.depth[u];
      if (s == 0 && R % g == 0) {
        const int64_t src = (((int64_t)b * NS + u) * a.Hkv + kvh) * DH;
        kx1[it] = Elem<EL>::load(kn, src + i);
        kx2[it] = Elem<EL>::load(kn, src + i + HALF);
        vx1[it] = vn[src + i];
        vx2[it] = vn[src + i + HALF];
      }
    }
  }
  const int Lb = a.L[b];
  if (mt * kSimtRows >= M) return;        // a row tile past this sequence's rows: the whole unit
  const bool first_cta = (s == 0 && mt == 0 && kvh == 0 && tid == 0);
  if (Lb < 0 || !seq_rows_ok(a.c, b, (int64_t)Lb + N)) {
    if (first_cta) a.status[b] = MEDUSA_ECAPACITY;
    return;
  }
  if (Lb > a.n_split * a.chunk) {           // max_prefix was below this sequence's length
    if (first_cta) a.status[b] = MEDUSA_EINVAL;
    return;
  }
  if (first_cta) a.status[b] = MEDUSA_OK;

  // RoPE table for the D + 1 distinct positions L + depth.
  for (int idx = tid; idx < (D + 1) * HALF; idx += kSimtThreads) {
    const int dep = idx / HALF, i = idx % HALF;
    float sn, cs;
    sincosf(rope_angle(Lb + dep, a.th_hi[i], a.th_lo[i]), &sn, &cs);
    tab_c[idx] = cs;
    tab_s[idx] = sn;
  }
  __syncthreads();

  // Rotated queries of this m-tile; in split 0 the rotated tree keys and the tree
  // values at cache rows L + u.  The destination rows are looked up first (a paged
  // cache reads its block table), then every store follows.
  EL* ck = (EL*)a.c.k;
  EL* cv = (EL*)a.c.v;
  int64_t dst[QIT];
#pragma unroll
  for (int it = 0; it < QIT; ++it) {
    const int R = mt * kSimtRows + (tid + it * kSimtThreads) / HALF;
    dst[it] = (s == 0 && R < M && R % g == 0) ? row_off(a.c, b, kvh, Lb + R / g) : -1;
  }
#pragma unroll
  for (int it = 0; it < QIT; ++it) {
    const int idx = tid + it * kSimtThreads;
    const int r = idx / HALF, i = idx % HALF;
    const int R = mt * kSimtRows + r;
    const int ti = rdep[it] * HALF + i;
    const float cs = tab_c[ti], sn = tab_s[ti];
    qs[r * DH + i] = R < M ? qx1[it] * cs - qx2[it] * sn : 0.f;
    qs[r * DH + i + HALF] = R < M ? qx2[it] * cs + qx1[it] * sn : 0.f;
    if (dst[it] >= 0) {
      const int64_t d0 = dst[it];
      const float y1 = kx1[it] * cs - kx2[it] * sn, y2 = kx2[it] * cs + kx1[it] * sn;
      Elem<EL>::store(ck, d0 + i, y1);
      Elem<EL>::store(ck, d0 + i + HALF, y2);
      cv[d0 + i] = vx1[it];
      cv[d0 + i + HALF] = vx2[it];
      if constexpr (sizeof(EL) == 2) {
        if (a.c.k_f16) {                          // the fp16 mirror of the rows just written
          uint16_t* mk = (uint16_t*)a.c.k_f16;
          uint16_t* mv = (uint16_t*)a.c.v_f16;
          mk[d0 + i] = bf16_bits_to_f16_bits(f32_to_bf16_bits(y1));
          mk[d0 + i + HALF] = bf16_bits_to_f16_bits(f32_to_bf16_bits(y2));
          mv[d0 + i] = bf16_bits_to_f16_bits(vx1[it]);
          mv[d0 + i + HALF] = bf16_bits_to_f16_bits(vx2[it]);
        }
      }
    }
  }
  __syncthreads();

  // Online softmax over this split's prefix keys.
  float m_r[4], l_r[4], o_r[4][PER_LANE];
#pragma unroll
  for (int rr = 0; rr < 4; ++rr) {
    m_r[rr] = -INFINITY;
    l_r[rr] = 0.f;
#pragma unroll
    for (int c = 0; c < PER_LANE; ++c) o_r[rr][c] = 0.f;
  }
  const int k_begin = s * a.chunk;
  const int k_end = min(Lb, k_begin + a.chunk);
  const EL* ckr = (const EL*)a.c.k;
  const EL* cvr = (const EL*)a.c.v;
  for (int kt0 = k_begin; kt0 < k_end; kt0 += kSimtKT) {
    // The tile's 16-byte vectors of this thread: all loads first (keys past the range
    // read as zeros), then the stores into shared memory.
    constexpr int VEC_PER_ROW = DH / EPV;
    constexpr int KIT = kSimtKT * VEC_PER_ROW / kSimtThreads;
    static_assert(KIT * kSimtThreads == kSimtKT * VEC_PER_ROW, "whole vectors per thread");
    uint4 kraw[KIT], vraw[KIT];
#pragma unroll
    for (int it = 0; it < KIT; ++it) {
      const int idx = tid + it * kSimtThreads;
      const int key = kt0 + idx / VEC_PER_ROW;
      kraw[it] = vraw[it] = make_uint4(0u, 0u, 0u, 0u);
      if (key < k_end) {
        const int64_t off = row_off(a.c, b, kvh, key) + (idx % VEC_PER_ROW) * EPV;
        kraw[it] = *reinterpret_cast<const uint4*>(ckr + off);
        vraw[it] = *reinterpret_cast<const uint4*>(cvr + off);
      }
    }
#pragma unroll
    for (int it = 0; it < KIT; ++it) {
      const int idx = tid + it * kSimtThreads;
      const int j = idx / VEC_PER_ROW, vi = idx % VEC_PER_ROW;
      float kf[EPV], vf[EPV];
      Elem<EL>::unpack(kraw[it], kf);
      Elem<EL>::unpack(vraw[it], vf);
#pragma unroll
      for (int e = 0; e < EPV; ++e) {
        kts[(vi * EPV + e) * (kSimtKT + 1) + j] = kf[e];
        vs[j * DH + vi * EPV + e] = vf[e];
      }
    }
    __syncthreads();
    const bool key_ok = kt0 + lane < k_end;
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int r = warp * 4 + rr;
      if (mt * kSimtRows + r >= M) continue;
      float sc = 0.f;
#pragma unroll 16
      for (int i = 0; i < DH; ++i) sc = fmaf(qs[r * DH + i], kts[i * (kSimtKT + 1) + lane], sc);
      sc = key_ok ? sc * a.scale_log2 : -INFINITY;
      const float m_new = fmaxf(m_r[rr], warp_max(sc));
      const float p = key_ok ? exp2f(sc - m_new) : 0.f;
      const float alpha = (m_r[rr] == -INFINITY) ? 0.f : exp2f(m_r[rr] - m_new);
      l_r[rr] = l_r[rr] * alpha + warp_sum(p);
#pragma unroll
      for (int c = 0; c < PER_LANE; ++c) o_r[rr][c] *= alpha;
#pragma unroll 8
      for (int j = 0; j < kSimtKT; ++j) {
        const float pj = __shfl_sync(0xffffffffu, p, j);
#pragma unroll
        for (int c = 0; c < PER_LANE; ++c) o_r[rr][c] = fmaf(pj, vs[j * DH + lane + 32 * c], o_r[rr][c]);
      }
      m_r[rr] = m_new;
    }
    __syncthreads();
  }

  // Partial of this split.
  const int unit = (b * a.Hkv + kvh) * a.n_mt + mt;
  const int64_t pbase = ((int64_t)unit * a.n_split + s) * kSimtRows;
#pragma unroll
  for (int rr = 0; rr < 4; ++rr) {
    const int r = warp * 4 + rr;
#pragma unroll
    for (int c = 0; c < PER_LANE; ++c) a.part_o[(pbase + r) * DH + lane + 32 * c] = o_r[rr][c];
    if (lane == 0) {
      a.part_ml[(pbase + r) * 2] = m_r[rr];
      a.part_ml[(pbase + r) * 2 + 1] = l_r[rr];
    }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int ticket = atomicAdd(&a.counter[unit], 1);
    last_flag = (ticket == a.n_split - 1);
  }
  __syncthreads();
  if (!last_flag) return;
  if (tid == 0) a.counter[unit] = 0;       // every split has arrived: ready for the next call
  __threadfence();

  // Merge the splits, then add the tree block.  The warp's four rows read their
  // partials together, split by split, and each row reads the K/V rows of up to
  // kAncGroup ancestors before it uses the first: the loads of a group share one
  // memory round trip.  The arithmetic and its order are those of a row-by-row,
  // ancestor-by-ancestor merge.
  float* out = a.out;
  const int W = t.n_words;
  bool live[4];
  float Mx[4], l[4], o[4][PER_LANE];
#pragma unroll
  for (int rr = 0; rr < 4; ++rr) {
    live[rr] = mt * kSimtRows + warp * 4 + rr < M;
    Mx[rr] = -INFINITY;
    l[rr] = 0.f;
#pragma unroll
    for (int c = 0; c < PER_LANE; ++c) o[rr][c] = 0.f;
  }
  for (int s2 = 0; s2 < a.n_split; ++s2) {
    const int64_t pr0 = ((int64_t)unit * a.n_split + s2) * kSimtRows + warp * 4;
#pragma unroll
    for (int rr = 0; rr < 4; ++rr)
      if (live[rr]) Mx[rr] = fmaxf(Mx[rr], __ldcg(&a.part_ml[(pr0 + rr) * 2]));
  }
  for (int s2 = 0; s2 < a.n_split; ++s2) {
    const int64_t pr0 = ((int64_t)unit * a.n_split + s2) * kSimtRows + warp * 4;
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      if (!live[rr]) continue;
      const float ms = __ldcg(&a.part_ml[(pr0 + rr) * 2]);
      const float ps = __ldcg(&a.part_ml[(pr0 + rr) * 2 + 1]);
      float po[PER_LANE];
#pragma unroll
      for (int c = 0; c < PER_LANE; ++c) po[c] = __ldcg(&a.part_o[(pr0 + rr) * DH + lane + 32 * c]);
      const bool empty = ms == -INFINITY;     // a split without keys adds nothing
      const float w = empty ? 0.f : exp2f(ms - Mx[rr]);
      l[rr] = empty ? l[rr] : fmaf(ps, w, l[rr]);
#pragma unroll
      for (int c = 0; c < PER_LANE; ++c) o[rr][c] = empty ? o[rr][c] : fmaf(po[c], w, o[rr][c]);
    }
  }
#pragma unroll
  for (int rr = 0; rr < 4; ++rr) {
    if (!live[rr]) continue;
    const int r = warp * 4 + rr;
    const int R = mt * kSimtRows + r;
    const int u = R / g, h = kvh * g + R % g;
    float mx = Mx[rr], ls = l[rr];
    float qv[PER_LANE];
#pragma unroll
    for (int c = 0; c < PER_LANE; ++c) qv[c] = qs[r * DH + lane + 32 * c];
    for (int wd = 0; wd < W; ++wd) {
      unsigned long long bits = t.anc[(int64_t)u * W + wd];    // the same for the whole warp
      while (bits) {
        int vv[kAncGroup], ti[kAncGroup];
        float kx[kAncGroup][PER_LANE], vx[kAncGroup][PER_LANE];
#pragma unroll
        for (int j = 0; j < kAncGroup; ++j) {
          vv[j] = bits ? wd * 64 + __ffsll((long long)bits) - 1 : -1;
          bits &= bits - 1;
          ti[j] = 0;
#pragma unroll
          for (int c = 0; c < PER_LANE; ++c) kx[j][c] = vx[j][c] = 0.f;
          if (vv[j] >= 0) {
            const int64_t kb = (((int64_t)b * NS + vv[j]) * a.Hkv + kvh) * DH;
            ti[j] = t.depth[vv[j]] * HALF;
#pragma unroll
            for (int c = 0; c < PER_LANE / 2; ++c) {
              kx[j][c] = Elem<EL>::load(kn, kb + lane + 32 * c);
              kx[j][c + PER_LANE / 2] = Elem<EL>::load(kn, kb + lane + 32 * c + HALF);
            }
#pragma unroll
            for (int c = 0; c < PER_LANE; ++c) vx[j][c] = Elem<EL>::load(vn, kb + lane + 32 * c);
          }
        }
#pragma unroll
        for (int j = 0; j < kAncGroup; ++j) {
          if (vv[j] < 0) continue;
          float kr[PER_LANE];
#pragma unroll
          for (int c = 0; c < PER_LANE / 2; ++c) {
            const int i = lane + 32 * c;
            const float x1 = kx[j][c], x2 = kx[j][c + PER_LANE / 2];
            kr[c] = x1 * tab_c[ti[j] + i] - x2 * tab_s[ti[j] + i];
            kr[c + PER_LANE / 2] = x2 * tab_c[ti[j] + i] + x1 * tab_s[ti[j] + i];
          }
          float dot = 0.f;
#pragma unroll
          for (int c = 0; c < PER_LANE; ++c) dot = fmaf(qv[c], kr[c], dot);
          const float sc = warp_sum(dot) * a.scale_log2;
          const float m_new = fmaxf(mx, sc);
          const float alpha = (mx == -INFINITY) ? 0.f : exp2f(mx - m_new);
          const float p = exp2f(sc - m_new);
          ls = ls * alpha + p;
#pragma unroll
          for (int c = 0; c < PER_LANE; ++c) o[rr][c] = fmaf(o[rr][c], alpha, p * vx[j][c]);
          mx = m_new;
        }
      }
    }
    const float inv_l = 1.f / ls;
    const int64_t ob = (((int64_t)b * NS + u) * a.Hq + h) * DH;
#pragma unroll
    for (int c = 0; c < PER_LANE; ++c) out[ob + lane + 32 * c] = o[rr][c] * inv_l;
    if (a.lse && lane == 0) a.lse[((int64_t)b * NS + u) * a.Hq + h] = (mx + log2f(ls)) * kLn2;
  }
}

template <typename EL, int DH>
cudaError_t run_simt(const AttnPlan& p, const SimtArgs& a, cudaStream_t st) {
  const size_t smem = sizeof(float) * ((size_t)2 * (p.D + 1) * (DH / 2) + kSimtRows * DH +
                                       DH * (kSimtKT + 1) + kSimtKT * DH);
  auto kern = attn_simt_kernel<EL, DH>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<dim3(p.n_split, p.n_mt, p.B * p.Hkv), kSimtThreads, smem, st>>>(a);
  return cudaGetLastError();
}

void rope_freqs(int dh, float base, float* hi, float* lo) {
  for (int i = 0; i < dh / 2; ++i) {
    const double th = pow((double)base, -2.0 * i / dh);
    hi[i] = (float)th;
    lo[i] = (float)(th - (double)hi[i]);
  }
}

}  // namespace

size_t attn_units(const AttnPlan& p) { return (size_t)p.B * p.Hkv * p.n_mt; }

AttnPlan plan_attn(const medusa_tree_t& t, int B, int Hq, const medusa_kv_t& c, int max_prefix) {
  AttnPlan p{};
  p.B = B;
  p.Hq = Hq;
  p.Hkv = c.n_kv_heads;
  p.g = Hq / c.n_kv_heads;
  p.dh = c.head_dim;
  p.N = t.n_rows;
  p.D = t.max_depth;
  p.max_prefix = max_prefix;
  p.path = attn_tc_supported(t, Hq, c) ? 1 : 0;
  if (p.path == 1) {
    attn_tc_plan(p);
  } else {
    p.mt_rows = kSimtRows;
    p.key_tile = kSimtKT;
    p.n_mt = (p.N * p.g + kSimtRows - 1) / kSimtRows;
    const int units = B * p.Hkv * p.n_mt;
    const int max_tiles = (max_prefix + kSimtKT - 1) / kSimtKT;
    int want = (4 * 152 + units - 1) / units;
    if (want > max_tiles) want = max_tiles;
    if (want < 1) want = 1;
    int tiles_per = (max_tiles + want - 1) / want;
    if (tiles_per < 1) tiles_per = 1;
    p.chunk = tiles_per * kSimtKT;
    p.n_split = max_prefix > 0 ? (max_prefix + p.chunk - 1) / p.chunk : 1;
    p.first = p.chunk;
  }
  if (p.path == 1) {            // the tensor-core path merges through DSMEM: no scratch
    p.off_counter = p.off_part_o = p.off_part_ml = p.off_tmap = 0;
    p.bytes = 256;
    return p;
  }
  const size_t units = (size_t)B * p.Hkv * p.n_mt;
  // The ticket counters live in a fixed region at the start of the workspace that
  // nothing else ever writes: the last CTA of each unit resets its counter, so the
  // region stays zero across calls whatever their shapes.  Partials follow it.
  size_t off = 0;
  p.off_counter = off;
  off = kAttnCounterBytes;
  p.off_part_o = off;
  off = align_up(off + units * p.n_split * p.mt_rows * p.dh * sizeof(float), 256);
  p.off_part_ml = off;
  off = align_up(off + units * p.n_split * p.mt_rows * 2 * sizeof(float), 256);
  p.off_tmap = off;
  off = align_up(off + (p.path == 1 ? 2 * 128 : 0), 256);
  p.bytes = off;
  return p;
}

cudaError_t launch_attn(const AttnPlan& p, const medusa_tree_t& t, const void* q,
                        const void* k_new, const void* v_new, const medusa_kv_t& c,
                        const int32_t* L, float rope_base, float scale, float* out, float* lse,
                        int32_t* status, void* ws, cudaStream_t st) {
  SimtArgs a{};
  rope_freqs(p.dh, rope_base, a.th_hi, a.th_lo);
  const float scale_log2 = scale * kLog2e;
  if (p.path == 1)
    return launch_attn_tc(p, t, q, k_new, v_new, c, L, a.th_hi, a.th_lo, scale_log2, out, lse,
                          status, ws, st);
  a.t = t;
  a.c = c;
  a.q = q;
  a.k_new = k_new;
  a.v_new = v_new;
  a.L = L;
  a.out = out;
  a.lse = lse;
  a.status = status;
  char* base = (char*)ws;
  a.counter = (int*)(base + p.off_counter);
  a.part_o = (float*)(base + p.off_part_o);
  a.part_ml = (float*)(base + p.off_part_ml);
  a.Hq = p.Hq;
  a.Hkv = p.Hkv;
  a.g = p.g;
  a.n_mt = p.n_mt;
  a.n_split = p.n_split;
  a.chunk = p.chunk;
  a.scale_log2 = scale_log2;
  const bool bf = c.dtype == MEDUSA_BF16;
  if (p.dh == 128) return bf ? run_simt<uint16_t, 128>(p, a, st) : run_simt<float, 128>(p, a, st);
  return bf ? run_simt<uint16_t, 64>(p, a, st) : run_simt<float, 64>(p, a, st);
}

// ---- fixed scratch for medusa_tree_attn_verify_static -----------------------------
// Device memory for callers that cannot allocate: a file-scope array, zero at module
// load.  Host code must not use the symbol itself as a pointer (on the host it only
// names the variable); the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_attn_static_scratch[MEDUSA_ATTN_STATIC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void* g_static_ptr[kMaxDevices] = {};
}  // namespace

cudaError_t attn_static_scratch(void** ptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (g_static_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_attn_static_scratch);   // with `dev` current
    if (e != cudaSuccess) return e;
    g_static_ptr[dev] = p;
  }
  *ptr = g_static_ptr[dev];
  return cudaSuccess;
}

}  // namespace medusa
