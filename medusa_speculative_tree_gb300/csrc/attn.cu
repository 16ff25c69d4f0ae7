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

  const EL* q = (const EL*)a.q;
  const EL* kn = (const EL*)a.k_new;
  const EL* vn = (const EL*)a.v_new;
  // Rotated queries of this m-tile.
  for (int idx = tid; idx < kSimtRows * HALF; idx += kSimtThreads) {
    const int r = idx / HALF, i = idx % HALF;
    const int R = mt * kSimtRows + r;
    float y1 = 0.f, y2 = 0.f;
    if (R < M) {
      const int u = R / g, h = kvh * g + R % g;
      const int64_t base = (((int64_t)b * NS + u) * a.Hq + h) * DH;
      const float x1 = Elem<EL>::load(q, base + i), x2 = Elem<EL>::load(q, base + i + HALF);
      const int ti = t.depth[u] * HALF + i;
      y1 = x1 * tab_c[ti] - x2 * tab_s[ti];
      y2 = x2 * tab_c[ti] + x1 * tab_s[ti];
    }
    qs[r * DH + i] = y1;
    qs[r * DH + i + HALF] = y2;
  }
  // Stage rotated tree keys and tree values at cache rows L + u (split 0 only).
  if (s == 0) {
    EL* ck = (EL*)a.c.k;
    EL* cv = (EL*)a.c.v;
    for (int idx = tid; idx < kSimtRows * HALF; idx += kSimtThreads) {
      const int r = idx / HALF, i = idx % HALF;
      const int R = mt * kSimtRows + r;
      if (R >= M || R % g != 0) continue;
      const int u = R / g;
      const int64_t src = (((int64_t)b * NS + u) * a.Hkv + kvh) * DH;
      const float x1 = Elem<EL>::load(kn, src + i), x2 = Elem<EL>::load(kn, src + i + HALF);
      const int ti = t.depth[u] * HALF + i;
      const int64_t dst = row_off(a.c, b, kvh, Lb + u);
      Elem<EL>::store(ck, dst + i, x1 * tab_c[ti] - x2 * tab_s[ti]);
      Elem<EL>::store(ck, dst + i + HALF, x2 * tab_c[ti] + x1 * tab_s[ti]);
      cv[dst + i] = vn[src + i];
      cv[dst + i + HALF] = vn[src + i + HALF];
      if constexpr (sizeof(EL) == 2) {
        if (a.c.k_f16) {                          // the fp16 mirror of the rows just written
          uint16_t* mk = (uint16_t*)a.c.k_f16;
          uint16_t* mv = (uint16_t*)a.c.v_f16;
          mk[dst + i] = bf16_bits_to_f16_bits(ck[dst + i]);
          mk[dst + i + HALF] = bf16_bits_to_f16_bits(ck[dst + i + HALF]);
          mv[dst + i] = bf16_bits_to_f16_bits(vn[src + i]);
          mv[dst + i + HALF] = bf16_bits_to_f16_bits(vn[src + i + HALF]);
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
    constexpr int VEC_PER_ROW = DH / EPV;
    for (int idx = tid; idx < kSimtKT * VEC_PER_ROW; idx += kSimtThreads) {
      const int j = idx / VEC_PER_ROW, vi = idx % VEC_PER_ROW;
      const int key = kt0 + j;
      float kf[EPV], vf[EPV];
      if (key < k_end) {
        const int64_t off = row_off(a.c, b, kvh, key) + vi * EPV;
        Elem<EL>::unpack(*reinterpret_cast<const uint4*>(ckr + off), kf);
        Elem<EL>::unpack(*reinterpret_cast<const uint4*>(cvr + off), vf);
      } else {
#pragma unroll
        for (int e = 0; e < EPV; ++e) { kf[e] = 0.f; vf[e] = 0.f; }
      }
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

  // Merge the splits, then add the tree block.
  float* out = a.out;
  const int W = t.n_words;
  for (int rr = 0; rr < 4; ++rr) {
    const int r = warp * 4 + rr;
    const int R = mt * kSimtRows + r;
    if (R >= M) continue;
    const int u = R / g, h = kvh * g + R % g;
    float Mx = -INFINITY;
    for (int s2 = 0; s2 < a.n_split; ++s2)
      Mx = fmaxf(Mx, __ldcg(&a.part_ml[(((int64_t)unit * a.n_split + s2) * kSimtRows + r) * 2]));
    float l = 0.f, o[PER_LANE];
#pragma unroll
    for (int c = 0; c < PER_LANE; ++c) o[c] = 0.f;
    for (int s2 = 0; s2 < a.n_split; ++s2) {
      const int64_t pr = ((int64_t)unit * a.n_split + s2) * kSimtRows + r;
      const float ms = __ldcg(&a.part_ml[pr * 2]);
      if (ms == -INFINITY) continue;
      const float w = exp2f(ms - Mx);
      l = fmaf(__ldcg(&a.part_ml[pr * 2 + 1]), w, l);
#pragma unroll
      for (int c = 0; c < PER_LANE; ++c) o[c] = fmaf(__ldcg(&a.part_o[pr * DH + lane + 32 * c]), w, o[c]);
    }
    float qv[PER_LANE];
#pragma unroll
    for (int c = 0; c < PER_LANE; ++c) qv[c] = qs[r * DH + lane + 32 * c];
    for (int wd = 0; wd < W; ++wd) {
      unsigned long long bits = t.anc[(int64_t)u * W + wd];
      while (bits) {
        const int v = wd * 64 + __ffsll((long long)bits) - 1;
        bits &= bits - 1;
        const int64_t kb = (((int64_t)b * NS + v) * a.Hkv + kvh) * DH;
        const int ti0 = t.depth[v] * HALF;
        float kr[PER_LANE];
#pragma unroll
        for (int c = 0; c < PER_LANE / 2; ++c) {
          const int i = lane + 32 * c;
          const float x1 = Elem<EL>::load(kn, kb + i), x2 = Elem<EL>::load(kn, kb + i + HALF);
          kr[c] = x1 * tab_c[ti0 + i] - x2 * tab_s[ti0 + i];
          kr[c + PER_LANE / 2] = x2 * tab_c[ti0 + i] + x1 * tab_s[ti0 + i];
        }
        float dot = 0.f;
#pragma unroll
        for (int c = 0; c < PER_LANE; ++c) dot = fmaf(qv[c], kr[c], dot);
        const float sc = warp_sum(dot) * a.scale_log2;
        const float m_new = fmaxf(Mx, sc);
        const float alpha = (Mx == -INFINITY) ? 0.f : exp2f(Mx - m_new);
        const float p = exp2f(sc - m_new);
        l = l * alpha + p;
#pragma unroll
        for (int c = 0; c < PER_LANE; ++c)
          o[c] = fmaf(o[c], alpha, p * Elem<EL>::load(vn, kb + lane + 32 * c));
        Mx = m_new;
      }
    }
    const float inv_l = 1.f / l;
    const int64_t ob = (((int64_t)b * NS + u) * a.Hq + h) * DH;
#pragma unroll
    for (int c = 0; c < PER_LANE; ++c) out[ob + lane + 32 * c] = o[c] * inv_l;
    if (a.lse && lane == 0) a.lse[((int64_t)b * NS + u) * a.Hq + h] = (Mx + log2f(l)) * kLn2;
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
