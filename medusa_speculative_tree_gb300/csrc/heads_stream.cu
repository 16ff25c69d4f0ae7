// Medusa heads as one persistent weight stream with in-stream top-k ([CN] "Medusa
// 的核心思路与系统位置"; [Math] "The Medusa head: math and shapes"; [M7.2] §0x02A,
// §0x04D; [PartII] Part 4).
//
// For one hidden row (T = 1, bf16), the round streams every head weight exactly once:
// W1_k (K x [d, d]), W_LM ([V, d], root = argmax) and W2_k (K x [V, d]).  A cooperative
// grid of one CTA per SM takes the 8-row groups of these matrices from one global
// counter, in stream order, so the stream never stops between matrices and a CTA that
// gets less bandwidth simply takes fewer groups:
//   W1_0..W1_{K-1}, the first half of W_LM, W2_0..W2_{K-1}, the second half of W_LM.
// The first half of W_LM sits between W1 and W2, so z is complete everywhere by the
// time any CTA needs it; the second half comes last, so the matrix whose top-k merge
// is exposed at the end is W_LM, whose top-k is a single entry.
//   - warp 8 (one lane) copies each group's 8 rows (up to 8 KiB each) with
//     cp.async.bulk into a 3-stage ring (192 KiB in flight per SM at d = 4096), and
//     copies the input row of the next matrix (h, or z_k once all W1 rows are counted)
//     into an x buffer ahead of the consumers;
//   - warps 0-7 each dot one row of a stage against the input row held in registers,
//     element pairs through packed fp32x2 FMAs, so shared memory serves only the
//     weights;
//   - a W1 row writes z_k = h + SiLU(W1_k h + b1_k); a vocabulary row feeds a
//     per-warp top-k list kept sorted across the warp's lanes (value desc, id asc);
//   - warp 9 merges the 8 warp lists of a matrix into the CTA's top-k and publishes
//     it; the CTA that completes a matrix merges all CTAs' lists into root or pool.
// Rows longer than 8 KiB (4096 < d <= 8192) are split in two halves (SPLIT = 2): a
// group is then 4 rows, warps 0-3 dot the first halves and own the rows, warps 4-7 dot
// the second halves against the second half of the input row and hand their partial
// sums to the owners through shared memory, so that every warp still holds at most
// 4096 input elements in registers and a stage still holds 64 KiB of 8 KiB segments.
// (Quarter rows, 2 rows per group in 5 stages of 32 KiB, measured 1.6x slower: the
// per-group overheads of 4 KiB segments dominate.)
// All waits are bounded; on a timeout the call records an error and root / pool
// become -1.
#include <float.h>
#include <limits.h>

#include "common.cuh"
#include "kernels.h"

namespace medusa {

namespace {

constexpr int kSConsumers = 8;                 // consumer warps = row parts per group
constexpr int kSProducer = 8;                  // warp index
constexpr int kSMerger = 9;                    // warp index
constexpr int kSThreads = 10 * 32;
// stages of the ring: 3 x 64 KiB, with whole rows or halves
__host__ __device__ constexpr int stream_stages(int) { return 3; }
constexpr int kSMaxU4 = 16;                    // 16-byte pieces of a row per lane (d <= 4096)
constexpr int kSMaxGrid = kHeadsStreamMaxGrid;

struct SCand {
  float v;
  int i;
};

struct StreamArgs {
  const uint16_t* h;          // [d]
  const uint16_t* w1;         // [K][d][d]
  const uint16_t* b1;         // [K][d] or null
  const uint16_t* w2;         // W2_k = w2 + k * w2_stride, [V][d]
  int64_t w2_stride;
  const uint16_t* w_lm;       // [V][d]
  int d, V, K, topk;
  float* z;                   // [K][d]
  float* logits_out;          // [K + 1][V] or null
  SCand* scand;               // [K + 1][G][topk], indexed by top-k matrix t
  int* err;
  int* cnt;                   // [0] warps done with W1, [1 + t] CTAs done with top-k matrix t,
                              // [K + 2] next group to hand out
  int32_t* root;
  int32_t* pool;              // [K][topk]
  uint64_t stall_ns;          // test hook (0 = off): wait this long for a counter nothing advances
};

// A counter slot of the zeroed counter block that no code path advances (the test hook
// waits on it).
constexpr int kStallSlot = (int)(kHeadsCounterBytes / sizeof(int)) - 5;
static_assert(MEDUSA_MAX_DEPTH + 2 < kStallSlot, "the counters of K heads reach cnt[K + 2]");

// Stream segments: W1 (K * g1 groups), W_LM first half (ga), W2 (K * gv), W_LM rest (gv - ga).
// Top-k matrix t: W2_t for t < K, W_LM for t = K; they publish in that order.
struct Layout {
  int K, g1, gv, ga;
  __device__ int base_lm_a() const { return K * g1; }
  __device__ int base_w2() const { return K * g1 + ga; }
  __device__ int base_lm_b() const { return K * g1 + ga + K * gv; }
  __device__ int total() const { return K * g1 + K * gv + gv; }
};

struct Item {
  int kind;      // 0 W1, 1 W_LM, 2 W2
  int k;         // head (W1, W2)
  int grp;       // 8-row group within the matrix
  int seq;       // stream matrix index: W1_k -> k, W_LM first half -> K, W2_k -> K + 1 + k, rest -> 2K + 1
};

__device__ __forceinline__ Item map_item(int i, const Layout& L) {
  Item it;
  if (i < L.base_lm_a()) {
    it.kind = 0; it.k = i / L.g1; it.grp = i % L.g1; it.seq = it.k;
  } else if (i < L.base_w2()) {
    it.kind = 1; it.k = 0; it.grp = i - L.base_lm_a(); it.seq = L.K;
  } else if (i < L.base_lm_b()) {
    const int r = i - L.base_w2();
    it.kind = 2; it.k = r / L.gv; it.grp = r % L.gv; it.seq = L.K + 1 + it.k;
  } else {
    it.kind = 1; it.k = 0; it.grp = L.ga + (i - L.base_lm_b()); it.seq = 2 * L.K + 1;
  }
  return it;
}

// Bounded wait that also ends when another warp of the CTA has given up.
__device__ __forceinline__ bool s_wait(uint32_t bar, uint32_t parity, const volatile int* abort_flag) {
  const uint64_t t0 = global_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try(bar, parity)) return true;
    if (*abort_flag) return false;
    if ((it & 255u) == 255u && global_ns() - t0 > 2000000000ull) return false;
  }
}

// One candidate from global memory, through L2 (written by other CTAs).
__device__ __forceinline__ SCand ld_cand_cg(const SCand* p) {
  const float2 f = __ldcg(reinterpret_cast<const float2*>(p));
  return SCand{f.x, __float_as_int(f.y)};
}

__device__ __forceinline__ void warp_argbest(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (ranks_before(ov, oi, v, i)) { v = ov; i = oi; }
  }
}

// Insert (v, id) into the sorted list of kk entries held one per lane (lv, li).
__device__ __forceinline__ void list_insert(float v, int id, int kk, float& lv, int& li) {
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

// 10 warps: the register file is shared as if by 12, 168 registers each; the input
// row (or its half) takes 128 of them.
template <int SPLIT>
__global__ void __launch_bounds__(kSThreads, 1) heads_stream_kernel(const StreamArgs a) {
  extern __shared__ __align__(16) uint8_t smem_s[];        // (bulk copies need 16 bytes)
  constexpr int RPG = kSConsumers / SPLIT;                 // rows per group (= owner warps)
  constexpr int NSTG = stream_stages(SPLIT);
  const int d = a.d, K = a.K, V = a.V;
  const int dp = d / SPLIT;                                 // elements of one row part
  const int seg = 2 * dp;                                   // bytes of one row part
  const int u4c = seg / 512;                                // 16-byte pieces per lane (<= 16)
  uint8_t* ring = smem_s;                                  // [stages][8][seg]
  uint8_t* xbuf = ring + NSTG * kSConsumers * seg;      // input row of the current matrix (h bf16 or z_k fp32)
  SCand* lists = reinterpret_cast<SCand*>(xbuf + 4 * d);   // [2][owners][32]
  float* partial = reinterpret_cast<float*>(lists + 2 * RPG * 32);   // [2][stages][parts - 1][RPG] part sums
  uint64_t* bars = reinterpret_cast<uint64_t*>(
      (reinterpret_cast<uintptr_t>(partial + 2 * NSTG * (SPLIT - 1) * RPG) + 7) & ~uintptr_t(7));
  __shared__ int abort_flag;
  const uint32_t full0 = smem_u32(&bars[0]), empty0 = smem_u32(&bars[NSTG]);
  const uint32_t lfull0 = smem_u32(&bars[2 * NSTG]), lfree0 = smem_u32(&bars[2 * NSTG + 2]);
  const uint32_t xfull = smem_u32(&bars[2 * NSTG + 4]), xempty = smem_u32(&bars[2 * NSTG + 5]);
  const uint32_t pdone0 = smem_u32(&bars[2 * NSTG + 6]);      // [stages] other parts summed
  const volatile int* abortp = &abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, c = blockIdx.x;
  Layout L;
  L.K = K;
  L.g1 = (d + RPG - 1) / RPG;
  L.gv = (V + RPG - 1) / RPG;
  L.ga = L.gv / 2;
  const int n_items = L.total();
  __shared__ int stage_item[NSTG];                      // group in each stage, -1 = no more

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < NSTG; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, kSConsumers);
    }
    for (int p = 0; p < 2; ++p) {
      mbar_init(lfull0 + 8 * p, RPG);
      mbar_init(lfree0 + 8 * p, 1);
    }
    mbar_init(xfull, 1);
    mbar_init(xempty, kSConsumers);
    if (SPLIT > 1)
      for (int s = 0; s < NSTG; ++s) mbar_init(pdone0 + 8 * s, kSConsumers - RPG);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  auto give_up = [&]() {          // the error flag first: whoever sees the abort sees it
    atomicExch(a.err, 1);
    __threadfence();
    *const_cast<volatile int*>(abortp) = 1;
  };

  if (warp == kSProducer) {
    // ---- weight stream --------------------------------------------------------------
    if (lane != 0) return;
    if (a.stall_ns != 0) {
      // Test hook: wait for a counter that nothing advances; after stall_ns give up
      // before any copy is issued, so the CTA's error path has nothing to drain.
      const uint64_t t0 = global_ns();
      for (;;) {
        int v;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(a.cnt + kStallSlot) : "memory");
        if (v != 0 || global_ns() - t0 > a.stall_ns) break;
      }
      give_up();
      return;
    }
    // Stage slots carry a group index, -2 (a marker: leave the W1 phase) or -1 (the end).
    int slot = 0, x_loads = 0, x_src = -2;
    bool z_ready = false;
    auto take_slot = [&](int& s) -> bool {
      s = slot % NSTG;
      return s_wait(empty0 + 8 * s, (uint32_t)(((slot / NSTG) & 1) ^ 1), abortp);
    };
    int next = atomicAdd(&a.cnt[K + 2], 1);
    for (;;) {
      const int idx = next;
      int s;
      if (idx >= n_items) {
        // no groups left: an empty-handed stage tells the consumers to stop
        if (!take_slot(s)) { give_up(); break; }
        stage_item[s] = -1;
        mbar_arrive(full0 + 8 * s);
        ++slot;
        break;
      }
      next = atomicAdd(&a.cnt[K + 2], 1);                   // the following group, ahead of time
      const Item it = map_item(idx, L);
      // The input row of the item's matrix (h, or z_k for W2_k) goes through the same
      // stream into the x buffer, once all consumer warps took the previous one.
      const int src = it.kind == 2 ? it.k : -1;
      if (src != x_src) {
        if (x_loads > 0 && !s_wait(xempty, (uint32_t)((x_loads - 1) & 1), abortp)) { give_up(); break; }
        if (src >= 0 && !z_ready) {
          // This CTA's consumers must be able to report their W1 rows before the wait
          // for everybody's: a marker stage lets them leave the W1 phase.
          if (!take_slot(s)) { give_up(); break; }
          stage_item[s] = -2;
          mbar_arrive(full0 + 8 * s);
          ++slot;
          // z is complete once every consumer warp of every CTA has finished its W1 rows
          const uint64_t t0 = global_ns();
          for (uint32_t sp = 0;; ++sp) {
            int v;
            asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(a.cnt) : "memory");
            if (v >= G * kSConsumers) { z_ready = true; break; }
            if (*abortp) break;
            if ((sp & 63u) == 63u && global_ns() - t0 > 2000000000ull) break;
          }
          if (!z_ready) { give_up(); break; }
          asm volatile("fence.proxy.async.global;" ::: "memory");   // the bulk copy reads what other SMs wrote
        }
        const uint32_t xb = src >= 0 ? 4u * d : 2u * d;
        mbar_expect_tx(xfull, xb);
        bulk_copy_g2s(smem_u32(xbuf), src >= 0 ? (const void*)(a.z + (int64_t)src * d) : (const void*)a.h, xb, xfull);
        x_src = src;
        ++x_loads;
      }
      if (!take_slot(s)) { give_up(); break; }
      stage_item[s] = idx;
      const uint16_t* base = it.kind == 0 ? a.w1 + (int64_t)it.k * d * d
                           : it.kind == 1 ? a.w_lm : a.w2 + (int64_t)it.k * a.w2_stride;
      const int n_rows = it.kind == 0 ? d : V;
      const int row0 = it.grp * RPG;
      const int rows = min(RPG, n_rows - row0);
      mbar_expect_tx(full0 + 8 * s, (uint32_t)(rows * SPLIT * seg));
      for (int h = 0; h < SPLIT; ++h)                       // slot h * RPG + r: part h of row r
        for (int r = 0; r < rows; ++r)
          bulk_copy_g2s(smem_u32(ring + (s * kSConsumers + h * RPG + r) * seg),
                        base + (int64_t)(row0 + r) * d + (int64_t)h * dp, (uint32_t)seg, full0 + 8 * s);
      ++slot;
    }
    // Copies still in flight (only after giving up) must land before the CTA exits.
    for (int n = slot - NSTG; n < slot; ++n)
      if (n >= 0) mbar_wait(full0 + 8 * (n % NSTG), (uint32_t)((n / NSTG) & 1), 100000000ull);
    if (x_loads > 0) mbar_wait(xfull, (uint32_t)((x_loads - 1) & 1), 100000000ull);
    return;
  }

  if (warp == kSMerger) {
    // ---- per-matrix top-k merges, in publication order t = 0..K ---------------------
    uint32_t ph_full[2] = {0u, 0u};
    for (int t = 0; t <= K; ++t) {
      // every CTA publishes one list per t (empty when it took no group of t)
      const int kk = t == K ? 1 : a.topk;
      const int p = t & 1;
      float bv = -INFINITY;
      int bi = INT_MAX;
      bool ok = false;
      if (!*abortp) {
        ok = __all_sync(0xffffffffu, s_wait(lfull0 + 8 * p, ph_full[p], abortp));
        ph_full[p] ^= 1u;
        if (!ok && lane == 0) give_up();
      }
      SCand* out = a.scand + ((int64_t)t * G + c) * a.topk;
      if (ok) {
        // one sorted list of kk entries per owner warp: entry e of warp w at lists[p][w][e]
        float ev[8];
        int ei[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int f = lane + 32 * q;                  // flattened index w * kk + e
          const int w = f / kk, e = f % kk;
          const bool valid = f < RPG * kk;
          ev[q] = valid ? lists[(p * RPG + w) * 32 + e].v : -INFINITY;
          ei[q] = valid ? lists[(p * RPG + w) * 32 + e].i : INT_MAX;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(lfree0 + 8 * p);     // the lists buffer may be refilled
        for (int r = 0; r < kk; ++r) {
          float v = -INFINITY;
          int i = INT_MAX, q_best = -1;
#pragma unroll
          for (int q = 0; q < 8; ++q)
            if (ei[q] != INT_MAX && (q_best < 0 || ranks_before(ev[q], ei[q], v, i))) { v = ev[q]; i = ei[q]; q_best = q; }
          float wv = v;
          int wi = i;
          warp_argbest(wv, wi);
          if (q_best >= 0 && wi == i && wi != INT_MAX) {
#pragma unroll
            for (int q = 0; q < 8; ++q)
              if (q == q_best) ei[q] = INT_MAX;
          }
          if (lane == r) { bv = wv; bi = wi; }
        }
      } else {
        if (lane == 0) mbar_arrive(lfree0 + 8 * p);
      }
      if (lane < a.topk) out[lane] = SCand{lane < kk ? bv : -INFINITY, lane < kk ? bi : INT_MAX};
      __threadfence();
      __syncwarp();
      int done = 0;
      if (lane == 0) done = atomicAdd(&a.cnt[1 + t], 1);
      done = __shfl_sync(0xffffffffu, done, 0);
      if (done != G - 1) continue;
      // ---- this CTA completed matrix t: merge all CTAs' sorted lists ----------------
      // Lane l keeps the current head of lists l, l + 32, ...; each round takes the best
      // head and advances its list (an L2 load).  The last matrix is W_LM, whose
      // one-entry top-k needs the heads only.
      __threadfence();
      const SCand* gl = a.scand + (int64_t)t * G * a.topk;
      auto entry = [&](int l, int e) -> SCand { return ld_cand_cg(gl + l * a.topk + e); };
      constexpr int kLpl = kSMaxGrid / 32;             // lists per lane
      float hv[kLpl];
      int hid[kLpl], hp[kLpl];
#pragma unroll
      for (int q = 0; q < kLpl; ++q) {
        const int l = lane + 32 * q;
        hp[q] = 0;
        hv[q] = -INFINITY;
        hid[q] = INT_MAX;
        if (l < G) {
          const SCand e = entry(l, 0);
          hv[q] = e.v;
          hid[q] = e.i;
        }
      }
      const bool bad = *reinterpret_cast<volatile int*>(a.err) != 0;
      for (int r = 0; r < kk; ++r) {
        float v = -INFINITY;
        int i = INT_MAX, q_best = -1;
#pragma unroll
        for (int q = 0; q < kLpl; ++q)
          if (hid[q] != INT_MAX && (q_best < 0 || ranks_before(hv[q], hid[q], v, i))) { v = hv[q]; i = hid[q]; q_best = q; }
        float wv = v;
        int wi = i;
        warp_argbest(wv, wi);
        if (q_best >= 0 && wi == i && wi != INT_MAX) {
#pragma unroll
          for (int q = 0; q < kLpl; ++q) {
            if (q != q_best) continue;
            const int l = lane + 32 * q;
            hp[q] += 1;
            if (hp[q] < kk) {
              const SCand e = entry(l, hp[q]);
              hv[q] = e.v;
              hid[q] = e.i;
            } else {
              hv[q] = -INFINITY;
              hid[q] = INT_MAX;
            }
          }
        }
        if (lane == 0) {
          const int id = (bad || wi == INT_MAX) ? -1 : wi;
          if (t == K) a.root[0] = id;
          else a.pool[(int64_t)t * a.topk + r] = id;
        }
      }
    }
    return;
  }

  // ---- consumer warps: one row of each group ------------------------------------------
  const int nv = dp / 256;                                  // 16-byte pieces per lane
  const int part = SPLIT == 1 ? 0 : warp / RPG;            // this warp's row part
  const int rw = SPLIT == 1 ? warp : warp % RPG;            // and row within the group
  const bool owner = SPLIT == 1 || part == 0;               // owners finish rows and keep lists
  float2 xr[kSMaxU4][4];                                    // input row (part), element pairs
  int cur_seq = -1, x_src = -2, x_loads = 0, cur_t = -1;
  bool w1_signalled = false;
  float lv = -INFINITY, lvm = -INFINITY;                    // this lane's entry of the W2 / W_LM list
  int li = INT_MAX, lim = INT_MAX;
  bool ok = true;
  // Hand the warp's sorted list of top-k matrix t to the merge warp.
  auto publish = [&](int t, float& pv, int& pi) -> bool {
    const int p = t & 1;
    if (t >= 2) {
      // The buffer was used by t - 2: wait until the merge warp read it.  The merge
      // warp arrives once for every t in order, so that is phase (t - 2) / 2.
      if (!__all_sync(0xffffffffu, s_wait(lfree0 + 8 * p, ((t - 2) >> 1) & 1, abortp))) return false;
    }
    lists[(p * RPG + warp) * 32 + lane] = SCand{pv, pi};
    __syncwarp();
    if (lane == 0) mbar_arrive(lfull0 + 8 * p);
    pv = -INFINITY;
    pi = INT_MAX;
    return true;
  };
  auto signal_w1 = [&]() {
    __threadfence();
    __syncwarp();
    if (lane == 0) atomicAdd(&a.cnt[0], 1);
    w1_signalled = true;
  };
  // W2 lists t < target are final for this CTA (groups arrive in stream order): hand
  // them out in order, the current one or an empty list for a matrix it never touched.
  int pub_next = 0;
  auto publish_upto = [&](int target) -> bool {
    while (pub_next < target) {
      const int t = pub_next;
      float ev = -INFINITY;
      int ei = INT_MAX;
      if (!(t == cur_t ? publish(t, lv, li) : publish(t, ev, ei))) return false;
      ++pub_next;
    }
    return true;
  };
  for (int n = 0; ok; ++n) {
    const int s = n % NSTG;
    if (!__all_sync(0xffffffffu, s_wait(full0 + 8 * s, (uint32_t)((n / NSTG) & 1), abortp))) {
      if (lane == 0) give_up();
      ok = false;
      break;
    }
    const int idx = stage_item[s];
    // (second-half warps arrive on the stage's partial-sum barrier at every use of the
    // stage, so that its phase counts stage uses)
    if (SPLIT > 1 && !owner && idx < 0 && lane == 0) mbar_arrive(pdone0 + 8 * s);
    if (idx == -1) break;                                   // no groups left
    if (idx == -2) {                                        // marker: leave the W1 phase
      if (!w1_signalled) signal_w1();
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * s);
      continue;
    }
    const Item it = map_item(idx, L);
    if (it.seq != cur_seq) {
      if (owner && !publish_upto(it.kind == 2 ? it.k : (it.seq == 2 * K + 1 ? K : 0))) {
        if (lane == 0) give_up();
        ok = false;
        break;
      }
      cur_t = it.kind == 2 ? it.k : -1;
      if (!w1_signalled && it.kind != 0) signal_w1();
      // input row into registers when its source changes (h for W1 and W_LM, z_k for
      // W2_k): the producer staged it in the x buffer
      const int src = it.kind == 2 ? it.k : -1;
      if (src != x_src) {
        if (!__all_sync(0xffffffffu, s_wait(xfull, (uint32_t)(x_loads & 1), abortp))) {
          if (lane == 0) give_up();
          ok = false;
          break;
        }
        if (src >= 0) {
          const float* zk = reinterpret_cast<const float*>(xbuf) + part * dp;
#pragma unroll
          for (int q = 0; q < kSMaxU4; ++q) {
            if (q < nv) {
              const float4 u0 = *reinterpret_cast<const float4*>(zk + 8 * (lane + 32 * q));
              const float4 u1 = *reinterpret_cast<const float4*>(zk + 8 * (lane + 32 * q) + 4);
              xr[q][0] = make_float2(u0.x, u0.y);
              xr[q][1] = make_float2(u0.z, u0.w);
              xr[q][2] = make_float2(u1.x, u1.y);
              xr[q][3] = make_float2(u1.z, u1.w);
            }
          }
        } else {
#pragma unroll
          for (int q = 0; q < kSMaxU4; ++q) {
            if (q < nv) {
              float f[8];
              Elem<uint16_t>::unpack(*reinterpret_cast<const uint4*>(xbuf + 2 * part * dp + 16 * (lane + 32 * q)), f);
#pragma unroll
              for (int e = 0; e < 4; ++e) xr[q][e] = make_float2(f[2 * e], f[2 * e + 1]);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(xempty);               // the x buffer may be refilled
        x_src = src;
        ++x_loads;
      }
      cur_seq = it.seq;
    }
    const int n_rows = it.kind == 0 ? d : V;
    const int row = it.grp * RPG + rw;
    float2 p[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
    if (row < n_rows) {
      const uint8_t* w = ring + (s * kSConsumers + warp) * seg;
      auto piece = [&](int q) {
        const uint4 v = *reinterpret_cast<const uint4*>(w + (lane + 32 * q) * 16);
        const uint32_t wq[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 wf = make_float2(__uint_as_float(wq[e] << 16), __uint_as_float(wq[e] & 0xFFFF0000u));
          p[e] = __ffma2_rn(wf, xr[q][e], p[e]);
        }
      };
      if (u4c == kSMaxU4) {
        // Row parts of 8 KiB (d = 4096, or 8192 in halves): a trip count known at compile
        // time lets every piece's load be issued ahead of the products; a bound known
        // only at run time measured nine times slower per piece.
#pragma unroll
        for (int q = 0; q < kSMaxU4; ++q) piece(q);
      } else {
#pragma unroll
        for (int q = 0; q < kSMaxU4; ++q)
          if (q < u4c) piece(q);
      }
    }
    __syncwarp();
    // this warp is done with the stage (an owner of split rows only once it has read
    // the part sums, so that no part warp reaches the stage's next use before that)
    if ((SPLIT == 1 || !owner) && lane == 0) mbar_arrive(empty0 + 8 * s);
    if (SPLIT == 1 && row >= n_rows) continue;
    float acc = ((p[0].x + p[0].y) + (p[1].x + p[1].y)) + ((p[2].x + p[2].y) + (p[3].x + p[3].y));
    acc = warp_sum(acc);
    acc = __shfl_sync(0xffffffffu, acc, 0);                 // one value for every lane
    if (SPLIT > 1) {
      const int pb = (n / NSTG) & 1;                        // part-sum buffer of this use
      if (!owner) {                                         // other part: hand the sum over
        if (lane == 0) {
          partial[((pb * NSTG + s) * (SPLIT - 1) + part - 1) * RPG + rw] = acc;
          mbar_arrive(pdone0 + 8 * s);                      // (release: the sum is visible)
        }
        __syncwarp();
        continue;
      }
      if (row < n_rows) {
        if (!__all_sync(0xffffffffu, s_wait(pdone0 + 8 * s, (uint32_t)((n / NSTG) & 1), abortp))) {
          if (lane == 0) give_up();
          ok = false;
          break;
        }
#pragma unroll
        for (int q = 1; q < SPLIT; ++q) acc += partial[((pb * NSTG + s) * (SPLIT - 1) + q - 1) * RPG + rw];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * s);
      if (row >= n_rows) continue;
    }
    if (it.kind == 0) {
      if (lane == 0) {
        float v = acc;
        if (a.b1) v += Elem<uint16_t>::load(a.b1, (int64_t)it.k * d + row);
        const float hv = Elem<uint16_t>::load(a.h, row);
        a.z[(int64_t)it.k * d + row] = hv + v / (1.f + expf(-v));   // h + SiLU(W1 h + b1)
      }
    } else if (it.kind == 2) {
      if (a.logits_out && lane == 0) a.logits_out[(int64_t)(1 + it.k) * V + row] = acc;
      list_insert(acc, row, a.topk, lv, li);
    } else {
      if (a.logits_out && lane == 0) a.logits_out[row] = acc;
      list_insert(acc, row, 1, lvm, lim);
    }
  }
  if (owner && ok && (!publish_upto(K) || !publish(K, lvm, lim))) { if (lane == 0) give_up(); ok = false; }
  if (!w1_signalled) signal_w1();
}

}  // namespace

int heads_stream_split(int d) { return d <= 4096 ? 1 : 2; }

size_t heads_stream_smem(int d) {
  const int split = heads_stream_split(d), rpg = kSConsumers / split, stg = stream_stages(split);
  const size_t part = ((size_t)2 * stg * (split - 1) * rpg * sizeof(float) + 7) & ~(size_t)7;
  return (size_t)stg * kSConsumers * 2 * (d / split) + 4 * (size_t)d + 2 * rpg * 32 * sizeof(SCand) + part +
         (3 * stg + 6) * sizeof(uint64_t);
}

bool heads_stream_supported(int T, int d, int V, int K, int topk, medusa_dtype dt, const void* h, const void* w1,
                            const void* w2, int64_t w2_stride, const void* w_lm, const void* b1) {
  auto al = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  // one stage segment per row (d <= 4096, 8 KiB rows) or per half row (d <= 8192)
  if (T != 1 || dt != MEDUSA_BF16 || K < 1 || d % 256 != 0 || d > 8192 || V < 2 || topk > 32) return false;
  if (d > 4096 && d % 512 != 0) return false;
  if (!h || !w1 || !w2 || !w_lm || !al(h) || !al(w1) || !al(w2) || !al(w_lm) || (w2_stride * 2) % 16 != 0 ||
      w2_stride < 0)
    return false;
  (void)b1;
  int dev = 0, coop = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (coop == 0 || sms < 1 || heads_stream_smem(d) > 227 * 1024) return false;
  // every CTA must be resident at once (one per SM)
  auto kern = heads_stream_split(d) == 1 ? heads_stream_kernel<1> : heads_stream_kernel<2>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)heads_stream_smem(d)) !=
      cudaSuccess)
    return false;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kSThreads, heads_stream_smem(d)) != cudaSuccess)
    return false;
  return per_sm >= 1;
}

cudaError_t launch_heads_stream(const HeadsPlan& p, const void* h, const void* w1, const void* b1, const void* w2,
                                int64_t w2_stride, const void* w_lm, int32_t* root, int32_t* pool,
                                float* logits_out, void* ws, cudaStream_t st) {
  char* base = (char*)ws;
  StreamArgs a{};
  a.h = (const uint16_t*)h;
  a.w1 = (const uint16_t*)w1;
  a.b1 = (const uint16_t*)b1;
  a.w2 = (const uint16_t*)w2;
  a.w2_stride = w2_stride;
  a.w_lm = (const uint16_t*)w_lm;
  a.d = p.d;
  a.V = p.V;
  a.K = p.K;
  a.topk = p.topk;
  a.z = (float*)(base + p.off_z);
  a.logits_out = logits_out;
  a.scand = (SCand*)(base + p.off_scand);
  a.err = (int*)(base + p.off_err);
  a.cnt = a.err + 4;
  a.root = root;
  a.pool = pool;
  a.stall_ns = test_stall_ns();
  const size_t smem = heads_stream_smem(p.d);
  auto kern = heads_stream_split(p.d) == 1 ? heads_stream_kernel<1> : heads_stream_kernel<2>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int G = sms < kSMaxGrid ? sms : kSMaxGrid;
  // error flag and counters start at zero
  e = cudaMemsetAsync(a.err, 0, kHeadsCounterBytes, st);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(G);
  cfg.blockDim = dim3(kSThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace medusa
