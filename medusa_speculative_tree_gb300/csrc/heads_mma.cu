// Medusa heads for several hidden rows at once on tcgen05 tensor cores ([CN] "Medusa
// 的核心思路与系统位置"; [Math] "The Medusa head: math and shapes"; [M7.2] §0x02A,
// §0x04D; [PartII] Part 4).
//
// With T >= 2 rows (batched serving: one frontier row per sequence) each weight row
// meets T inputs, which the CUDA cores can no longer absorb at HBM speed; the weight
// stream becomes a skinny GEMM: D[r][n] = sum_k W[r][k] X[n][k] for 128-row groups of
// W (the M of the MMA) against the input rows.  h is exactly bf16, so W1 h and W_LM h
// take the T rows of h as they are (N = T rounded up to 16; the rows past T are the
// copy's zero fill).  z is not: its rows are bf16 pairs (N = 2T rounded up to 32), row
// 2t holding bf16(z_t) and row 2t + 1 bf16(z_t - bf16(z_t)), so the sum of the two
// columns carries z_t to ~2^-16 relative.  Columns past the used rows are never read.
//
// Passes of more than 128 rows (up to 256: the all-rows variant) would need 512 input
// columns as pairs, more than one MMA takes.  They run "wide" instead: the input rows are
// single (h is exactly bf16; z is stored as fp16, ~2^-11 relative) and the W2 tiles are
// re-encoded in shared memory from bf16 to fp16 (exact for |w| in [2^-14, 65504]) by
// four converter warps, so that W2 z is one fp16 MMA; W1 h and W_LM h stay bf16 MMAs
// on the rows of h.
// A pass then reads the weights once for twice as many rows.
//
// One persistent CTA per SM (cooperative launch) takes 128-row groups from a global
// counter in stream order: W1_0..W1_{K-1}, the first half of W_LM, W2_0..W2_{K-1}, the
// rest of W_LM.
//   - warp 0 (one lane): TMA producer.  Each stage holds up to four 64-column K chunks
//     of the group (128 x 64 bf16, 16 KiB each) and of the inputs (rows of h or of z,
//     x 64 bf16), both K-major with the 128-byte swizzle; W2 stages wait until every W1
//     group has written z;
//   - warp 1: owns TMEM; one lane issues tcgen05.mma (kind::f16, bf16 in, fp32 out)
//     into one of two TMEM accumulators;
//   - warps 2-5: epilogue, thread = output row (TMEM lane).  A W1 row writes
//     z_k = h + SiLU(W1_k h + b1_k) for every input row (a bf16 pair, or fp16 when
//     wide); a vocabulary row writes its T logits.  Top-k then runs on the logits.
// All waits are bounded; on a timeout the call records an error (the top-k merge then
// writes -1).
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace medusa {

namespace {

constexpr int kMThreads = 6 * 32;
constexpr int kMConvWarp0 = 6;               // wide passes: converter warps 6-9
constexpr int kMConvWarps = 4;
constexpr int kMThreadsWide = (6 + kMConvWarps) * 32;
constexpr int kMRows = 128;                  // rows of W per group (MMA M)
constexpr int kMKc = 64;                     // K columns per stage (one 128-byte swizzle row)

struct MmaArgs {
  const uint16_t* h;          // [T][d] bf16
  const uint16_t* b1;         // [K][d] or null
  int d, V, K, T, N;          // N = input rows of z (2T, or T when wide, rounded up to 32)
  int NH;                     // input rows of h (T rounded up to 16)
  int w2_shared;              // W2 heads share one matrix
  uint16_t* z_hl;             // [K][N][d] bf16 pairs of z, or (wide) fp16 z
  float* logits;              // [T][K + 1][V]
  int* err;
  int* cnt;                   // [0] W1 row quarters written (4 per group), [1] next group to hand out
  int n_stages;
  int bps;                    // 64-column K chunks (TMA boxes) per stage
  uint32_t stage_bytes;
};

struct MLayout {
  int K, g1, gv, ga;
  __device__ int base_lm_a() const { return K * g1; }
  __device__ int base_w2() const { return K * g1 + ga; }
  __device__ int base_lm_b() const { return K * g1 + ga + K * gv; }
  __device__ int total() const { return K * g1 + K * gv + gv; }
};

struct MItem {
  int kind;      // 0 W1, 1 W_LM, 2 W2
  int k;
  int grp;
};

__device__ __forceinline__ MItem mmap_item(int i, const MLayout& L) {
  MItem it;
  if (i < L.base_lm_a()) {
    it.kind = 0; it.k = i / L.g1; it.grp = i % L.g1;
  } else if (i < L.base_w2()) {
    it.kind = 1; it.k = 0; it.grp = i - L.base_lm_a();
  } else if (i < L.base_lm_b()) {
    const int r = i - L.base_w2();
    it.kind = 2; it.k = r / L.gv; it.grp = r % L.gv;
  } else {
    it.kind = 1; it.k = 0; it.grp = L.ga + (i - L.base_lm_b());
  }
  return it;
}

__device__ __forceinline__ bool m_wait(uint32_t bar, uint32_t parity, const volatile int* abort_flag) {
  const uint64_t t0 = global_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try(bar, parity)) return true;
    if (*abort_flag) return false;
    if ((it & 255u) == 255u && global_ns() - t0 > 2000000000ull) return false;
  }
}

// bf16 x8 (uint4) -> fp16 x8, exact for magnitudes in [2^-14, 65504].
__device__ __forceinline__ uint32_t f16x2_of(float a, float b) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
  return r;
}
__device__ __forceinline__ uint4 bf16x8_to_f16x8_m(uint4 v) {
  uint4 o;
  o.x = f16x2_of(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u));
  o.y = f16x2_of(__uint_as_float(v.y << 16), __uint_as_float(v.y & 0xFFFF0000u));
  o.z = f16x2_of(__uint_as_float(v.z << 16), __uint_as_float(v.z & 0xFFFF0000u));
  o.w = f16x2_of(__uint_as_float(v.w << 16), __uint_as_float(v.w & 0xFFFF0000u));
  return o;
}

template <bool WIDE>
__global__ void __launch_bounds__(WIDE ? kMThreadsWide : kMThreads, 1)
    heads_mma_kernel(const __grid_constant__ CUtensorMap tmW1, const __grid_constant__ CUtensorMap tmLM,
                     const __grid_constant__ CUtensorMap tmW2, const __grid_constant__ CUtensorMap tmH,
                     const __grid_constant__ CUtensorMap tmZ, const MmaArgs a) {
  extern __shared__ uint8_t smem_m[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_m) + 1023) & ~uintptr_t(1023));
  const int S = a.n_stages, N = a.N, NH = a.NH, d = a.d, K = a.K, V = a.V, T = a.T;
  const int NA = N > NH ? N : NH;                    // accumulator columns (and B box rows of a stage)
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + (size_t)S * a.stage_bytes);
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ int stage_item[16];                     // group of each stage, -1 = no more groups
  __shared__ int dgrp[2];                            // group of each accumulator, -1 = no more
  const uint32_t full0 = smem_u32(&bars[0]), empty0 = smem_u32(&bars[S]);
  const uint32_t dfull0 = smem_u32(&bars[2 * S]), dempty0 = smem_u32(&bars[2 * S + 2]);
  const uint32_t drain = smem_u32(&bars[2 * S + 4]);
  const uint32_t conv0 = smem_u32(&bars[2 * S + 5]);            // wide: [S] stage converted
  const volatile int* abortp = &abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  MLayout L;
  L.K = K;
  L.g1 = (d + kMRows - 1) / kMRows;
  L.gv = (V + kMRows - 1) / kMRows;
  L.ga = L.gv / 2;
  const int n_items = L.total();
  const int bps = a.bps;
  const int n_k = d / (kMKc * bps);                  // stages per group
  const uint32_t a_bytes = kMRows * kMKc * 2, b_bytes = (uint32_t)NA * kMKc * 2;   // one box slot each
  const uint32_t tmem_cols = (uint32_t)(2 * NA <= 32 ? 32 : 2 * NA <= 64 ? 64 : 2 * NA <= 128 ? 128 : 2 * NA <= 256 ? 256 : 512);

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int p = 0; p < 2; ++p) {
      mbar_init(dfull0 + 8 * p, 1);
      mbar_init(dempty0 + 8 * p, 4);                 // the four epilogue warps
    }
    mbar_init(drain, 1);
    if (WIDE)
      for (int s = 0; s < S; ++s) mbar_init(conv0 + 8 * s, kMConvWarps);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_slot)),
                 "r"(tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  bool ok = true;
  int slot = 0;                                      // producer: stage slots used
  auto give_up = [&]() {
    *const_cast<volatile int*>(abortp) = 1;
    atomicExch(a.err, 1);
  };

  if (warp == 0) {
    // ---- TMA producer ----------------------------------------------------------------
    if (lane == 0) {
      bool z_ready = false;
      auto take_slot = [&](int& s) -> bool {
        s = slot % S;
        return m_wait(empty0 + 8 * s, (uint32_t)(((slot / S) & 1) ^ 1), abortp);
      };
      int next = atomicAdd(&a.cnt[1], 1);
      for (;;) {
        const int idx = next;
        int s;
        if (idx >= n_items) {
          if (!take_slot(s)) { ok = false; break; }
          stage_item[s] = -1;
          mbar_arrive(full0 + 8 * s);
          ++slot;
          break;
        }
        next = atomicAdd(&a.cnt[1], 1);
        const MItem it = mmap_item(idx, L);
        if (it.kind == 2 && !z_ready) {
          // W2 inputs are z: every W1 group must have written its rows
          const uint64_t t0 = global_ns();
          for (uint32_t sp = 0;; ++sp) {
            int v;
            asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(a.cnt) : "memory");
            if (v >= 4 * K * L.g1) { z_ready = true; break; }   // four epilogue warps per group
            if (*abortp) break;
            if ((sp & 63u) == 63u && global_ns() - t0 > 2000000000ull) break;
          }
          if (!z_ready) { ok = false; break; }
          asm volatile("fence.proxy.async.global;" ::: "memory");   // TMA reads what other SMs wrote
        }
        for (int kc = 0; kc < n_k && ok; ++kc) {
          if (!take_slot(s)) { ok = false; break; }
          stage_item[s] = idx;
          // A boxes (weights) first, then B boxes (inputs), bps of each
          const uint32_t sA = smem_u32(sm + (size_t)s * a.stage_bytes), sB = sA + bps * a_bytes;
          const uint32_t bar = full0 + 8 * s;
          mbar_expect_tx(bar, (uint32_t)bps * (a_bytes + (uint32_t)(it.kind == 2 ? N : NH) * kMKc * 2));
          const int r0 = it.grp * kMRows;
          for (int bx = 0; bx < bps; ++bx) {
            const int col = (kc * bps + bx) * kMKc;
            const uint32_t dA = sA + bx * a_bytes, dB = sB + bx * b_bytes;
            if (it.kind == 0) tma_load_2d(dA, &tmW1, col, it.k * d + r0, bar);
            else if (it.kind == 1) tma_load_2d(dA, &tmLM, col, r0, bar);
            else if (a.w2_shared) tma_load_2d(dA, &tmW2, col, r0, bar);
            else tma_load_3d(dA, &tmW2, col, r0, it.k, bar);
            if (it.kind == 2) tma_load_2d(dB, &tmZ, col, it.k * N, bar);
            else tma_load_2d(dB, &tmH, col, 0, bar);
          }
          ++slot;
        }
        if (!ok) break;
      }
      if (!ok) give_up();
    }
  } else if (warp == 1) {
    // ---- MMA issue: one group = n_k stages into accumulator g & 1 ------------------------
    if (lane == 0) {
      const uint32_t idesc_z = WIDE ? idesc_f16(kMRows, N, false) : idesc_bf16(kMRows, N);
      const uint32_t idesc_x = idesc_bf16(kMRows, NH);            // W1 h, W_LM h
      uint32_t idesc = idesc_x;
      int u = 0;
      for (int g = 0; ok; ++g) {
        const int db = g & 1;
        for (int kc = 0; kc < n_k; ++kc, ++u) {
          const int s = u % S;
          // (wide: the converter warps pass every stage on, W2 stages re-encoded to fp16)
          if (!m_wait((WIDE ? conv0 : full0) + 8 * s, (uint32_t)((u / S) & 1), abortp)) { ok = false; break; }
          if (kc == 0) {
            const int idx = stage_item[s];
            // the accumulator must have been read out (group g - 2) before it is reused
            if (g >= 2 && !m_wait(dempty0 + 8 * db, (uint32_t)(((g >> 1) - 1) & 1), abortp)) { ok = false; break; }
            if (idx < 0) {                               // no more groups: tell the epilogue
              dgrp[db] = -1;
              mbar_arrive(dfull0 + 8 * db);
              g = -2;                                    // leave the outer loop
              break;
            }
            dgrp[db] = idx;
            __threadfence_block();
            idesc = mmap_item(idx, L).kind == 2 ? idesc_z : idesc_x;
          }
          tc_fence_after();
          const uint32_t sA = smem_u32(sm + (size_t)s * a.stage_bytes), sB = sA + bps * a_bytes;
          for (int bx = 0; bx < bps; ++bx) {
#pragma unroll
            for (int kk = 0; kk < kMKc / 16; ++kk)
              umma_f16(tmem + (uint32_t)(db * NA), sw128_desc(sA + bx * a_bytes + kk * 32, 16, 1024),
                       sw128_desc(sB + bx * b_bytes + kk * 32, 16, 1024), idesc, (kc > 0 || bx > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(empty0 + 8 * s);                   // the stage is free once these MMAs are done
          if (kc == n_k - 1) umma_commit(dfull0 + 8 * db);
        }
        if (g < 0) break;
      }
      if (!ok) give_up();
    }
  } else if (WIDE && warp >= kMConvWarp0) {
    // ---- wide: W2 tiles bf16 -> fp16 in place; every stage is passed on -----------------
    const int ct = threadIdx.x - kMConvWarp0 * 32;
    for (int u = 0;; ++u) {
      const int s = u % S;
      if (!__all_sync(0xffffffffu, m_wait(full0 + 8 * s, (uint32_t)((u / S) & 1), abortp))) { ok = false; break; }
      const int idx = *reinterpret_cast<volatile int*>(&stage_item[s]);
      if (idx >= 0 && mmap_item(idx, L).kind == 2) {
        uint4* p = reinterpret_cast<uint4*>(sm + (size_t)s * a.stage_bytes);
        const int n4 = bps * (int)(a_bytes / 16);
        for (int i = ct; i < n4; i += kMConvWarps * 32) p[i] = bf16x8_to_f16x8_m(p[i]);
        fence_proxy_async();                         // the MMA reads these through the async proxy
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(conv0 + 8 * s);
      if (idx < 0) break;                            // the end marker: no more stages
    }
    if (!ok && lane == 0) give_up();
  } else {
    // ---- epilogue: thread = output row ---------------------------------------------------
    const int q = warp & 3;                            // TMEM lane quadrant of this warp
    const int r = 32 * q + lane;
    for (int g = 0;; ++g) {
      const int db = g & 1;
      if (!__all_sync(0xffffffffu, m_wait(dfull0 + 8 * db, (uint32_t)((g >> 1) & 1), abortp))) { ok = false; break; }
      const int idx = *reinterpret_cast<volatile int*>(&dgrp[db]);
      if (idx < 0) break;
      tc_fence_after();
      const MItem it = mmap_item(idx, L);
      const int n_rows = it.kind == 0 ? d : V;
      const int row = it.grp * kMRows + r;
      // one accumulator column per input row, except z's bf16 pairs (two columns)
      const bool single = WIDE || it.kind != 2;
      const int ncol = it.kind == 2 ? N : NH;
      bool bad = false;
      auto emit = [&](int t, float x) {
        if (it.kind == 0) {
          float zv = x;
          if (a.b1) zv += Elem<uint16_t>::load(a.b1, (int64_t)it.k * d + row);
          const float z = Elem<uint16_t>::load(a.h, (int64_t)t * d + row) + zv / (1.f + expf(-zv));
          if (WIDE) {
            const __half zh = __float2half_rn(z);
            bad |= !(fabsf(z) <= 65504.f);             // z outside fp16's range (or not finite)
            a.z_hl[((int64_t)it.k * N + t) * d + row] = __half_as_ushort(zh);
          } else {
            const uint16_t hi = f32_to_bf16_bits(z);
            const uint16_t lo = f32_to_bf16_bits(z - __uint_as_float((uint32_t)hi << 16));
            a.z_hl[((int64_t)it.k * N + 2 * t) * d + row] = hi;
            a.z_hl[((int64_t)it.k * N + 2 * t + 1) * d + row] = lo;
          }
        } else {
          const int m = it.kind == 1 ? 0 : 1 + it.k;
          a.logits[((int64_t)t * (K + 1) + m) * V + row] = x;
        }
      };
      for (int c0 = 0; c0 < ncol; c0 += 32) {
        float v[32];
        tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(db * NA + c0), v);
        if (row >= n_rows) continue;
        if (single) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (c0 + j >= T) break;
            emit(c0 + j, v[j]);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (c0 / 2 + j >= T) break;
            emit(c0 / 2 + j, v[2 * j] + v[2 * j + 1]);
          }
        }
      }
      if (bad) atomicExch(a.err, 1);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dempty0 + 8 * db);
      if (it.kind == 0) {
        // this warp's 32 rows of z are written: count them (4 per W1 group)
        __threadfence();
        __syncwarp();
        if (lane == 0) atomicAdd(&a.cnt[0], 1);
      }
    }
    if (!ok && lane == 0) give_up();
  }

  // ---- join, drain after a failure, free TMEM ----------------------------------------
  __syncthreads();
  if (*abortp) {
    if (warp == 0 && lane == 0)
      for (int n = slot - S; n < slot; ++n)
        if (n >= 0) mbar_wait(full0 + 8 * (n % S), (uint32_t)((n / S) & 1), 100000000ull);
    if (warp == 1 && lane == 0) {
      umma_commit(drain);
      mbar_wait(drain, 0, 100000000ull);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(tmem_cols) : "memory");
  }
}

}  // namespace

size_t heads_mma_rows(int T, bool wide) {
  if (wide) return (size_t)((T + 31) / 32 * 32);                     // single rows
  return (size_t)((2 * T + 31) / 32 * 32);                           // bf16 pairs
}

namespace {
// Rows of h as the MMA input (16 per instruction step) and the larger of the two row
// counts, which sizes the stage slots and the accumulators.
int heads_mma_h_rows(int T) { return (T + 15) / 16 * 16; }
int heads_mma_acc_rows(int T, bool wide) {
  const int N = (int)heads_mma_rows(T, wide), NH = heads_mma_h_rows(T);
  return N > NH ? N : NH;
}
}  // namespace

namespace {
// A stage holds bps boxes of weights (128 x 64) and of inputs (N x 64): as many K
// chunks per stage as still leave four stages, else two (fewer, larger stages cost
// the MMA lane fewer waits per byte; more stages keep more bytes in flight).
size_t mma_stage_bytes(int N, int bps) { return (size_t)bps * ((size_t)kMRows * kMKc * 2 + (size_t)N * kMKc * 2); }
constexpr int kMBarSlots = 64;              // mbarriers after the stages: full, empty, 2 x 2 accumulator, drain, conv
constexpr size_t kMBudget = 227 * 1024 - 1024 - kMBarSlots * 8;
int mma_bps(int N, int d) {
  // at least four stages in flight when two or more chunks per stage allow it
  // (measured: 16 rows, 2 chunks x 5 stages beat 4 chunks x 2 stages by 2%)
  for (int bps = 4; bps > 1; bps >>= 1)
    if ((d / kMKc) % bps == 0 && kMBudget / mma_stage_bytes(N, bps) >= 4) return bps;
  for (int bps = 4; bps > 1; bps >>= 1)
    if ((d / kMKc) % bps == 0 && kMBudget / mma_stage_bytes(N, bps) >= 2) return bps;
  return 1;
}
int mma_stages(int N, int d) {
  int s = (int)(kMBudget / mma_stage_bytes(N, mma_bps(N, d)));
  return s > 12 ? 12 : s;
}
size_t mma_smem(int N, int d) {
  return 1024 + (size_t)mma_stages(N, d) * mma_stage_bytes(N, mma_bps(N, d)) + kMBarSlots * 8;
}
static_assert(3 * 12 + 5 <= kMBarSlots, "barrier slots of the most stages");

bool encode_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows,
               CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {(cuuint32_t)kMKc, box_rows}, estr[2] = {1, 1};
  return fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_w2(CUtensorMap* map, const void* base, int d, int V, int K, int64_t stride) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)V, (cuuint64_t)K};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)stride * 2};
  cuuint32_t box[3] = {(cuuint32_t)kMKc, (cuuint32_t)kMRows, 1}, estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

bool heads_mma_supported(int T, int d, int V, int K, medusa_dtype dt, const void* h, const void* w1, const void* w2,
                         int64_t w2_stride, const void* w_lm) {
  auto al = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (T < 2 || dt != MEDUSA_BF16 || K < 1 || d % kMKc != 0 || V < 1) return false;
  const bool wide = heads_mma_wide(T);
  const int per_pass = wide ? kHeadsMmaWideRows : kHeadsMmaMaxRows;
  if (T > per_pass) T = per_pass;                          // more rows run in passes of this many
  if (!h || !w1 || !w2 || !w_lm || !al(h) || !al(w1) || !al(w2) || !al(w_lm)) return false;
  if (w2_stride < 0 || (w2_stride * 2) % 16 != 0 || (w2_stride != 0 && w2_stride < (int64_t)V * d)) return false;
  if (!encode_fn()) return false;
  int dev = 0, coop = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
  const int NA = heads_mma_acc_rows(T, wide);
  if (coop == 0 || mma_stages(NA, d) < 2) return false;
  auto kern = wide ? heads_mma_kernel<true> : heads_mma_kernel<false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)mma_smem(NA, d)) != cudaSuccess)
    return false;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, wide ? kMThreadsWide : kMThreads,
                                                    mma_smem(NA, d)) != cudaSuccess)
    return false;
  return per_sm >= 1;
}

cudaError_t launch_heads_mma(const HeadsPlan& p, bool wide, const void* h, const void* w1, const void* b1,
                             const void* w2, int64_t w2_stride, const void* w_lm, float* logits, void* ws,
                             cudaStream_t st) {
  char* base = (char*)ws;
  const int T = p.T, d = p.d, V = p.V, K = p.K;
  const int N = (int)heads_mma_rows(T, wide), NH = heads_mma_h_rows(T), NA = heads_mma_acc_rows(T, wide);
  uint16_t* z_hl = (uint16_t*)(base + p.off_zhl);
  int* err = (int*)(base + p.off_err);
  CUtensorMap mw1, mlm, mw2, mh, mz;
  const bool shared = w2_stride == 0;
  if (!encode_2d(&mw1, w1, d, (uint64_t)K * d, kMRows) || !encode_2d(&mlm, w_lm, d, V, kMRows) ||
      !(shared ? encode_2d(&mw2, w2, d, V, kMRows) : encode_w2(&mw2, w2, d, V, K, w2_stride)) ||
      !encode_2d(&mh, h, d, T, NH) ||                      // rows past T: the copy's zero fill
      !encode_2d(&mz, z_hl, d, (uint64_t)K * N, N,
                 wide ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16))
    return cudaErrorInvalidValue;
  MmaArgs a{};
  a.h = (const uint16_t*)h;
  a.b1 = (const uint16_t*)b1;
  a.d = d; a.V = V; a.K = K; a.T = T; a.N = N; a.NH = NH;
  a.w2_shared = shared ? 1 : 0;
  a.z_hl = z_hl;
  a.logits = logits;
  a.err = err;
  a.cnt = err + 4;
  a.bps = mma_bps(NA, d);
  a.n_stages = mma_stages(NA, d);
  a.stage_bytes = (uint32_t)mma_stage_bytes(NA, a.bps);
  cudaError_t e;
  const size_t smem = mma_smem(NA, d);
  auto kern = wide ? heads_mma_kernel<true> : heads_mma_kernel<false>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sms);
  cfg.blockDim = dim3(wide ? kMThreadsWide : kMThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, mw1, mlm, mw2, mh, mz, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace medusa
