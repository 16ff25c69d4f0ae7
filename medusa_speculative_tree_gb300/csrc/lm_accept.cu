// Acceptance with the target's vocabulary projection folded in ([M7.2] §0x07B: the
// round's C_LMproj with F_LMproj = 2 N d V, and a unique-row posterior instead of
// gathered path logits; §0x07C: dense target logits hold N V elements; §0x04D,
// §0x04E for what acceptance reads).
//
// Acceptance reads, of each internal row's logits x = W_LM h, only the argmax, the max,
// partition function and first moment of x / T, and x at the token of each child.  The
// projection runs on tcgen05 tensor cores and keeps exactly those, so the [rows x V]
// logits are never written:
//   lm_gather_kernel   the internal rows' hidden states, packed as the GEMM's N side
//                      (bf16, zero padding columns), and every internal row's children
//                      (row, token) in ascending row order;
//   lm_stats_kernel    one persistent CTA per SM over 128-row groups of W_LM (the MMA's
//                      M).  With more than 256 columns the CTAs form P interleaved
//                      sets, one per pass of up to 256 columns (CTA i serves pass
//                      i % P); every set walks the same group order, so the sets read
//                      each group of W_LM at about the same time and all but the first
//                      read mostly hit L2.  Within a set, CTA c takes groups c, c + n,
//                      2n + c, ... (n CTAs per set):
//                        warp 0 (one lane)  TMA of W_LM boxes and of the packed rows;
//                        warp 1             owns TMEM; one lane issues tcgen05.mma
//                                           (kind::f16, bf16 operands, fp32 accumulate)
//                                           into one of two accumulators;
//                        warps 2-5          epilogue: each warp moves its 32 vocabulary
//                                           rows x 32 columns through a private
//                                           shared-memory tile, then lane c folds
//                                           column c (one internal row) over those 32
//                                           ids and records the child tokens it meets;
//                      at the end the four warps' statistics are merged per column and
//                      written as that CTA's chunk of the row;
//   select (accept.cu) merges the CTAs' chunks per row and decides the paths.
// Up to four passes of 256 columns (B x n_internal rows) run in one launch.
// All waits are bounded; a timeout sets an error flag and every sequence then
// publishes nothing (accept_len = -1).
#include <climits>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace medusa {

namespace {

constexpr int kLThreads = 6 * 32;
constexpr int kLRows = 128;           // vocabulary rows per group (MMA M)
constexpr int kLKc = 64;              // K columns per TMA box (one 128-byte swizzle row)
constexpr int kLMaxCols = 256;        // columns per pass (MMA N)
constexpr int kLMaxPass = 4;          // passes (CTA sets) of one launch
constexpr int kLKids = MEDUSA_MAX_TOPK;   // children of a row: distinct ranks of one head
constexpr int kTileStride = 33;       // epilogue tile row stride (floats): conflict-free columns
constexpr size_t kLMergeBytes = (size_t)4 * kLMaxCols * sizeof(RowPart);   // per-warp statistics at the end

struct LmArgs {
  int V, d, N, NI;
  int n_pass;                   // CTA sets of this launch, one per pass
  int col0[kLMaxPass];          // first column of each pass (column = b * NI + internal index)
  int n_cols[kLMaxPass];        // valid columns of each pass
  int n_mma[kLMaxPass];         // MMA N: n_cols rounded up to 32 (32-column TMEM loads stay aligned)
  int n_cta;                    // CTAs per set: the statistics chunks of a column
  float inv_temp;
  const int32_t* e_tok;   // [cols_pad][kLKids] child tokens
  const int32_t* e_row;   // [cols_pad][kLKids] child rows
  const int32_t* e_cnt;   // [cols_pad]
  float* edge_x;          // [B][N] logit of row v's token at its parent
  RowPart* part;          // [B * NI][n_cta]
  int* err;
  int n_stages, bps;
  uint32_t stage_bytes;         // stage stride, sized for the widest pass
};

__device__ __forceinline__ bool l_wait(uint32_t bar, uint32_t parity, const volatile int* abort_flag) {
  const uint64_t t0 = global_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try(bar, parity)) return true;
    if (*abort_flag) return false;
    if ((it & 255u) == 255u && global_ns() - t0 > 2000000000ull) return false;
  }
}

// One block per column: its hidden row into X (zeros for padding columns) and its
// children, found by one warp scanning the parent array in ascending row order.
// Block 0 also clears the error flag of this call.
__global__ void lm_gather_kernel(medusa_tree_t t, int B, int d, const uint16_t* __restrict__ hidden,
                                 const int32_t* __restrict__ tokens, uint16_t* __restrict__ X,
                                 int32_t* __restrict__ e_tok, int32_t* __restrict__ e_row,
                                 int32_t* __restrict__ e_cnt, int* __restrict__ err) {
  const int col = blockIdx.x;
  if (col == 0 && threadIdx.x == 0) *err = 0;
  // Columns b * NI + ii: internal row ii of sequence b (NI, N: the batch's bounds when
  // templates are per sequence; a column past its sequence's internal rows is padding).
  const int NI = t.n_internal, N = t.n_rows;
  const int b = col < B * NI ? col / NI : 0;
  const medusa_tree_t tb = seq_tree(t, b);
  const bool valid = col < B * NI && col % NI < tb.n_internal;
  const int u = valid ? tb.internal[col % NI] : 0;
  const int Nb = tb.n_rows;
  const uint4* src = reinterpret_cast<const uint4*>(hidden + ((int64_t)b * N + u) * d);
  uint4* dst = reinterpret_cast<uint4*>(X + (int64_t)col * d);
  for (int i = threadIdx.x; i < d / 8; i += blockDim.x) dst[i] = valid ? src[i] : make_uint4(0u, 0u, 0u, 0u);
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int cnt = 0;
    for (int v0 = 1; valid && v0 < Nb; v0 += 32) {
      const int v = v0 + lane;
      const bool kid = v < Nb && tb.parent[v] == u;
      const unsigned m = __ballot_sync(0xffffffffu, kid);
      if (kid) {
        const int slot = cnt + __popc(m & ((1u << lane) - 1u));
        if (slot < kLKids) {
          e_tok[col * kLKids + slot] = tokens[(int64_t)b * N + v];
          e_row[col * kLKids + slot] = v;
        }
      }
      cnt += __popc(m);
    }
    if (lane == 0) e_cnt[col] = cnt < kLKids ? cnt : kLKids;
  }
}

// Argmax of the raw logits, the lowest id among equal values.
__device__ __forceinline__ void lm_fold_argmax(float x, int id, float& av, int& ai) {
  if (ranks_before(x, id, av, ai)) {
    av = x;
    ai = id;
  }
}

// Merge chunk statistics q into (m, z, s1) and the argmax (log-sum-exp with first moment).
__device__ __forceinline__ void lm_merge(float& m, float& z, float& s1, float& av, int& ai, const RowPart& q) {
  if (ranks_before(q.amax_v, q.amax_i, av, ai)) {
    av = q.amax_v;
    ai = q.amax_i;
  }
  if (q.z <= 0.f) return;
  if (z <= 0.f) {
    m = q.m;
    z = q.z;
    s1 = q.s1;
    return;
  }
  const float mn = fmaxf(m, q.m);
  const float a = expf(m - mn), c = expf(q.m - mn);
  s1 = a * (s1 + (m - mn) * z) + c * (q.s1 + (q.m - mn) * q.z);
  z = a * z + c * q.z;
  m = mn;
}

template <bool TYP>
__global__ void __launch_bounds__(kLThreads, 1)
    lm_stats_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX0,
                    const __grid_constant__ CUtensorMap tmX1, const __grid_constant__ CUtensorMap tmX2,
                    const __grid_constant__ CUtensorMap tmX3, const LmArgs a) {
  extern __shared__ uint8_t smem_l[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_l) + 1023) & ~uintptr_t(1023));
  const int pass = blockIdx.x % a.n_pass, cta = blockIdx.x / a.n_pass, n_cta = a.n_cta;
  const int S = a.n_stages, NM = a.n_mma[pass], bps = a.bps;
  const int col0 = a.col0[pass], n_cols = a.n_cols[pass];
  const CUtensorMap* tmX = pass == 0 ? &tmX0 : pass == 1 ? &tmX1 : pass == 2 ? &tmX2 : &tmX3;
  // stages, then (at the end) the merge buffer in the same bytes, then the tiles
  const size_t region = (size_t)S * a.stage_bytes > kLMergeBytes ? (size_t)S * a.stage_bytes : kLMergeBytes;
  float* tiles = reinterpret_cast<float*>(sm + region);                          // [4][32][33]
  uint64_t* bars = reinterpret_cast<uint64_t*>(tiles + 4 * 32 * kTileStride);
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  const uint32_t full0 = smem_u32(&bars[0]), empty0 = smem_u32(&bars[S]);
  const uint32_t dfull0 = smem_u32(&bars[2 * S]), dempty0 = smem_u32(&bars[2 * S + 2]);
  const uint32_t drain = smem_u32(&bars[2 * S + 4]);
  const volatile int* abortp = &abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_groups = (a.V + kLRows - 1) / kLRows;
  const int n_k = a.d / (kLKc * bps);                // stages per group
  const uint32_t a_bytes = kLRows * kLKc * 2, b_bytes = (uint32_t)NM * kLKc * 2;
  const uint32_t tmem_cols = (uint32_t)(2 * NM <= 32 ? 32 : 2 * NM <= 64 ? 64 : 2 * NM <= 128 ? 128 : 2 * NM <= 256 ? 256 : 512);

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
    // ---- TMA producer: every group of this CTA, n_k stages each ----------------------
    if (lane == 0) {
      const uint32_t tx = (uint32_t)bps * (a_bytes + b_bytes);   // bytes of this pass's stage
      for (int g = cta; g < n_groups && ok; g += n_cta) {
        for (int kc = 0; kc < n_k; ++kc) {
          const int s = slot % S;
          if (!l_wait(empty0 + 8 * s, (uint32_t)(((slot / S) & 1) ^ 1), abortp)) {
            ok = false;
            break;
          }
          const uint32_t sA = smem_u32(sm + (size_t)s * a.stage_bytes), sB = sA + bps * a_bytes;
          const uint32_t bar = full0 + 8 * s;
          mbar_expect_tx(bar, tx);
          for (int bx = 0; bx < bps; ++bx) {
            const int col = (kc * bps + bx) * kLKc;
            tma_load_2d(sA + bx * a_bytes, &tmW, col, g * kLRows, bar);
            tma_load_2d(sB + bx * b_bytes, tmX, col, col0, bar);
          }
          ++slot;
        }
      }
      if (!ok) give_up();
    }
  } else if (warp == 1) {
    // ---- MMA issue: group gl of this CTA into accumulator gl & 1 -----------------------
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(kLRows, NM);
      int u = 0;
      for (int gl = 0; ok && cta + gl * n_cta < n_groups; ++gl) {
        const int db = gl & 1;
        // the accumulator must have been read out (group gl - 2) before it is reused
        if (gl >= 2 && !l_wait(dempty0 + 8 * db, (uint32_t)(((gl >> 1) - 1) & 1), abortp)) {
          ok = false;
          break;
        }
        for (int kc = 0; kc < n_k; ++kc, ++u) {
          const int s = u % S;
          if (!l_wait(full0 + 8 * s, (uint32_t)((u / S) & 1), abortp)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sA = smem_u32(sm + (size_t)s * a.stage_bytes), sB = sA + bps * a_bytes;
          for (int bx = 0; bx < bps; ++bx) {
#pragma unroll
            for (int kk = 0; kk < kLKc / 16; ++kk)
              umma_f16(tmem + (uint32_t)(db * NM), sw128_desc(sA + bx * a_bytes + kk * 32, 16, 1024),
                       sw128_desc(sB + bx * b_bytes + kk * 32, 16, 1024), idesc,
                       (kc > 0 || bx > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(empty0 + 8 * s);                   // the stage is free once these MMAs are done
        }
        if (!ok) break;
        umma_commit(dfull0 + 8 * db);
      }
      if (!ok) give_up();
    }
  } else {
    // ---- epilogue: warp q = warp % 4 reads TMEM lanes [32q, 32q + 32) ----------------------
    const int q = warp & 3;
    float* tile = tiles + q * 32 * kTileStride;
    // running statistics of column 32 ch + lane, ch < NM / 32
    float st_m[kLMaxCols / 32], st_z[kLMaxCols / 32], st_s1[kLMaxCols / 32], st_av[kLMaxCols / 32];
    int st_ai[kLMaxCols / 32];
#pragma unroll
    for (int ch = 0; ch < kLMaxCols / 32; ++ch) {
      st_m[ch] = -INFINITY;
      st_z[ch] = 0.f;
      st_s1[ch] = 0.f;
      st_av[ch] = -INFINITY;
      st_ai[ch] = INT_MAX;
    }
    for (int gl = 0; cta + gl * n_cta < n_groups; ++gl) {
      const int g = cta + gl * n_cta;
      const int db = gl & 1;
      if (!__all_sync(0xffffffffu, l_wait(dfull0 + 8 * db, (uint32_t)((gl >> 1) & 1), abortp))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int id0 = g * kLRows + 32 * q;            // vocabulary id of tile row 0
#pragma unroll
      for (int ch = 0; ch < kLMaxCols / 32; ++ch) {
        if (32 * ch >= NM) break;                      // uniform
        float v[32];
        tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(db * NM + 32 * ch), v);
#pragma unroll
        for (int j = 0; j < 32; ++j) tile[lane * kTileStride + j] = v[j];   // row = lane (one vocabulary id)
        __syncwarp();
        const int c = 32 * ch + lane;                  // this lane's column
        if (c < n_cols) {
          const int n_valid = min(32, a.V - id0);      // ids past V are padding rows of W_LM
          float av = st_av[ch];
          int ai = st_ai[ch];
          for (int i = 0; i < n_valid; ++i) lm_fold_argmax(tile[i * kTileStride + lane], id0 + i, av, ai);
          st_av[ch] = av;
          st_ai[ch] = ai;
          if (TYP && n_valid > 0) {
            float mb = -INFINITY;
            for (int i = 0; i < n_valid; ++i) mb = fmaxf(mb, tile[i * kTileStride + lane] * a.inv_temp);
            float m = st_m[ch], z = st_z[ch], s1 = st_s1[ch];
            if (z == 0.f) {
              m = mb;
            } else if (mb > m) {
              const float sc = expf(m - mb);
              s1 = sc * (s1 + (m - mb) * z);
              z *= sc;
              m = mb;
            }
            for (int i = 0; i < n_valid; ++i) {
              const float dlt = tile[i * kTileStride + lane] * a.inv_temp - m;
              const float ev = expf(dlt);
              z += ev;
              s1 = fmaf(ev, dlt, s1);
            }
            st_m[ch] = m;
            st_z[ch] = z;
            st_s1[ch] = s1;
            // the logit of each child's token, where that token is one of these ids
            const int cg = col0 + c;
            const int nk = a.e_cnt[cg];
            for (int e = 0; e < nk; ++e) {
              const int r = a.e_tok[cg * kLKids + e] - id0;
              if (r >= 0 && r < n_valid) {
                const int b = cg / a.NI;
                a.edge_x[(int64_t)b * a.N + a.e_row[cg * kLKids + e]] = tile[r * kTileStride + lane];
              }
            }
          }
        }
        __syncwarp();                                  // the tile is rewritten by the next chunk
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dempty0 + 8 * db);
    }
    if (!ok && lane == 0) give_up();

    // ---- merge the four warps' statistics per column; write this CTA's chunk -----------
    // (the stage buffers are free: the last accumulator was complete, so every copy and
    // MMA has finished)
    // (after a failure copies may still be landing: the statistics are void anyway)
    // One array per statistic ([4][kLMaxCols] each): a warp's stores and a thread's
    // loads touch consecutive 4-byte words, free of bank conflicts.
    float* mg_m = reinterpret_cast<float*>(sm);
    float* mg_z = mg_m + 4 * kLMaxCols;
    float* mg_s1 = mg_z + 4 * kLMaxCols;
    float* mg_av = mg_s1 + 4 * kLMaxCols;
    int* mg_ai = reinterpret_cast<int*>(mg_av + 4 * kLMaxCols);
    const bool intact = *abortp == 0;
#pragma unroll
    for (int ch = 0; ch < kLMaxCols / 32; ++ch) {
      if (32 * ch >= NM || !intact) break;
      const int e = q * kLMaxCols + 32 * ch + lane;
      mg_m[e] = st_m[ch];
      mg_z[e] = st_z[ch];
      mg_s1[e] = st_s1[ch];
      mg_av[e] = st_av[ch];
      mg_ai[e] = st_ai[ch];
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");   // the four epilogue warps
    for (int c = (warp - 2) * 32 + lane; intact && c < n_cols; c += 128) {
      float m = -INFINITY, z = 0.f, s1 = 0.f, av = -INFINITY;
      int ai = INT_MAX;
      for (int w = 0; w < 4; ++w) {
        const int e = w * kLMaxCols + c;
        RowPart r;
        r.m = mg_m[e];
        r.z = mg_z[e];
        r.s1 = mg_s1[e];
        r.amax_v = mg_av[e];
        r.amax_i = mg_ai[e];
        lm_merge(m, z, s1, av, ai, r);
      }
      RowPart out;
      out.m = m;
      out.z = z;
      out.s1 = s1;
      out.amax_v = av;
      out.amax_i = ai;
      out.pad[0] = out.pad[1] = out.pad[2] = 0;
      a.part[(int64_t)(col0 + c) * n_cta + cta] = out;
    }
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

// Stage layout: bps boxes of W_LM (128 x 64) and of the packed rows (NM x 64) per
// stage; as many boxes per stage as still leave four stages, else two.
size_t lm_stage_bytes(int NM, int bps) { return (size_t)bps * ((size_t)kLRows * kLKc * 2 + (size_t)NM * kLKc * 2); }
// alignment slack, the epilogue tiles, and the barriers (2 S + 5 <= 21 of 8 bytes)
constexpr size_t kLFixed = 1024 + 4 * 32 * kTileStride * sizeof(float) + 32 * 8;
constexpr size_t kLBudget = 227 * 1024 - kLFixed;
int lm_bps(int NM, int d) {
  for (int bps = 4; bps > 1; bps >>= 1)
    if ((d / kLKc) % bps == 0 && kLBudget / lm_stage_bytes(NM, bps) >= 4) return bps;
  return 1;
}
int lm_stages(int NM, int d) {
  int s = (int)(kLBudget / lm_stage_bytes(NM, lm_bps(NM, d)));
  return s > 8 ? 8 : s;                  // at most 8 stages: 2 * 8 + 5 barriers fit the 32 reserved
}
size_t lm_smem(int NM, int d) {
  const size_t stages = (size_t)lm_stages(NM, d) * lm_stage_bytes(NM, lm_bps(NM, d));
  return kLFixed + (stages > kLMergeBytes ? stages : kLMergeBytes);   // the merge reuses the stages
}

bool encode_rows(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {(cuuint32_t)kLKc, box_rows}, estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool lm_accept_supported(int d, int V) {
  if (d < kLKc || d % kLKc != 0 || V < 1 || !encode_fn()) return false;
  return lm_stages(kLMaxCols, d) >= 2;
}

LmAcceptPlan plan_lm_accept(const medusa_tree_t& t, int B, int V, int d) {
  LmAcceptPlan p{};
  p.B = B;
  p.V = V;
  p.d = d;
  p.NI = t.n_internal;
  p.cols = B * t.n_internal;
  p.cols_pad = (p.cols + 31) / 32 * 32;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // CTAs per pass set: the SMs shared by the sets of the widest launch
  int sets = (p.cols + kLMaxCols - 1) / kLMaxCols;
  if (sets > kLMaxPass) sets = kLMaxPass;
  if (sets < 1) sets = 1;
  p.n_chunks = sms / sets;
  size_t off = 0;
  p.off_x = off;
  off = align_up(off + (size_t)p.cols_pad * d * 2, 256);
  p.off_etok = off;
  off = align_up(off + (size_t)p.cols_pad * kLKids * 4, 256);
  p.off_erow = off;
  off = align_up(off + (size_t)p.cols_pad * kLKids * 4, 256);
  p.off_ecnt = off;
  off = align_up(off + (size_t)p.cols_pad * 4, 256);
  p.off_edge_x = off;
  off = align_up(off + (size_t)B * t.n_rows * 4, 256);
  p.off_part = off;
  off = align_up(off + (size_t)(p.cols > 0 ? p.cols : 1) * p.n_chunks * sizeof(RowPart), 256);
  p.off_err = off;
  off = align_up(off + 16, 256);
  p.bytes = off;
  return p;
}

cudaError_t launch_lm_accept(const LmAcceptPlan& p, const medusa_tree_t& t, const void* hidden, const void* w_lm,
                             const int32_t* tokens, int mode, float temperature, float epsilon, float delta,
                             int32_t* best_path, int32_t* accept_len, int32_t* out_tokens, int32_t* out_rows,
                             int32_t* frontier_row, void* ws, cudaStream_t st, const CommitArgs& cm) {
  char* base = static_cast<char*>(ws);
  uint16_t* X = reinterpret_cast<uint16_t*>(base + p.off_x);
  int32_t* e_tok = reinterpret_cast<int32_t*>(base + p.off_etok);
  int32_t* e_row = reinterpret_cast<int32_t*>(base + p.off_erow);
  int32_t* e_cnt = reinterpret_cast<int32_t*>(base + p.off_ecnt);
  float* edge_x = reinterpret_cast<float*>(base + p.off_edge_x);
  RowPart* part = reinterpret_cast<RowPart*>(base + p.off_part);
  int* err = reinterpret_cast<int*>(base + p.off_err);
  cudaError_t e;
  const bool typ = mode == MEDUSA_ACCEPT_TYPICAL;
  if (p.cols == 0) {
    if ((e = cudaMemsetAsync(err, 0, sizeof(int), st)) != cudaSuccess) return e;
  } else {
    lm_gather_kernel<<<p.cols_pad, 256, 0, st>>>(t, p.B, p.d, (const uint16_t*)hidden, tokens, X, e_tok, e_row,
                                                 e_cnt, err);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    CUtensorMap mw;
    if (!encode_rows(&mw, w_lm, p.d, p.V, kLRows)) return cudaErrorInvalidValue;
    // launches of up to kLMaxPass passes; the first pass of a launch is its widest
    for (int l0 = 0; l0 < p.cols; l0 += kLMaxPass * kLMaxCols) {
      LmArgs a{};
      CUtensorMap mx[kLMaxPass];
      a.n_pass = 0;
      for (int c0 = l0; c0 < p.cols && a.n_pass < kLMaxPass; c0 += kLMaxCols, ++a.n_pass) {
        const int n_cols = p.cols - c0 < kLMaxCols ? p.cols - c0 : kLMaxCols;
        const int NM = (n_cols + 31) / 32 * 32;
        if (!encode_rows(&mx[a.n_pass], X, p.d, p.cols_pad, NM)) return cudaErrorInvalidValue;
        a.col0[a.n_pass] = c0;
        a.n_cols[a.n_pass] = n_cols;
        a.n_mma[a.n_pass] = NM;
      }
      for (int i = a.n_pass; i < kLMaxPass; ++i) mx[i] = mx[0];
      const int NM = a.n_mma[0];
      a.V = p.V;
      a.d = p.d;
      a.N = t.n_rows;
      a.NI = p.NI;
      a.n_cta = p.n_chunks;
      a.inv_temp = 1.f / temperature;
      a.e_tok = e_tok;
      a.e_row = e_row;
      a.e_cnt = e_cnt;
      a.edge_x = edge_x;
      a.part = part;
      a.err = err;
      a.bps = lm_bps(NM, p.d);
      a.n_stages = lm_stages(NM, p.d);
      a.stage_bytes = (uint32_t)lm_stage_bytes(NM, a.bps);
      const size_t smem = lm_smem(NM, p.d);
      auto kern = typ ? lm_stats_kernel<true> : lm_stats_kernel<false>;
      if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
        return e;
      kern<<<p.n_chunks * a.n_pass, kLThreads, smem, st>>>(mw, mx[0], mx[1], mx[2], mx[3], a);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
  }
  return launch_select_parts(t, p.B, p.V, p.n_chunks, part, edge_x, err, tokens, mode, temperature, epsilon, delta,
                             best_path, accept_len, out_tokens, out_rows, frontier_row, st, cm);
}

}  // namespace medusa
