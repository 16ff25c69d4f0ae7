// Tree verification attention on tcgen05 tensor cores (bf16 KV cache, head_dim 128).
//
// Split-KV over the committed prefix like the CUDA-core kernel in attn.cu, written for
// sm_103a.  The splits of one (sequence, KV head, 128-row tile) unit form a thread-block
// cluster and merge their partials through distributed shared memory, so no partial
// ever goes to global memory.  Split 0 also streams the N tree rows as extra 64-key
// tiles, masked by one 64-bit ancestor word per row and tile, so the whole tree block
// runs on the tensor cores as well.
//
// One CTA = 128 query rows (tree row x GQA member, the M of the MMA) and one split of
// the prefix, 2 CTAs per SM.  Its eight warps are specialised and run as a pipeline
// coupled by mbarriers, so loading, converting, multiplying and the softmax of
// successive 64-key tiles overlap:
//   - warp 4 (one lane): TMA producer, K and V tiles (128-byte swizzle) into a 2-stage
//     ring;
//   - warps 6-7: re-encode each landed tile from bf16 to fp16 in place (exact for
//     |x| in [2^-14, 65504]); tree-row key tiles are rotated (RoPE at L + depth) on
//     the way;
//   - warp 5 (one lane): allocates TMEM and issues tcgen05.mma: S = Q K^T (M=128,
//     N=64, K=128) into one of two TMEM S buffers, then O += P V (M=128, N=128, K=64)
//     with P read from TMEM and O accumulated in TMEM;
//   - warps 0-3: thread t owns query row t (= TMEM lane t).  They rotate and stage
//     the queries, then run the online softmax: read S with tcgen05.ld, write P over
//     it as fp16 with tcgen05.st, and rescale O in TMEM when the running max grows.
// Operands are fp16: the rotated queries (pre-multiplied by scale * log2 e, so S comes
// out in log2 units) and P are rounded to fp16 (10-bit mantissa; bf16's 7 bits would
// cost ~1.6e-3 relative error each).
// Every mbarrier wait is bounded and also ends when another role has given up; then
// the CTA records MEDUSA_ETIMEOUT for the sequence, waits (bounded) for its
// outstanding copies and MMAs, frees TMEM and still joins the cluster barriers.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace medusa {

namespace {

constexpr int kTcRows = 128;        // query rows per CTA
constexpr int kTcKeys = 64;         // rows of a K/V copy box (and keys per tile with one query tile)
constexpr int kDH = 128;
constexpr int kHalf = kDH / 2;
constexpr uint32_t kTmemO = 128;   // per query tile: S buffers in columns [0, 64), [64, 128); O in [128, 256)

constexpr int kQBytes = kTcRows * kDH * 2;       // 2 K-blocks of [128 rows x 128 B]

constexpr int kErrTimeout = MEDUSA_ETIMEOUT;
constexpr int kMaxClusterSplits = 8;   // splits of a unit form one portable cluster

struct TcArgs {
  medusa_tree_t t;
  medusa_kv_t c;
  const uint16_t* q;
  const uint16_t* k_new;
  const uint16_t* v_new;
  const int32_t* L;
  float* out;
  float* lse;
  int32_t* status;
  int B, Hq, Hkv, g, n_mt, n_split, chunk, first;
  float scale_log2;
  uint64_t stall_ns;     // test hook (0 = off): wait this long on a barrier nothing completes
  float th_hi[64], th_lo[64];
};

// Eight non-blocking phase tests in one round trip: all tests are issued before any
// result is used.  Bit i of the result: phase parity p[i] of barrier b[i] has completed.
__device__ __forceinline__ uint32_t mbar_test8(const uint32_t (&b)[8], const uint32_t (&p)[8]) {
  uint32_t m;
  asm volatile(
      "{\n\t.reg .pred q0, q1, q2, q3, q4, q5, q6, q7;\n\t.reg .u32 r0, r1, r2, r3, r4, r5, r6, r7;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 q0, [%1], %9;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 q1, [%2], %10;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 q2, [%3], %11;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 q3, [%4], %12;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 q4, [%5], %13;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 q5, [%6], %14;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 q6, [%7], %15;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 q7, [%8], %16;\n\t"
      "selp.u32 r0, 1, 0, q0;\n\tselp.u32 r1, 2, 0, q1;\n\tselp.u32 r2, 4, 0, q2;\n\tselp.u32 r3, 8, 0, q3;\n\t"
      "selp.u32 r4, 16, 0, q4;\n\tselp.u32 r5, 32, 0, q5;\n\tselp.u32 r6, 64, 0, q6;\n\tselp.u32 r7, 128, 0, q7;\n\t"
      "or.b32 r0, r0, r1;\n\tor.b32 r2, r2, r3;\n\tor.b32 r4, r4, r5;\n\tor.b32 r6, r6, r7;\n\t"
      "or.b32 r0, r0, r2;\n\tor.b32 r4, r4, r6;\n\tor.b32 %0, r0, r4;\n\t}"
      : "=r"(m)
      : "r"(b[0]), "r"(b[1]), "r"(b[2]), "r"(b[3]), "r"(b[4]), "r"(b[5]), "r"(b[6]), "r"(b[7]), "r"(p[0]),
        "r"(p[1]), "r"(p[2]), "r"(p[3]), "r"(p[4]), "r"(p[5]), "r"(p[6]), "r"(p[7])
      : "memory");
  return m;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// 2^x on the MUFU unit (ex2.approx, relative error ~2^-22); 2^-inf = +0.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Shared::cluster address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem_addr(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ float2 ld_dsmem_f2(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0,%1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// bf16 x8 (uint4) -> fp16 x8 (uint4), exact for normal-range values.
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 v) {
  uint4 o;
  o.x = pack_half2(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u));
  o.y = pack_half2(__uint_as_float(v.y << 16), __uint_as_float(v.y & 0xFFFF0000u));
  o.z = pack_half2(__uint_as_float(v.z << 16), __uint_as_float(v.z & 0xFFFF0000u));
  o.w = pack_half2(__uint_as_float(v.w << 16), __uint_as_float(v.w & 0xFFFF0000u));
  return o;
}

__device__ __forceinline__ int64_t row_off_tc(const medusa_kv_t& c, int b, int kvh, int row) {
  if (c.page_size == 0) return (((int64_t)b * c.n_kv_heads + kvh) * c.capacity + row) * c.head_dim;
  const int page = c.block_table[(int64_t)b * c.max_blocks + row / c.page_size];
  return (((int64_t)page * c.n_kv_heads + kvh) * c.page_size + row % c.page_size) * c.head_dim;
}


// Wait for a phase; gives up (false) after ~limit_ns (2 s by default) or as soon as
// another role of the CTA has set the abort flag.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, const volatile int* abort_flag,
                                              uint64_t limit_ns = 2000000000ull) {
  const uint64_t t0 = global_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try(bar, parity)) return true;
    if (*abort_flag) return false;
    if ((it & 255u) == 255u && global_ns() - t0 > limit_ns) return false;
  }
}



// Re-encode one K or V tile (2 blocks of [KT rows x 128 B], bf16) to fp16 in place;
// rows of keys >= k_valid become zero.  Thread ct of the kConvThreads converter
// threads; all its loads are issued before the first store, so their latencies overlap.
template <int kConvThreads, int KT>
__device__ __forceinline__ void convert_tile(uint8_t* tile, int k_valid, int ct) {
  uint4* p = reinterpret_cast<uint4*>(tile);
  constexpr int kIter = (KT * kDH * 2 / 16) / kConvThreads;
  uint4 v[kIter];
#pragma unroll
  for (int i = 0; i < kIter; ++i) v[i] = p[i * kConvThreads + ct];
#pragma unroll
  for (int i = 0; i < kIter; ++i) {
    const int idx = i * kConvThreads + ct;
    const int row = (idx % (KT * 8)) / 8;             // 16-byte chunks: 8 per row, 8 KT per block
    p[idx] = row < k_valid ? bf16x8_to_f16x8(v[i]) : make_uint4(0, 0, 0, 0);
  }
}

// A tile already in fp16 (read from the cache's fp16 mirror): only the rows of keys
// >= k_valid become zero (rows past a sequence's prefix may hold anything).
template <int kConvThreads, int KT>
__device__ __forceinline__ void zero_tail(uint8_t* tile, int k_valid, int ct) {
  if (k_valid >= KT) return;
  uint4* p = reinterpret_cast<uint4*>(tile);
  constexpr int kIter = (KT * kDH * 2 / 16) / kConvThreads;
#pragma unroll
  for (int i = 0; i < kIter; ++i) {
    const int idx = i * kConvThreads + ct;
    if ((idx % (KT * 8)) / 8 >= k_valid) p[idx] = make_uint4(0, 0, 0, 0);
  }
}

// Tree-row key tile of KT rows: bf16 -> RoPE at L + depth[v] (fp32) -> fp16, in place.
// Row r of the tile is tree row v0 + r; dims i and i + 64 sit in the two blocks at the same
// swizzled position.  Rows >= n_valid become zero.  `dep[i]` is the depth of the row
// that iteration i of thread ct touches (loaded before the tile landed).
template <int kConvThreads>
__device__ __forceinline__ int rotate_row(int i, int ct) { return (i * kConvThreads + ct) >> 3; }

template <int kConvThreads, int KT>
__device__ __forceinline__ void convert_rotate_tile(uint8_t* tile, int n_valid, const int* dep,
                                                    const float* tab_c, const float* tab_s, int ct) {
  constexpr int kRotIter = (KT * 8) / kConvThreads;
#pragma unroll
  for (int i = 0; i < kRotIter; ++i) {
    const int idx = i * kConvThreads + ct;
    const int row = idx >> 3, c = idx & 7;
    const int off = row * 128 + ((c ^ (row & 7)) * 16);
    uint4* p0 = reinterpret_cast<uint4*>(tile + off);
    uint4* p1 = reinterpret_cast<uint4*>(tile + KT * 128 + off);
    if (row < n_valid) {
      float x1[8], x2[8];
      Elem<uint16_t>::unpack(*p0, x1);
      Elem<uint16_t>::unpack(*p1, x2);
      const int ti = dep[i] * kHalf + 8 * c;
      float y1[8], y2[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float cs = tab_c[ti + e], sn = tab_s[ti + e];
        y1[e] = x1[e] * cs - x2[e] * sn;
        y2[e] = x2[e] * cs + x1[e] * sn;
      }
      *p0 = make_uint4(pack_half2(y1[0], y1[1]), pack_half2(y1[2], y1[3]), pack_half2(y1[4], y1[5]),
                       pack_half2(y1[6], y1[7]));
      *p1 = make_uint4(pack_half2(y2[0], y2[1]), pack_half2(y2[2], y2[3]), pack_half2(y2[4], y2[5]),
                       pack_half2(y2[6], y2[7]));
    } else {
      *p0 = make_uint4(0, 0, 0, 0);
      *p1 = make_uint4(0, 0, 0, 0);
    }
  }
}

// Kernel configuration: QT query tiles of 128 rows per CTA share every K/V tile (one
// copy, one conversion); NS stages of KT keys in the ring.
//  QT = 1: KT = 64, two S buffers per query tile (S of the next tile is computed while
//          the softmax works on this one); two CTAs per SM.
//  QT = 2: KT = 128, one S buffer per query tile; the two tiles alternate on the tensor
//          cores (S and P V of one tile while the softmax works on the other).  128-key
//          tiles make the S MMAs 128 wide, which run at the full rate, where 64-wide
//          ones, with both operands in shared memory, are held to about two thirds
//          of it by their operand traffic.  One CTA per SM.
template <int QT, int NS>
struct TcCfg {
  static constexpr int kKT = 64 * QT;                // keys per tile
  static constexpr int kSB = QT == 1 ? 2 : 1;        // S buffers per query tile
  static constexpr int kKBytes = kKT * kDH * 2;      // one K (or V) tile: 2 dim blocks of [KT rows x 128 B]
  static constexpr int kStageBytes = 2 * kKBytes;
  static constexpr int kSoftWarps = 4 * QT;          // warps [0, 4 QT): one thread per query row
  static constexpr int kProdWarp = 4 * QT;           // TMA producer
  static constexpr int kMmaWarp = 4 * QT + 1;        // TMEM owner and MMA issuer
  static constexpr int kConvWarp0 = 4 * QT + 2;      // converter warps: one per SM sub-partition
  static constexpr int kConvWarps = QT == 2 ? 4 : 2; // (two when two CTAs share an SM)
  static constexpr int kConvThreads = 32 * kConvWarps;
  static constexpr int kRotIter = (kKT * 8) / kConvThreads;
  static constexpr int kThreads = 32 * (4 * QT + 2 + kConvWarps);
  static constexpr int kRows = kTcRows * QT;
  static constexpr uint32_t kTmemCols = 256u * QT;   // per query tile: S [0, 128) (two 64-wide or one 128-wide), O [128, 256)
  static constexpr int kOffK = kQBytes * QT;                    // K ring: NS slots of kKBytes
  static constexpr int kOffV = kOffK + NS * kKBytes;            // V ring: NS slots of kKBytes
  static constexpr int kOffTable = kOffV + NS * kKBytes;        // rope cos/sin, then barriers
  static constexpr int kPages = kKT / 16;            // pages of a paged tile
  // barrier slots
  // K and V have rings of their own: a K slot is released when the S MMAs that read it
  // complete, well before the P V MMAs release the V slot of the same tile.
  static constexpr int kBarFullK = 0;                // [NS] K slot landed (TMA transaction bytes)
  static constexpr int kBarFullV = NS;               // [NS] V slot landed
  static constexpr int kBarConvK = 2 * NS;           // [NS] K tile converted (one arrival per converter thread)
  static constexpr int kBarConvV = 3 * NS;           // [NS] V tile converted
  static constexpr int kBarEmptyK = 4 * NS;          // [NS] K slot consumed by the S MMAs (tcgen05.commit)
  static constexpr int kBarEmptyV = 5 * NS;          // [NS] V slot consumed by the P V MMAs
  static constexpr int kBarSFull = 6 * NS;                   // [QT][kSB] S buffer written (tcgen05.commit)
  static constexpr int kBarPFull = kBarSFull + QT * kSB;     // [QT][kSB] P written over S (one arrival per softmax warp)
  static constexpr int kBarODone = kBarPFull + QT * kSB;     // [QT][kSB] P V MMAs complete
  static constexpr int kBarQReady = kBarODone + QT * kSB;    // queries staged (one arrival per warp)
  static constexpr int kBarDrain = kBarQReady + 1;           // final commit on the error path
  static constexpr int kBarQFull = kBarQReady + 2;           // query tiles landed
  static constexpr int kBarNever = kBarQReady + 3;           // test hook: never completes
  static constexpr int kBarOFinal = kBarQReady + 4;          // QT = 2: every MMA complete (one commit)
  static constexpr int kNumBars = kBarQReady + 5;
  // the merge reuses the query and stage buffers: [rows][32] float4 O, then (m, l)
  static_assert(QT * kQBytes + NS * kStageBytes >= kRows * (kDH * 4 + 8), "merge buffers do not fit");
};

template <bool PAGED, int QT, int NS>
__global__ void __launch_bounds__(TcCfg<QT, NS>::kThreads, (QT == 1 && NS == 2) ? 2 : 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const __grid_constant__ CUtensorMap tmKn, const __grid_constant__ CUtensorMap tmVn,
                   const __grid_constant__ CUtensorMap tmQ, const TcArgs a) {
  using C = TcCfg<QT, NS>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int D = a.t.max_depth;                        // (a bound over the batch with per-sequence templates)
  float* tab_c = reinterpret_cast<float*>(sm + C::kOffTable);     // [(D+1)][64]
  float* tab_s = tab_c + (D + 1) * kHalf;
  uint64_t* bars = reinterpret_cast<uint64_t*>(
      (reinterpret_cast<uintptr_t>(tab_s + (D + 1) * kHalf) + 7) & ~uintptr_t(7));
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ medusa_tree_t s_tree;                  // this sequence's template

  const int ct_idx = blockIdx.x, s = blockIdx.y;     // ct_idx: which QT row tiles
  // Units of longer sequences start first (longest-processing-time order, which packs
  // the SMs better when the prefix lengths differ): blockIdx.z / Hkv counts the
  // sequences by decreasing length, ties by index.  Thread t < B ranks sequence t.
  __shared__ int sel_b;
  const int kvh = blockIdx.z % a.Hkv;
  int b = blockIdx.z / a.Hkv;
  if (a.B > 1 && a.B <= C::kThreads) {
    if (threadIdx.x < a.B) {
      const int Lt = a.L[threadIdx.x];
      int rank = 0;
      for (int o = 0; o < a.B; ++o) {
        const int Lo = a.L[o];
        rank += (Lo > Lt || (Lo == Lt && o < (int)threadIdx.x)) ? 1 : 0;
      }
      if (rank == b) sel_b = threadIdx.x;
    }
    __syncthreads();
    b = sel_b;
  }
  if (threadIdx.x == 0) s_tree = seq_tree(a.t, b);
  __syncthreads();
  const medusa_tree_t& t = s_tree;
  // NSTR: row stride of q, k_new, v_new and out (the batch's bound); N: this sequence's rows
  const int NSTR = a.t.n_rows, N = t.n_rows, g = a.g, M = N * g;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (C::kRows * ct_idx >= M) return;               // row tiles past this sequence's rows: the whole cluster
  const int Lb = a.L[b];
  const bool first_cta = (s == 0 && ct_idx == 0 && kvh == 0 && tid == 0);
  if (Lb < 0 || !seq_rows_ok(a.c, b, (int64_t)Lb + N)) {
    if (first_cta) a.status[b] = MEDUSA_ECAPACITY;
    return;
  }
  if (Lb > a.first + (a.n_split - 1) * a.chunk) {
    if (first_cta) a.status[b] = MEDUSA_EINVAL;
    return;
  }
  // (status[b] was cleared before the launch; CTAs write errors only, so no CTA can
  // overwrite another's error with success)

  // Rows of this CTA: tiles QT * ct_idx .. + QT - 1 of 128 rows; CTA row r (= softmax
  // thread r) is global row R = 128 * QT * ct_idx + r.  A softmax warp whose 32 rows
  // all lie past the end is idle.
  const int row0 = C::kRows * ct_idx;
  const int rows_valid = min(C::kRows, M - row0);
  const bool soft = warp < C::kSoftWarps;
  const bool live = soft && warp * 32 < rows_valid;            // warp-uniform
  const int R = row0 + tid;
  const bool row_ok = soft && R < M;
  const int u = row_ok ? R / g : 0;
  const int qt = warp >> 2;                                   // query tile of a softmax warp
  const int qt_live = min(QT, (rows_valid + kTcRows - 1) / kTcRows);   // tiles with rows

  const uint32_t bar0 = smem_u32(bars);
  auto BAR = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };

  // Keys of this split.  Each sequence spreads its own ceil(L / KT) prefix tiles over
  // the n_split splits, so a short sequence does not leave splits idle while one of
  // them streams everything.  The tree tiles count as work of split 0, which takes
  // that many fewer prefix tiles.
  constexpr int KT = C::kKT;
  const int ns = a.n_split;
  const int tiles_b = (Lb + KT - 1) / KT;
  const int n_tree_all = (N + KT - 1) / KT;
  const int first_t = ns > 1 ? min(max((tiles_b + n_tree_all + ns - 1) / ns - n_tree_all, 0), tiles_b) : tiles_b;
  const int chunk_t = ns > 1 ? (tiles_b - first_t + ns - 2) / (ns - 1) : 0;
  const int t_begin = s == 0 ? 0 : min(tiles_b, first_t + (s - 1) * chunk_t);
  const int t_end = s == 0 ? first_t : min(tiles_b, first_t + s * chunk_t);
  const int k_begin = t_begin * KT;
  const int k_end = min(Lb, t_end * KT);
  // Tiles: the split's prefix keys, then (split 0 only) the N tree rows, KT per tile.
  // A tree tile t covers rows [KT t, KT t + KT), exactly ancestor-mask words
  // (KT / 64) t .. (KT / 64) t + KT / 64 - 1.
  const int n_pre = k_end > k_begin ? (k_end - k_begin + KT - 1) / KT : 0;
  const int n_tree = (s == 0) ? (N + KT - 1) / KT : 0;
  const int n_tiles = n_pre + n_tree;
  auto tile_valid = [&](int j) -> int {        // rows of tile j before the end of its range
    return j >= n_pre ? N - (j - n_pre) * KT : k_end - (k_begin + j * KT);
  };
  // Pages of a paged prefix tile j (block-table entries), loaded ahead of its copy.
  auto load_pages = [&](int j, int* pg) {
    if (PAGED && j < n_pre) {
      const int k0 = k_begin + j * KT;
      const int np = (min(KT, k_end - k0) + 15) / 16;
      const int32_t* bt = a.c.block_table + (int64_t)b * a.c.max_blocks + k0 / 16;
#pragma unroll
      for (int p = 0; p < C::kPages; ++p) pg[p] = p < np ? __ldg(bt + p) : 0;
    } else {
#pragma unroll
      for (int p = 0; p < C::kPages; ++p) pg[p] = 0;
    }
  };
  // TMA of K (kv = 0) or V (kv = 1) of tile j into slot j % NS of its ring (the slot's
  // full barrier counts the bytes).  A slot holds 2 dim blocks (dims [0, 64), [64, 128))
  // of [KT rows x 128 B]; a copy box is 64 rows (a page of 16 rows when paged).
  auto issue_kv = [&](int kv, int j, const int* page) {
    const int st = j % NS;
    const uint32_t bar = BAR((kv ? C::kBarFullV : C::kBarFullK) + st);
    const uint32_t dst = smem_u32(sm + (kv ? C::kOffV : C::kOffK) + st * C::kKBytes);
    const CUtensorMap* tm = kv ? &tmV : &tmK;
    const CUtensorMap* tmn = kv ? &tmVn : &tmKn;
    constexpr uint32_t kBlk = KT * 128;         // bytes of one dim block
    const int k0 = k_begin + j * KT;
    if (j >= n_pre) {
      const int v0 = (j - n_pre) * KT;
      mbar_expect_tx(bar, C::kKBytes);
#pragma unroll
      for (int h = 0; h < KT / 64; ++h) {
        tma_load_4d(dst + h * 8192, tmn, 0, kvh, v0 + 64 * h, b, bar);
        tma_load_4d(dst + kBlk + h * 8192, tmn, 64, kvh, v0 + 64 * h, b, bar);
      }
    } else if (!PAGED) {
      mbar_expect_tx(bar, C::kKBytes);
#pragma unroll
      for (int h = 0; h < KT / 64; ++h) {
        tma_load_4d(dst + h * 8192, tm, 0, k0 + 64 * h, kvh, b, bar);
        tma_load_4d(dst + kBlk + h * 8192, tm, 64, k0 + 64 * h, kvh, b, bar);
      }
    } else {
      const int np = (min(KT, k_end - k0) + 15) / 16;
      mbar_expect_tx(bar, (uint32_t)np * 2 * 2048);
#pragma unroll
      for (int p = 0; p < C::kPages; ++p) {
        if (p < np) {
          tma_load_4d(dst + p * 2048, tm, 0, 0, kvh, page[p], bar);
          tma_load_4d(dst + kBlk + p * 2048, tm, 64, 0, kvh, page[p], bar);
        }
      }
    }
  };

  // The producer lane initialises the barriers and starts the first copies at once;
  // the other threads touch the barriers only after the __syncthreads below.
  int n_issued = 0;                // tiles whose K and V copies have both been issued
  int n_issued_k = -1;             // on an abort between the K and V copies of a tile: K's count
  if (tid == C::kProdWarp * 32) {
    abort_flag = 0;
    for (int st = 0; st < NS; ++st) {
      mbar_init(BAR(C::kBarFullK + st), 1);
      mbar_init(BAR(C::kBarFullV + st), 1);
      mbar_init(BAR(C::kBarConvK + st), C::kConvThreads);
      mbar_init(BAR(C::kBarConvV + st), C::kConvThreads);
      mbar_init(BAR(C::kBarEmptyK + st), 1);
      mbar_init(BAR(C::kBarEmptyV + st), 1);
    }
    for (int p = 0; p < QT * C::kSB; ++p) {
      mbar_init(BAR(C::kBarSFull + p), 1);
      mbar_init(BAR(C::kBarPFull + p), 4);
      mbar_init(BAR(C::kBarODone + p), 1);
    }
    mbar_init(BAR(C::kBarQReady), C::kThreads / 32);
    mbar_init(BAR(C::kBarDrain), 1);
    mbar_init(BAR(C::kBarQFull), 1);
    mbar_init(BAR(C::kBarNever), 1);
    mbar_init(BAR(C::kBarOFinal), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    // the query tiles first: rows (u, group member) of each tile, 64 dims per copy
    mbar_expect_tx(BAR(C::kBarQFull), kQBytes * QT);
    for (int q = 0; q < QT; ++q) {
      const uint32_t sQ = smem_u32(sm + q * kQBytes);
      const int u0 = (QT * ct_idx + q) * (kTcRows / g);
      tma_load_4d(sQ, &tmQ, 0, kvh * g, u0, b, BAR(C::kBarQFull));
      tma_load_4d(sQ + 16384, &tmQ, 64, kvh * g, u0, b, BAR(C::kBarQFull));
    }
    int pgs[NS][C::kPages];        // all first-stage lookups in flight together
#pragma unroll
    for (int k = 0; k < NS; ++k) load_pages(k, pgs[k]);
#pragma unroll
    for (int k = 0; k < NS; ++k)
      if (k < n_tiles) {
        issue_kv(0, k, pgs[k]);
        issue_kv(1, k, pgs[k]);
      }
    n_issued = min(n_tiles, NS);
  }
  if (warp == C::kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_slot)),
                 "r"(C::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  for (int idx = tid; idx < (D + 1) * kHalf; idx += C::kThreads) {
    const int dep = idx / kHalf, i = idx % kHalf;
    float sn, cs;
    sincosf(rope_angle(Lb + dep, a.th_hi[i], a.th_lo[i]), &sn, &cs);
    tab_c[idx] = cs;
    tab_s[idx] = sn;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const volatile int* abortp = &abort_flag;

  constexpr uint32_t kIdS = idesc_f16(kTcRows, KT, false);
  constexpr uint32_t kIdO = idesc_f16(kTcRows, kDH, true);
  bool ok = true;
  float m_run = -INFINITY, l_run = 0.f;

  // ---- queries: every warp of the CTA takes part ----------------------------------
  // The query tiles landed by TMA as bf16, K-major with the 128-byte swizzle (dims i
  // and i + 64 of a row at the same position of the two 64-dim blocks).  Each row is
  // rotated in place at L + depth, pre-multiplied by scale * log2 e and stored as fp16.
  // An item is one row's dims [8c, 8c + 8) and [64 + 8c, 64 + 8c + 8).
  // (wait outcomes are made warp-uniform: the softmax's TMEM accesses are warp-collective)
  if (a.stall_ns != 0) {
    // Test hook: a wait on a barrier that nothing completes runs out after stall_ns;
    // the CTA then takes its error path at once (every role sees the abort flag).
    if (!wait_or_abort(BAR(C::kBarNever), 0, abortp, a.stall_ns)) {
      ok = false;
      *const_cast<volatile int*>(abortp) = 1;
    }
  }
  if (!__all_sync(0xffffffffu, wait_or_abort(BAR(C::kBarQFull), 0, abortp))) ok = false;
  if (ok) {
    for (int it = tid; it < rows_valid * 8; it += C::kThreads) {
      const int r = it >> 3, c = it & 7;
      const int tr = r & (kTcRows - 1);
      const int ti0 = __ldg(t.depth + (row0 + r) / g) * kHalf + 8 * c;
      uint4* q0 = reinterpret_cast<uint4*>(sm + (r / kTcRows) * kQBytes + tr * 128) + (c ^ (tr & 7));
      uint4* q1 = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(q0) + 16384);
      float x1[8], x2[8], y1[8], y2[8];
      Elem<uint16_t>::unpack(*q0, x1);
      Elem<uint16_t>::unpack(*q1, x2);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float cs = tab_c[ti0 + e], sn = tab_s[ti0 + e];
        y1[e] = (x1[e] * cs - x2[e] * sn) * a.scale_log2;
        y2[e] = (x2[e] * cs + x1[e] * sn) * a.scale_log2;
      }
      *q0 = make_uint4(pack_half2(y1[0], y1[1]), pack_half2(y1[2], y1[3]), pack_half2(y1[4], y1[5]),
                       pack_half2(y1[6], y1[7]));
      *q1 = make_uint4(pack_half2(y2[0], y2[1]), pack_half2(y2[2], y2[3]), pack_half2(y2[4], y2[5]),
                       pack_half2(y2[6], y2[7]));
    }
  }
  fence_proxy_async();
  __syncwarp();
  if (lane == 0) mbar_arrive(BAR(C::kBarQReady));

  if (warp == C::kProdWarp) {
    // ---- TMA producer: K of tile j >= NS once the S MMAs of tile j - NS freed its K
    //      slot, then V once the P V MMAs of tile j - NS freed its V slot ----------------
    // The block-table entries of a paged tile are loaded one tile ahead of its copies.
    if (lane == 0) {
      int pa[C::kPages], pb[C::kPages];
      load_pages(n_issued, pa);
      load_pages(n_issued + 1, pb);
      for (int j = n_issued; j < n_tiles; ++j) {
        if (!wait_or_abort(BAR(C::kBarEmptyK + j % NS), ((j / NS) - 1) & 1, abortp)) {
          ok = false;
          break;
        }
        issue_kv(0, j, pa);
        if (!wait_or_abort(BAR(C::kBarEmptyV + j % NS), ((j / NS) - 1) & 1, abortp)) {
          ok = false;
          n_issued_k = j + 1;
          break;
        }
        issue_kv(1, j, pa);
        n_issued = j + 1;
#pragma unroll
        for (int p = 0; p < C::kPages; ++p) pa[p] = pb[p];
        load_pages(j + 2, pb);
      }
    }
  } else if (warp == C::kMmaWarp) {
    // ---- MMA issue ------------------------------------------------------------------
    if constexpr (QT == 1) {
      // S(j) = Q K_j^T into TMEM buffer j & 1 once K_j is converted and the P V MMAs of
      // tile j - 2, whose P occupied that buffer, have been issued (this thread's MMAs
      // run in the order it issues them, so S(j) writes the buffer only after they have
      // read it); O += P(j) V_j once the softmax has written P(j) and V_j is converted.
      // Whichever is ready goes first,
      // S before P V when both are; all conditions are tested in one round trip.
      // Completion of P V(j) is signalled on slot j & 1, so that a slot's phase never
      // runs more than one ahead of its waiters.  Every commit covers all MMAs issued
      // before it.
      if (lane == 0) {
        if (!wait_or_abort(BAR(C::kBarQReady), 0, abortp)) ok = false;
        int js = 0, jp = 0;
        uint64_t t_idle = global_ns();
        for (uint32_t spin = 0; ok && jp < n_tiles;) {
          bool did = false;
          // (a test of a tile that does not exist reads a barrier harmlessly and is ignored)
          const uint32_t tb[8] = {BAR(C::kBarConvK + js % NS), BAR(C::kBarConvK + js % NS),
                                  BAR(C::kBarPFull + (jp & 1)), BAR(C::kBarConvV + jp % NS),
                                  BAR(C::kBarConvK + js % NS), BAR(C::kBarConvK + js % NS),
                                  BAR(C::kBarConvK + js % NS), BAR(C::kBarConvK + js % NS)};
          const uint32_t tp[8] = {(uint32_t)(js / NS) & 1u, (uint32_t)(js / NS) & 1u, (uint32_t)(jp >> 1) & 1u,
                                  (uint32_t)(jp / NS) & 1u, 0u, 0u, 0u, 0u};
          const uint32_t ready = mbar_test8(tb, tp);
          if (js < n_tiles && js <= jp + 1 && (ready & 1u)) {
            const int st = js % NS, sb = js & 1;
            tc_fence_after();
            const uint32_t aK = smem_u32(sm + C::kOffK + st * C::kKBytes);
            const uint32_t sQ = smem_u32(sm);
#pragma unroll
            for (int kk = 0; kk < kDH / 16; ++kk) {
              const uint64_t ad = sw128_desc(sQ + (kk / 4) * 16384 + (kk % 4) * 32, 16, 1024);
              const uint64_t bd = sw128_desc(aK + (kk / 4) * (KT * 128) + (kk % 4) * 32, 16, 1024);
              umma_f16(tmem + 64u * sb, ad, bd, kIdS, kk > 0 ? 1u : 0u);
            }
            umma_commit(BAR(C::kBarSFull + sb));
            umma_commit(BAR(C::kBarEmptyK + st));
            ++js;
            did = true;
          }
          if (jp < js && (ready & 4u) && (ready & 8u)) {
            const int st = jp % NS, sb = jp & 1;
            tc_fence_after();
            const uint32_t aV = smem_u32(sm + C::kOffV + st * C::kKBytes);
#pragma unroll
            for (int kk = 0; kk < KT / 16; ++kk) {
              const uint64_t bd = sw128_desc(aV + kk * 2048, KT * 128, 1024);   // MN-major: dim blocks KT x 128 B apart
              umma_f16_ts(tmem + kTmemO, tmem + 64u * sb + 8u * kk, bd, kIdO, (jp > 0 || kk > 0) ? 1u : 0u);
            }
            umma_commit(BAR(C::kBarEmptyV + st));
            umma_commit(BAR(C::kBarODone + sb));
            ++jp;
            did = true;
          }
          if (did) {
            spin = 0;
            t_idle = global_ns();
          } else if (*abortp || ((++spin & 255u) == 0 && global_ns() - t_idle > 2000000000ull)) {
            ok = false;
          }
        }
        // O is final once the last P V MMAs have completed.
        if (ok && n_tiles > 0 &&
            !wait_or_abort(BAR(C::kBarODone + ((n_tiles - 1) & 1)), ((n_tiles - 1) >> 1) & 1, abortp))
          ok = false;
      }
    } else {
      // Two query tiles, one S buffer each, in a fixed order:
      //   S(0, 0), S(1, 0), then for every tile j: P V(0, j), S(0, j + 1), P V(1, j),
      //   S(1, j + 1).
      // S(q, j + 1) overwrites the P of (q, j) in TMEM.  The MMAs of this one issuing
      // thread run in the order it issues them, so S(q, j + 1), issued after P V(q, j),
      // writes those columns only after P V(q, j) has read them: it is issued at once,
      // and the tensor cores go from one query tile's MMAs to the other's without a
      // round trip through a completion barrier.  (When S(q, j + 1) lands, every MMA
      // issued before it has completed, P V(q, j) included: the softmax's rescale of O
      // relies on that.)  A K slot is released after the last query tile's S of its
      // tile, a V slot after the last P V; one final commit tells when O is complete.
      // Each S / P barrier completes once per tile: the phase of tile j is j & 1.
      if (lane == 0) {
        if (!wait_or_abort(BAR(C::kBarQReady), 0, abortp)) ok = false;
        auto issue_s = [&](int q, int j) -> bool {
          const int st = j % NS;
          if (q == 0 && !wait_or_abort(BAR(C::kBarConvK + st), (j / NS) & 1, abortp)) return false;
          tc_fence_after();
          const uint32_t aK = smem_u32(sm + C::kOffK + st * C::kKBytes);
          const uint32_t sQ = smem_u32(sm + q * kQBytes);
#pragma unroll
          for (int kk = 0; kk < kDH / 16; ++kk) {
            const uint64_t ad = sw128_desc(sQ + (kk / 4) * 16384 + (kk % 4) * 32, 16, 1024);
            const uint64_t bd = sw128_desc(aK + (kk / 4) * (KT * 128) + (kk % 4) * 32, 16, 1024);
            umma_f16(tmem + 256u * q, ad, bd, kIdS, kk > 0 ? 1u : 0u);
          }
          umma_commit(BAR(C::kBarSFull + q));
          if (q == qt_live - 1) umma_commit(BAR(C::kBarEmptyK + st));
          return true;
        };
        auto issue_pv = [&](int q, int j) -> bool {
          const int st = j % NS;
          if (q == 0 && !wait_or_abort(BAR(C::kBarConvV + st), (j / NS) & 1, abortp)) return false;
          if (!wait_or_abort(BAR(C::kBarPFull + q), j & 1, abortp)) return false;
          tc_fence_after();
          const uint32_t aV = smem_u32(sm + C::kOffV + st * C::kKBytes);
#pragma unroll
          for (int kk = 0; kk < KT / 16; ++kk) {
            const uint64_t bd = sw128_desc(aV + kk * 2048, KT * 128, 1024);   // MN-major: dim blocks KT x 128 B apart
            umma_f16_ts(tmem + 256u * q + kTmemO, tmem + 256u * q + 8u * kk, bd, kIdO, (j > 0 || kk > 0) ? 1u : 0u);
          }
          if (q == qt_live - 1) umma_commit(BAR(C::kBarEmptyV + st));
          return true;
        };
        // a query tile past the last row (qt_live == 1) is skipped entirely
        if (ok && n_tiles > 0) {
          for (int q = 0; q < qt_live && ok; ++q) ok = issue_s(q, 0);
          for (int j = 0; ok && j < n_tiles; ++j) {
            for (int q = 0; q < qt_live && ok; ++q) {
              ok = issue_pv(q, j);
              if (ok && j + 1 < n_tiles) ok = issue_s(q, j + 1);
            }
          }
          // O is final once every MMA issued above has completed.
          if (ok) {
            umma_commit(BAR(C::kBarOFinal));
            ok = wait_or_abort(BAR(C::kBarOFinal), 0, abortp);
          }
        }
      }
    }
  } else if (warp >= C::kConvWarp0) {
    // ---- bf16 -> fp16 conversion (tree keys also rotated) ------------------------------
    const int ct = tid - C::kConvWarp0 * 32;
    const bool mirror = a.c.k_f16 != nullptr;       // the cache has an fp16 mirror
    for (int j = 0; j < n_tiles; ++j) {
      const int st = j % NS;
      uint8_t* tK = sm + C::kOffK + st * C::kKBytes;
      uint8_t* tV = sm + C::kOffV + st * C::kKBytes;
      const int k_valid = tile_valid(j);
      int dep[C::kRotIter];
      if (j >= n_pre) {
#pragma unroll
        for (int i = 0; i < C::kRotIter; ++i) {
          const int r = rotate_row<C::kConvThreads>(i, ct);
          dep[i] = r < k_valid ? __ldg(t.depth + (j - n_pre) * KT + r) : 0;
        }
      }
      if (!wait_or_abort(BAR(C::kBarFullK + st), (j / NS) & 1, abortp)) {
        ok = false;
        break;
      }
      // (prefix tiles of a cache with an fp16 mirror arrive in fp16 already)
      if (j >= n_pre) convert_rotate_tile<C::kConvThreads, KT>(tK, k_valid, dep, tab_c, tab_s, ct);
      else if (mirror) zero_tail<C::kConvThreads, KT>(tK, k_valid, ct);
      else convert_tile<C::kConvThreads, KT>(tK, k_valid, ct);
      fence_proxy_async();
      mbar_arrive(BAR(C::kBarConvK + st));
      if (!wait_or_abort(BAR(C::kBarFullV + st), (j / NS) & 1, abortp)) {
        ok = false;
        break;
      }
      if (j < n_pre && mirror) zero_tail<C::kConvThreads, KT>(tV, k_valid, ct);
      else convert_tile<C::kConvThreads, KT>(tV, k_valid, ct);
      fence_proxy_async();
      mbar_arrive(BAR(C::kBarConvV + st));
    }
    // Stage the rotated tree keys and the tree values at cache rows L + u while the
    // softmax finishes.  Split 0 runs the tree tiles and finishes last, so the other
    // splits share this work (unit u goes to split 1 + u mod (n_split - 1)).  An item
    // is one unit's dims [8c, 8c + 8) and [64 + 8c, 64 + 8c + 8), the pairs that the
    // rotation mixes.
    const int stagers = ns > 1 ? ns - 1 : 1;
    const int my_stage = ns > 1 ? s - 1 : 0;
    if (ok && my_stage >= 0) {
      const int u_lo = row0 / g, u_hi = (row0 + rows_valid - 1) / g + 1;
      const int u_first = u_lo + ((my_stage - u_lo % stagers) % stagers + stagers) % stagers;
      const int n_mine = u_first < u_hi ? (u_hi - u_first + stagers - 1) / stagers : 0;
      uint16_t* ck = (uint16_t*)a.c.k;
      uint16_t* cv = (uint16_t*)a.c.v;
      for (int it = ct; it < n_mine * 8; it += C::kConvThreads) {
        const int uu = u_first + (it >> 3) * stagers, c = it & 7;
        const int64_t src = (((int64_t)b * NSTR + uu) * a.Hkv + kvh) * kDH + 8 * c;
        const uint4 ka = __ldg(reinterpret_cast<const uint4*>(a.k_new + src));
        const uint4 kb = __ldg(reinterpret_cast<const uint4*>(a.k_new + src + kHalf));
        const uint4 va = __ldg(reinterpret_cast<const uint4*>(a.v_new + src));
        const uint4 vb = __ldg(reinterpret_cast<const uint4*>(a.v_new + src + kHalf));
        const int ti0 = __ldg(t.depth + uu) * kHalf + 8 * c;
        const int64_t dst = row_off_tc(a.c, b, kvh, Lb + uu) + 8 * c;
        float x1[8], x2[8];
        Elem<uint16_t>::unpack(ka, x1);
        Elem<uint16_t>::unpack(kb, x2);
        uint32_t y1[4], y2[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float c0 = tab_c[ti0 + 2 * e], s0 = tab_s[ti0 + 2 * e];
          const float c1 = tab_c[ti0 + 2 * e + 1], s1 = tab_s[ti0 + 2 * e + 1];
          const uint32_t a0 = f32_to_bf16_bits(x1[2 * e] * c0 - x2[2 * e] * s0);
          const uint32_t a1 = f32_to_bf16_bits(x1[2 * e + 1] * c1 - x2[2 * e + 1] * s1);
          const uint32_t b0 = f32_to_bf16_bits(x2[2 * e] * c0 + x1[2 * e] * s0);
          const uint32_t b1 = f32_to_bf16_bits(x2[2 * e + 1] * c1 + x1[2 * e + 1] * s1);
          y1[e] = a0 | (a1 << 16);
          y2[e] = b0 | (b1 << 16);
        }
        const uint4 ya = make_uint4(y1[0], y1[1], y1[2], y1[3]), yb = make_uint4(y2[0], y2[1], y2[2], y2[3]);
        *reinterpret_cast<uint4*>(ck + dst) = ya;
        *reinterpret_cast<uint4*>(ck + dst + kHalf) = yb;
        *reinterpret_cast<uint4*>(cv + dst) = va;
        *reinterpret_cast<uint4*>(cv + dst + kHalf) = vb;
        if (mirror) {                              // the fp16 mirror of the rows just written
          uint16_t* mk = (uint16_t*)a.c.k_f16;
          uint16_t* mv = (uint16_t*)a.c.v_f16;
          *reinterpret_cast<uint4*>(mk + dst) = bf16x8_to_f16x8(ya);
          *reinterpret_cast<uint4*>(mk + dst + kHalf) = bf16x8_to_f16x8(yb);
          *reinterpret_cast<uint4*>(mv + dst) = bf16x8_to_f16x8(va);
          *reinterpret_cast<uint4*>(mv + dst + kHalf) = bf16x8_to_f16x8(vb);
        }
      }
    }
  } else {
    // ---- softmax warps: thread tid owns CTA row tid; warp w reads TMEM lanes of
    //      quadrant w % 4 of query tile w / 4 --------------------------------------------
    // Online softmax.  O accumulates in TMEM across tiles.  The running max m_run is
    // raised only when a tile's max exceeds it by more than 2^8 (log2 units); then O
    // and l are rescaled.  Otherwise P = 2^(s - m_run) <= 256, which fp16 and the fp32
    // accumulators hold exactly enough; the final normalisation uses the same m_run,
    // so the result is the same softmax.
    constexpr float kRescale = 8.f;
    const uint32_t lane_base = ((uint32_t)((warp & 3) * 32) << 16) + 256u * qt;
    // (a query tile past the last row has no MMAs: its warps skip the loop)
    if constexpr (QT == 1) {
    for (int j = 0; ok && j < n_tiles; ++j) {
      const int sb = j & 1;
      const bool tree_tile = j >= n_pre;
      const int k_valid = tile_valid(j);
      const uint64_t vis = (tree_tile && row_ok) ? __ldg(t.anc + (int64_t)u * t.n_words + (j - n_pre)) : 0ull;
      // wait outcomes are made warp-uniform: the TMEM accesses below are warp-collective
      if (!__all_sync(0xffffffffu, wait_or_abort(BAR(C::kBarSFull + sb), (j >> 1) & 1, abortp))) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (live) {
        float sv[kTcKeys];
        tmem_ld64(tmem + lane_base + 64u * sb, sv);
        if (tree_tile) {
#pragma unroll
          for (int c = 0; c < kTcKeys; ++c) sv[c] = ((vis >> c) & 1ull) ? sv[c] : -INFINITY;
        } else if (k_valid < kTcKeys) {
#pragma unroll
          for (int c = 0; c < kTcKeys; ++c) sv[c] = c < k_valid ? sv[c] : -INFINITY;
        }
        float mxp[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int c = 0; c < kTcKeys; c += 4) {
          mxp[0] = fmax3(mxp[0], sv[c], sv[c + 1]);
          mxp[1] = fmax3(mxp[1], sv[c + 2], sv[c + 3]);
        }
        const float mx = fmaxf(mxp[0], mxp[1]);
        // The TMEM accesses of a rescale are warp-collective: the warp rescales when any
        // of its rows needs it, the other rows scale by 1.  O must hold P V of tile j - 1
        // first (a row that needs a rescale has seen an earlier tile, so j >= 1).
        const bool first = (m_run == -INFINITY);
        const bool need = !first && (mx > m_run + kRescale);
        if (first) m_run = mx;                           // O holds nothing yet for this row
        if (__any_sync(0xffffffffu, need)) {
          if (!__all_sync(0xffffffffu,
                          wait_or_abort(BAR(C::kBarODone + ((j - 1) & 1)), ((j - 1) >> 1) & 1, abortp))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float alpha = need ? fast_exp2(m_run - mx) : 1.f;
          l_run *= alpha;
#pragma unroll 1
          for (int q8 = 0; q8 < kDH / 16; ++q8) {
            float ov[16];
            tmem_ld16(tmem + lane_base + kTmemO + 16 * q8, ov);
#pragma unroll
            for (int i = 0; i < 16; ++i) ov[i] *= alpha;
            tmem_st16(tmem + lane_base + kTmemO + 16 * q8, ov);
          }
          if (need) m_run = mx;
        }
        const float mref = (m_run == -INFINITY) ? 0.f : m_run;   // a fully masked row keeps P = 0
        // pairs of keys through the packed fp32x2 adds; four partial sums
        const float2 nm = make_float2(-mref, -mref);
        float2 ps[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        float pk[kTcKeys / 2];                   // P as fp16 pairs, key 2i in the low half
#pragma unroll
        for (int i = 0; i < kTcKeys / 2; ++i) {
          const float2 d = __fadd2_rn(make_float2(sv[2 * i], sv[2 * i + 1]), nm);
          const float2 pp = make_float2(fast_exp2(d.x), fast_exp2(d.y));
          ps[i & 3] = __fadd2_rn(ps[i & 3], pp);
          pk[i] = __uint_as_float(pack_half2(pp.x, pp.y));
        }
        const float2 s01 = __fadd2_rn(ps[0], ps[1]), s23 = __fadd2_rn(ps[2], ps[3]);
        const float2 s4 = __fadd2_rn(s01, s23);
        l_run += s4.x + s4.y;
        tmem_st32(tmem + lane_base + 64u * sb, pk);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(C::kBarPFull + sb));
    }
    } else {
    // Two query tiles of 128-key tiles, one S buffer each.  When S(q, j) lands, the P V
    // MMAs of (q, j - 1) have completed (S(q, j) was issued after them), so O may be
    // rescaled at once.  P is written as fp16 pairs over the S columns already read.
    // While a row has no reference yet (its first tile with keys) the tile is read twice
    // from TMEM, 64 scores at a time: once for the max, once for P.  After that each half
    // is read once: its max is taken from the same registers, and only when it exceeds
    // the reference by more than 2^8 is the reference raised (rare), which rescales O, l,
    // the partial sums and the P of the first half already written by the same factor.
    const uint32_t sbase = tmem + lane_base;
    for (int j = 0; ok && qt < qt_live && j < n_tiles; ++j) {
      const bool tree_tile = j >= n_pre;
      const int k_valid = tile_valid(j);
      uint64_t vis0 = 0ull, vis1 = 0ull;
      if (tree_tile && row_ok) {
        const int w0 = 2 * (j - n_pre);
        vis0 = __ldg(t.anc + (int64_t)u * t.n_words + w0);
        vis1 = w0 + 1 < t.n_words ? __ldg(t.anc + (int64_t)u * t.n_words + w0 + 1) : 0ull;
      }
      // wait outcomes are made warp-uniform: the TMEM accesses below are warp-collective
      if (!__all_sync(0xffffffffu, wait_or_abort(BAR(C::kBarSFull + qt), j & 1, abortp))) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (live) {
        auto load_half = [&](int h, float* sv) {     // scores of keys [64h, 64h + 64), masked
          tmem_ld64(sbase + 64u * h, sv);
          if (tree_tile) {
            const uint64_t vh = h ? vis1 : vis0;
#pragma unroll
            for (int c = 0; c < 64; ++c) sv[c] = ((vh >> c) & 1ull) ? sv[c] : -INFINITY;
          } else if (k_valid < KT) {
#pragma unroll
            for (int c = 0; c < 64; ++c) sv[c] = 64 * h + c < k_valid ? sv[c] : -INFINITY;
          }
        };
        auto max64 = [&](const float* sv) -> float {
          float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
          for (int c = 0; c < 64; c += 4) {
            m0 = fmax3(m0, sv[c], sv[c + 1]);
            m1 = fmax3(m1, sv[c + 2], sv[c + 3]);
          }
          return fmaxf(m0, m1);
        };
        // O *= alpha (per row) in TMEM; warp-collective.
        auto rescale_o = [&](float alpha) {
#pragma unroll 1
          for (int q8 = 0; q8 < kDH / 16; ++q8) {
            float ov[16];
            tmem_ld16(sbase + kTmemO + 16 * q8, ov);
#pragma unroll
            for (int i = 0; i < 16; ++i) ov[i] *= alpha;
            tmem_st16(sbase + kTmemO + 16 * q8, ov);
          }
        };
        float2 ps[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        // P = 2^(s - m_run) of one half as fp16 pairs over S columns [32h, 32h + 32)
        auto write_p = [&](int h, const float* sv) {
          const float mref = (m_run == -INFINITY) ? 0.f : m_run;   // a fully masked row keeps P = 0
          const float2 nm = make_float2(-mref, -mref);
          float pk[32];                            // key 2i in the low half
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float2 d = __fadd2_rn(make_float2(sv[2 * i], sv[2 * i + 1]), nm);
            const float2 pp = make_float2(fast_exp2(d.x), fast_exp2(d.y));
            ps[i & 3] = __fadd2_rn(ps[i & 3], pp);
            pk[i] = __uint_as_float(pack_half2(pp.x, pp.y));
          }
          tmem_st32_nowait(sbase + 32u * h, pk);
        };
        if (__any_sync(0xffffffffu, m_run == -INFINITY)) {
          // no reference yet for some row: the tile's max first
          float mx = -INFINITY;
#pragma unroll 1
          for (int h = 0; h < 2; ++h) {
            float sv[64];
            load_half(h, sv);
            mx = fmaxf(mx, max64(sv));
          }
          const bool first = (m_run == -INFINITY);
          const bool need = !first && (mx > m_run + kRescale);
          if (first) m_run = mx;                         // O holds nothing yet for this row
          if (__any_sync(0xffffffffu, need)) {
            const float alpha = need ? fast_exp2(m_run - mx) : 1.f;
            l_run *= alpha;
            rescale_o(alpha);
            if (need) m_run = mx;
          }
#pragma unroll 1
          for (int h = 0; h < 2; ++h) {
            float sv[64];
            load_half(h, sv);
            write_p(h, sv);
          }
        } else {
#pragma unroll 1
          for (int h = 0; h < 2; ++h) {
            float sv[64];
            load_half(h, sv);
            const float mx = max64(sv);
            const bool need = mx > m_run + kRescale;
            if (__any_sync(0xffffffffu, need)) {
              const float alpha = need ? fast_exp2(m_run - mx) : 1.f;
              l_run *= alpha;
#pragma unroll
              for (int i = 0; i < 4; ++i) ps[i] = make_float2(ps[i].x * alpha, ps[i].y * alpha);
              rescale_o(alpha);
              if (h == 1) {                              // the first half's P, already written
                tmem_wait_st();
                float pk[32];
                tmem_ld32(sbase, pk);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                  const uint32_t w = __float_as_uint(pk[i]);
                  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w));
                  pk[i] = __uint_as_float(pack_half2(f.x * alpha, f.y * alpha));
                }
                tmem_st32(sbase, pk);
              }
              if (need) m_run = mx;
            }
            write_p(h, sv);
          }
        }
        tmem_wait_st();
        const float2 s01 = __fadd2_rn(ps[0], ps[1]), s23 = __fadd2_rn(ps[2], ps[3]);
        const float2 s4 = __fadd2_rn(s01, s23);
        l_run += s4.x + s4.y;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(C::kBarPFull + qt));
    }
    }
  }

  // ---- join ------------------------------------------------------------------------
  if (!ok) {
    *const_cast<volatile int*>(abortp) = 1;
    atomicExch(&a.status[b], kErrTimeout);
  }
  __syncthreads();
  const bool failed = *abortp != 0;
  if (failed) {
    // Drain (bounded) what this CTA may still have in flight before its shared memory
    // and TMEM are reused or released: the query copies, the last copy into each stage,
    // and all MMAs.
    if (warp == C::kProdWarp && lane == 0) {
      mbar_wait(BAR(C::kBarQFull), 0, 100000000ull);
      const int nk = n_issued_k >= 0 ? n_issued_k : n_issued;
      for (int j = nk - NS; j < nk; ++j)
        if (j >= 0) mbar_wait(BAR(C::kBarFullK + j % NS), (j / NS) & 1, 100000000ull);
      for (int j = n_issued - NS; j < n_issued; ++j)
        if (j >= 0) mbar_wait(BAR(C::kBarFullV + j % NS), (j / NS) & 1, 100000000ull);
    }
    if (warp == C::kMmaWarp && lane == 0) {
      umma_commit(BAR(C::kBarDrain));
      mbar_wait(BAR(C::kBarDrain), 0, 100000000ull);
    }
    __syncthreads();
  }

  // ---- merge the splits of this unit inside the cluster --------------------------
  // Every CTA leaves its row partials (O, m, l) in its own shared memory (the Q and
  // stage buffers are free now: all copies and MMAs have completed), the cluster
  // synchronises, and CTA `s` merges rows s, s + n_split, ... by reading all splits'
  // partials through distributed shared memory.  A second cluster barrier keeps every
  // CTA's partials alive until all readers are done.  Every CTA reaches both barriers
  // on every path.
  float4* po = reinterpret_cast<float4*>(sm);                  // [rows][32] float4, swizzled
  float2* pml = reinterpret_cast<float2*>(sm + C::kRows * kDH * 4);   // [rows] (m, l)
  if (live) {
    const uint32_t lane_base = ((uint32_t)((warp & 3) * 32) << 16) + 256u * qt;
    if (!failed && n_tiles > 0) {
      tc_fence_after();
#pragma unroll
      for (int q4 = 0; q4 < kDH / 32; ++q4) {
        float ov[32];
        tmem_ld32(tmem + lane_base + kTmemO + 32 * q4, ov);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          po[tid * 32 + ((q4 * 8 + i) ^ (tid & 31))] =
              make_float4(ov[4 * i], ov[4 * i + 1], ov[4 * i + 2], ov[4 * i + 3]);
      }
      pml[tid] = make_float2(m_run, l_run);
    } else {
#pragma unroll 4
      for (int k = 0; k < 32; ++k) po[tid * 32 + k] = make_float4(0.f, 0.f, 0.f, 0.f);
      pml[tid] = make_float2(-INFINITY, 0.f);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::kTmemCols) : "memory");
  }
  cluster_sync_all();

  const uint32_t po_base = smem_u32(po), pml_base = smem_u32(pml);
  constexpr int kWarps = C::kThreads / 32;
  constexpr int kPair = 2;                   // rows per warp per pass: their loads overlap
  const int stride = kWarps * ns;
  for (int r0 = s + warp * ns; r0 < rows_valid; r0 += kPair * stride) {
    // (m, l) of split `lane` and this lane's float4 of every split's O, for both rows,
    // all requested before any is used: one round trip through distributed shared memory.
    float2 ml[kPair];
    float4 v[kPair][kMaxClusterSplits];
#pragma unroll
    for (int h = 0; h < kPair; ++h) {
      const int r = r0 + h * stride;
      const bool in = r < rows_valid;
      const uint32_t off = po_base + (uint32_t)(r * 32 + (lane ^ (r & 31))) * 16;
      ml[h] = (in && lane < ns) ? ld_dsmem_f2(dsmem_addr(pml_base + r * 8, lane)) : make_float2(-INFINITY, 0.f);
#pragma unroll
      for (int s2 = 0; s2 < kMaxClusterSplits; ++s2)
        v[h][s2] = (in && s2 < ns) ? ld_dsmem_f4(dsmem_addr(off, s2)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int h = 0; h < kPair; ++h) {
      const int r = r0 + h * stride;
      if (r >= rows_valid) break;                   // warp-uniform
      float Mx = ml[h].x;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) Mx = fmaxf(Mx, __shfl_xor_sync(0xffffffffu, Mx, o));
      const float w_l = (ml[h].x == -INFINITY) ? 0.f : fast_exp2(ml[h].x - Mx);
      float l = w_l * ml[h].y;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int s2 = 0; s2 < kMaxClusterSplits; ++s2) {
        const float w = __shfl_sync(0xffffffffu, w_l, s2);
        acc.x = fmaf(v[h][s2].x, w, acc.x);
        acc.y = fmaf(v[h][s2].y, w, acc.y);
        acc.z = fmaf(v[h][s2].z, w, acc.z);
        acc.w = fmaf(v[h][s2].w, w, acc.w);
      }
      const float il = 1.f / l;
      const int Rr = row0 + r;
      const int ur = Rr / g, hr = kvh * g + Rr % g;
      if (!failed) {
        const float4 o = make_float4(acc.x * il, acc.y * il, acc.z * il, acc.w * il);
        reinterpret_cast<float4*>(a.out + (((int64_t)b * NSTR + ur) * a.Hq + hr) * kDH)[lane] = o;
        if (a.lse && lane == 0) a.lse[((int64_t)b * NSTR + ur) * a.Hq + hr] = (Mx + log2f(l)) * kLn2;
        // An fp16 operand that overflowed (|x| > 65504 in K, V or a scaled rotated query)
        // becomes inf, and a score of +inf, a value of inf or a query of inf turns the
        // row's softmax into NaN: an output that is not finite reports MEDUSA_ERANGE.
        const bool fin = isfinite(o.x) && isfinite(o.y) && isfinite(o.z) && isfinite(o.w);
        if (__any_sync(0xffffffffu, !fin) && lane == 0) atomicExch(&a.status[b], MEDUSA_ERANGE);
      }
    }
  }
  cluster_sync_all();
}

// ---- host side --------------------------------------------------------------------

bool encode_kv_map(CUtensorMap* map, void* base, const medusa_kv_t& c, int B) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[4], strides[3];
  cuuint32_t box[4], estr[4] = {1, 1, 1, 1};
  const cuuint64_t row = (cuuint64_t)c.head_dim * 2;
  if (c.page_size == 0) {
    dims[0] = c.head_dim; dims[1] = c.capacity; dims[2] = c.n_kv_heads; dims[3] = B;
    strides[0] = row; strides[1] = row * c.capacity; strides[2] = row * c.capacity * c.n_kv_heads;
    box[0] = 64; box[1] = kTcKeys; box[2] = 1; box[3] = 1;
  } else {
    dims[0] = c.head_dim; dims[1] = c.page_size; dims[2] = c.n_kv_heads; dims[3] = c.n_pages;
    strides[0] = row; strides[1] = row * c.page_size; strides[2] = row * c.page_size * c.n_kv_heads;
    box[0] = 64; box[1] = c.page_size; box[2] = 1; box[3] = 1;
  }
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Rows [B][N][H][dh] (queries, or the tree rows k_new / v_new) as a 4-D tensor
// (dh, H, N, B); a box is 64 dims of `box_h` consecutive heads of `box_n`
// consecutive tree rows.
bool encode_rows_map(CUtensorMap* map, const void* base, int B, int N, int H, int box_h, int box_n) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t row = (cuuint64_t)kDH * 2;
  cuuint64_t dims[4] = {(cuuint64_t)kDH, (cuuint64_t)H, (cuuint64_t)N, (cuuint64_t)B};
  cuuint64_t strides[3] = {row, row * H, row * H * N};
  cuuint32_t box[4] = {64, (cuuint32_t)box_h, (cuuint32_t)box_n, 1}, estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int QT, int NS>
size_t tc_smem_bytes(int D) {
  using C = TcCfg<QT, NS>;
  return 1024 + C::kOffTable + (size_t)2 * (D + 1) * kHalf * sizeof(float) + 8 + C::kNumBars * 8;
}

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool attn_tc_supported(const medusa_tree_t& t, int Hq, const medusa_kv_t& c) {
  (void)t;
  // a query tile is one TMA box of whole GQA groups
  const int g = c.n_kv_heads > 0 ? Hq / c.n_kv_heads : 0;
  return c.dtype == MEDUSA_BF16 && c.head_dim == kDH && (c.page_size == 0 || c.page_size == 16) && g > 0 &&
         kTcRows % g == 0 && encode_fn() != nullptr;
}

namespace {

// Co-resident clusters of n CTAs of one kernel shape, from the occupancy calculator
// (thread-block clusters live inside one GPC, so n CTAs that need a whole SM each fit
// floor(SMs of the GPC / n) times per GPC); cached per shape and n.
template <int QT, int NS>
int max_clusters(int n, int D) {
  static std::mutex mu;
  static int cache[kMaxClusterSplits + 1] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (cache[n] != 0) return cache[n];
  const size_t smem = tc_smem_bytes<QT, NS>(D);
  auto kern = attn_tc_kernel<false, QT, NS>;
  int c = 0;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, n, 1);
    cfg.blockDim = dim3(TcCfg<QT, NS>::kThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = n;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&c, kern, &cfg) != cudaSuccess) c = 0;
  }
  cudaGetLastError();                 // a failed query leaves no sticky error behind
  cache[n] = c > 0 ? c : -1;
  return cache[n];
}

int clusters_for(int qt, int stages, int n, int D) {
  if (qt == 2) return max_clusters<2, 2>(n, D);
  if (stages == 4) return max_clusters<1, 4>(n, D);
  return max_clusters<1, 2>(n, D);
}

}  // namespace

// Kernel shape and split choice.  With two or more row tiles per unit, one CTA takes
// two of them (QT = 2, 128-key tiles, two stages: 192 KB of shared memory, one CTA
// per SM), so that every K/V tile is copied and converted once for 256 rows and the
// two tiles keep the tensor cores busy in turn.  A single row tile runs two CTAs per
// SM (QT = 1, 64-key tiles, two stages), which overlaps one CTA's prologue and merge
// with the other's main loop.
// The number of splits n (one cluster of n CTAs per unit, n <= kMaxClusterSplits,
// at least rows/16 keys' worth of tiles per split) minimises a time model measured on
// GB300: a CTA costs F + T_t per tile (F: prologue, merge and launch; T_t: one tile;
// QT = 1: 10 + 1.8 us per 64 keys, QT = 2: 15 + 2.2 us per 128 keys), and only
// `clusters(n)` clusters run at once (occupancy calculator for one CTA per SM; with
// two CTAs per SM, 2 x SMs / n).  One sequence: whole
// waves of identical clusters.  Several sequences of unknown lengths (at most the
// maximum prefix; taken as half of it on average): the longest split or the total
// work over the cluster slots, whichever is larger.  The tree tiles count as work of
// split 0, which takes that many fewer prefix tiles, so that the splits end together.
// MEDUSA_ATTN_TC_SHAPE="QT,NS" (one of 1,2 / 1,4 / 2,2) overrides the shape and
// MEDUSA_ATTN_TC_SPLITS=n the number of splits (at most the plan's maximum).
void attn_tc_plan(AttnPlan& p) {
  const int M = p.N * p.g;
  const int n_tiles_q = (M + kTcRows - 1) / kTcRows;
  int qt = n_tiles_q >= 2 ? 2 : 1, stages = 2;
  if (const char* e = std::getenv("MEDUSA_ATTN_TC_SHAPE")) {
    int a = 0, b = 0;
    if (std::sscanf(e, "%d,%d", &a, &b) == 2 && ((a == 1 && (b == 2 || b == 4)) || (a == 2 && b == 2))) {
      qt = a;
      stages = b;
    }
  }
  p.qt = qt;
  p.stages = stages;
  p.mt_rows = kTcRows * qt;
  const int KT = 64 * qt;
  p.key_tile = KT;
  p.n_mt = (M + p.mt_rows - 1) / p.mt_rows;
  const int units = p.B * p.Hkv * p.n_mt;
  int sms = 148, dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int per_sm = (qt == 1 && stages == 2) ? 2 : 1;
  const int tiles_unit = (p.max_prefix + KT - 1) / KT;
  const int n_tree = (p.N + KT - 1) / KT;
  const int rows = M < kTcRows ? M : kTcRows;
  int min_tiles = ((rows + 15) / 16 + qt - 1) / qt;
  if (min_tiles < 2) min_tiles = 2;
  int max_split = tiles_unit / min_tiles;
  if (max_split > kMaxClusterSplits) max_split = kMaxClusterSplits;
  if (max_split < 1) max_split = 1;
  const double F = qt == 2 ? 15.0 : 10.0, Tt = qt == 2 ? 2.2 : 1.8;
  const int tiles = tiles_unit + n_tree;
  int best = 1;
  double best_t = 1e300;
  for (int n = 1; n <= max_split; ++n) {
    // Clusters of CTAs that need a whole SM are limited by the GPCs (occupancy
    // calculator); with two CTAs per SM the clusters fill the SMs' second slots too,
    // which the calculator does not count (measured: 32 clusters of 8 co-resident).
    int cl = per_sm > 1 ? per_sm * sms / n : clusters_for(qt, stages, n, p.D);
    if (cl < 1) cl = per_sm * sms / n;           // occupancy query unavailable: an estimate
    if (cl < 1) cl = 1;
    const double per_max = F + Tt * ((tiles + n - 1) / n);
    double t;
    if (p.B == 1) {
      t = std::ceil(units / (double)cl) * per_max;
    } else {
      const double per_avg = F + Tt * std::ceil(0.5 * tiles / n);
      t = std::max(per_max, units * per_avg / cl);
    }
    if (t <= best_t * (1.0 + 1e-9)) { best_t = t; best = n; }   // ties: more, smaller splits
  }
  if (const char* e = std::getenv("MEDUSA_ATTN_TC_SPLITS")) {   // tuning override
    const int n = std::atoi(e);
    if (n >= 1 && n <= max_split) best = n;
  }
  const int per = (tiles_unit + n_tree + best - 1) / best;
  int first_tiles = per - n_tree;
  if (first_tiles < 0) first_tiles = 0;
  if (first_tiles > tiles_unit || best == 1) first_tiles = tiles_unit;
  const int rest = tiles_unit - first_tiles;
  int chunk_tiles = best > 1 ? (rest + best - 2) / (best - 1) : 1;
  if (chunk_tiles < 1) chunk_tiles = 1;
  p.first = first_tiles * KT;
  p.chunk = chunk_tiles * KT;
  p.n_split = 1 + (rest + chunk_tiles - 1) / chunk_tiles;
}

namespace {

template <bool PAGED, int QT, int NS>
cudaError_t launch_shape(cudaLaunchConfig_t& cfg, int D, const CUtensorMap& mk, const CUtensorMap& mv,
                         const CUtensorMap& mkn, const CUtensorMap& mvn, const CUtensorMap& mq, const TcArgs& a) {
  const size_t smem = tc_smem_bytes<QT, NS>(D);
  cfg.blockDim = dim3(TcCfg<QT, NS>::kThreads);
  cfg.dynamicSmemBytes = smem;
  cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<PAGED, QT, NS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  return cudaLaunchKernelEx(&cfg, attn_tc_kernel<PAGED, QT, NS>, mk, mv, mkn, mvn, mq, a);
}

template <bool PAGED>
cudaError_t launch_paged(const AttnPlan& p, cudaLaunchConfig_t& cfg, const CUtensorMap& mk, const CUtensorMap& mv,
                         const CUtensorMap& mkn, const CUtensorMap& mvn, const CUtensorMap& mq, const TcArgs& a) {
  if (p.qt == 2) return launch_shape<PAGED, 2, 2>(cfg, p.D, mk, mv, mkn, mvn, mq, a);
  if (p.stages == 4) return launch_shape<PAGED, 1, 4>(cfg, p.D, mk, mv, mkn, mvn, mq, a);
  return launch_shape<PAGED, 1, 2>(cfg, p.D, mk, mv, mkn, mvn, mq, a);
}

}  // namespace

cudaError_t launch_attn_tc(const AttnPlan& p, const medusa_tree_t& t, const void* q,
                           const void* k_new, const void* v_new, const medusa_kv_t& c,
                           const int32_t* L, const float* th_hi, const float* th_lo,
                           float scale_log2, float* out, float* lse, int32_t* status, void* ws,
                           cudaStream_t st) {
  CUtensorMap mk, mv, mkn, mvn, mq;
  // prefix tiles come from the fp16 mirror when the cache has one (the same layout)
  if (!encode_kv_map(&mk, c.k_f16 ? c.k_f16 : c.k, c, p.B) || !encode_kv_map(&mv, c.v_f16 ? c.v_f16 : c.v, c, p.B) ||
      !encode_rows_map(&mkn, k_new, p.B, t.n_rows, p.Hkv, 1, kTcKeys) ||
      !encode_rows_map(&mvn, v_new, p.B, t.n_rows, p.Hkv, 1, kTcKeys) ||
      !encode_rows_map(&mq, q, p.B, t.n_rows, p.Hq, p.g, kTcRows / p.g))
    return cudaErrorInvalidValue;
  TcArgs a{};
  a.t = t;
  a.c = c;
  a.q = (const uint16_t*)q;
  a.k_new = (const uint16_t*)k_new;
  a.v_new = (const uint16_t*)v_new;
  a.L = L;
  a.out = out;
  a.lse = lse;
  a.status = status;
  (void)ws;                                        // the cluster merge needs no workspace
  a.B = p.B;
  a.Hq = p.Hq;
  a.Hkv = p.Hkv;
  a.g = p.g;
  a.n_mt = p.n_mt;
  a.n_split = p.n_split;
  a.chunk = p.chunk;
  a.first = p.first;
  a.scale_log2 = scale_log2;
  a.stall_ns = test_stall_ns();
  for (int i = 0; i < 64; ++i) {
    a.th_hi[i] = th_hi[i];
    a.th_lo[i] = th_lo[i];
  }
  // every CTA of a sequence may record an error; none records success
  cudaError_t ce = cudaMemsetAsync(status, 0, sizeof(int32_t) * (size_t)p.B, st);
  if (ce != cudaSuccess) return ce;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.n_mt, p.n_split, p.B * p.Hkv);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = p.n_split;           // the splits of one unit
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = c.page_size == 0 ? launch_paged<false>(p, cfg, mk, mv, mkn, mvn, mq, a)
                                         : launch_paged<true>(p, cfg, mk, mv, mkn, mvn, mq, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace medusa
