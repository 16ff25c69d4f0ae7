// Shared device helpers for the Medusa verify-round kernels (sm_103a).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "medusa_gb300.h"

namespace medusa {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// bf16 <-> fp32 without cuda_bf16.h intrinsics: bf16 is the top half of an fp32.
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

// Round-to-nearest-even fp32 -> bf16 bits (finite inputs).
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
  uint32_t u = __float_as_uint(f);
  uint32_t rounding = 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)((u + rounding) >> 16);
}

// fp16 bits of a bf16 value (exact for magnitudes in [2^-14, 65504]): the value of a
// bf16 cache's fp16 mirror.
__device__ __forceinline__ uint16_t bf16_bits_to_f16_bits(uint16_t b) {
  const __half h = __float2half_rn(__uint_as_float((uint32_t)b << 16));
  return *reinterpret_cast<const uint16_t*>(&h);
}

// Element traits: float storage or bf16 storage (raw uint16_t bits).
template <typename EL> struct Elem;
template <> struct Elem<float> {
  static constexpr int kPerVec = 4;  // elements per 16-byte vector
  __device__ __forceinline__ static float load(const float* p, int64_t i) { return p[i]; }
  __device__ __forceinline__ static void store(float* p, int64_t i, float v) { p[i] = v; }
  __device__ __forceinline__ static void unpack(const uint4& v, float* f) {
    f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
  }
};
template <> struct Elem<uint16_t> {
  static constexpr int kPerVec = 8;
  __device__ __forceinline__ static float load(const uint16_t* p, int64_t i) {
    return bf16_bits_to_f32(p[i]);
  }
  __device__ __forceinline__ static void store(uint16_t* p, int64_t i, float v) {
    p[i] = f32_to_bf16_bits(v);
  }
  __device__ __forceinline__ static void unpack(const uint4& v, float* f) {
    f[0] = __uint_as_float(v.x << 16); f[1] = __uint_as_float(v.x & 0xFFFF0000u);
    f[2] = __uint_as_float(v.y << 16); f[3] = __uint_as_float(v.y & 0xFFFF0000u);
    f[4] = __uint_as_float(v.z << 16); f[5] = __uint_as_float(v.z & 0xFFFF0000u);
    f[6] = __uint_as_float(v.w << 16); f[7] = __uint_as_float(v.w & 0xFFFF0000u);
  }
};

// 128-bit streaming load that bypasses L1 allocation (weights are read once).
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Ranking order used for argmax and top-k: larger value first, ties to the lower id.
__device__ __forceinline__ bool ranks_before(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// Accurate RoPE angle: pos * theta reduced to [-pi, pi] in fp32 with the frequency
// carried as a hi/lo pair and 2*pi split Cody-Waite style, so that positions of
// 10^5 and beyond keep ~1e-7 rad of accuracy.  pos is an exact integer.
__device__ __forceinline__ float rope_angle(int pos, float theta_hi, float theta_lo) {
  const float kTwoPiHi = 6.28318548202514648f;       // fp32(2*pi)
  const float kTwoPiLo = -1.7484555314695172e-07f;   // 2*pi - kTwoPiHi
  const float kInvTwoPi = 0.15915494309189535f;
  float p = (float)pos;                                // exact for |pos| < 2^24
  float x_hi = p * theta_hi;
  float x_err = fmaf(p, theta_hi, -x_hi);              // exact rounding error of x_hi
  float x_lo = fmaf(p, theta_lo, x_err);
  float k = rintf(x_hi * kInvTwoPi);
  float r = fmaf(-k, kTwoPiHi, x_hi);                  // exact when |r| is small
  r = r + fmaf(-k, kTwoPiLo, x_lo);
  return r;
}

// The template of sequence b: its own when t is a per-sequence batch (t.per_seq set;
// t's counts are then bounds over the batch and the row stride of per-row tensors),
// else t itself.
__device__ __forceinline__ medusa_tree_t seq_tree(const medusa_tree_t& t, int b) {
  if (t.per_seq == nullptr) return t;
  return t.per_seq[b];
}

// Rows [0, rows_end) of sequence b exist in the cache.  Contiguous caches check the
// capacity; paged caches also need a valid page for the last row (a sequence owns
// a prefix of its block-table row; unused entries are negative).
__device__ __forceinline__ bool seq_rows_ok(const medusa_kv_t& c, int b, int64_t rows_end) {
  if (rows_end > c.capacity) return false;
  if (c.page_size == 0 || rows_end <= 0) return true;
  const int64_t blk = (rows_end - 1) / c.page_size;
  if (blk >= c.max_blocks) return false;
  const int page = c.block_table[(int64_t)b * c.max_blocks + blk];
  return page >= 0 && page < c.n_pages;
}

// Element offset of (sequence b, kv head, row) in a contiguous or paged cache.
__device__ __forceinline__ int64_t cache_row_offset(const medusa_kv_t& c, int b, int kvh, int row) {
  if (c.page_size == 0)
    return (((int64_t)b * c.n_kv_heads + kvh) * c.capacity + row) * c.head_dim;
  const int page = c.block_table[(int64_t)b * c.max_blocks + row / c.page_size];
  return (((int64_t)page * c.n_kv_heads + kvh) * c.page_size + row % c.page_size) * c.head_dim;
}

// ---- mbarrier helpers (shared by the TMA-fed kernels) ----------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase with the given parity to complete; gives up after ~`limit_ns`.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns = 2000000000ull) {
  const uint64_t t0 = global_ns();
  for (uint32_t it = 0;; ++it) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return true;
    if ((it & 1023u) == 1023u && global_ns() - t0 > limit_ns) return false;
  }
}

// One non-blocking probe of the phase with the given parity.
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Non-blocking test of the phase with the given parity (never suspends the thread,
// unlike try_wait): for loops that poll several barriers.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// 1-D bulk copy global -> shared, completion counted on an mbarrier (16-byte aligned
// addresses, size a multiple of 16 bytes).
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

}  // namespace medusa
