// Internal helpers shared by the kernels of libseed.so (not part of the C-ABI).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "seed.h"

namespace seedk {

constexpr int kDK = 128;         // key / state-size dimension supported by the kernels
constexpr int kMaxCols = SEED_MAX_COLUMNS;

// ---------------------------------------------------------------------------
// factor element types: 16-byte chunks, conversions
// ---------------------------------------------------------------------------

template <typename TF> struct Elem;

template <> struct Elem<float> {
  static constexpr int kPer16B = 4;
  __device__ static inline void unpack(const uint4 &c, float (&x)[4]) {
    x[0] = __uint_as_float(c.x); x[1] = __uint_as_float(c.y);
    x[2] = __uint_as_float(c.z); x[3] = __uint_as_float(c.w);
  }
  __device__ static inline float round(float x) { return x; }
  __device__ static inline void store(float *p, float x) { *p = x; }
  __device__ static inline float load(const float *p) { return *p; }
};

template <> struct Elem<__nv_bfloat16> {
  static constexpr int kPer16B = 8;
  __device__ static inline void unpack(const uint4 &c, float (&x)[8]) {
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  // value the element holds after a round-to-nearest-even store
  __device__ static inline float round(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }
  __device__ static inline void store(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }
  __device__ static inline float load(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
};

template <> struct Elem<__half> {
  static constexpr int kPer16B = 8;
  __device__ static inline void unpack(const uint4 &c, float (&x)[8]) {
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[i]));
      x[2 * i] = f.x;
      x[2 * i + 1] = f.y;
    }
  }
  __device__ static inline float round(float x) { return __half2float(__float2half_rn(x)); }
  __device__ static inline void store(__half *p, float x) { *p = __float2half_rn(x); }
  __device__ static inline float load(const __half *p) { return __half2float(*p); }
};

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy
// as 1, 2, 3", SC'11): the random bits of stochastic rounding and of the
// synthetic workloads
// ---------------------------------------------------------------------------
constexpr uint32_t kPhiloxM0 = 0xD2511F53u, kPhiloxM1 = 0xCD9E8D57u;
constexpr uint32_t kPhiloxW0 = 0x9E3779B9u, kPhiloxW1 = 0xBB67AE85u;

__device__ __forceinline__ uint4 philox(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                        uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) { k0 += kPhiloxW0; k1 += kPhiloxW1; }
    const uint32_t hi0 = __umulhi(kPhiloxM0, c0), lo0 = kPhiloxM0 * c0;
    const uint32_t hi1 = __umulhi(kPhiloxM1, c2), lo1 = kPhiloxM1 * c2;
    const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
  }
  return make_uint4(c0, c1, c2, c3);
}

// ---------------------------------------------------------------------------
// Storage rounding of factor elements: round to nearest even, or stochastic
// (up with probability equal to the fraction of the gap below x, so the stored
// value is x on average).  Stochastic bits come from Philox keyed by the
// caller's sr_seed, with the counter (pool column, element, purpose), so a run
// is reproducible for a given seed.
// ---------------------------------------------------------------------------
enum { kRoundNearest = 0, kRoundStochastic = 1 };
enum { kSrAppend = 0, kSrRebuildU = 1, kSrRebuildW = 2 };  // purpose word of the counter

__device__ __forceinline__ uint4 sr_bits(uint64_t seed, int64_t col, uint32_t elem, uint32_t purpose) {
  return philox((uint32_t)col, (uint32_t)((uint64_t)col >> 32), elem, purpose, (uint32_t)seed,
                (uint32_t)(seed >> 32));
}

template <typename TF> struct SrRound;
template <> struct SrRound<float> {
  __device__ static inline float apply(float x, uint32_t) { return x; }
};
template <> struct SrRound<__nv_bfloat16> {
  // bf16 keeps the top 16 bits of the fp32 pattern: add 16 random low bits, truncate
  __device__ static inline float apply(float x, uint32_t bits) {
    if (!isfinite(x)) return Elem<__nv_bfloat16>::round(x);
    const uint32_t u = __float_as_uint(x) + (bits & 0xffffu);
    return __uint_as_float(u & 0xffff0000u);
  }
};
template <> struct SrRound<__half> {
  // fp16: in its normal range drop the 13 low mantissa bits after adding 13 random
  // ones (truncation toward zero); in its subnormal range (|x| < 2^-14) choose
  // between the two neighbouring multiples of 2^-24 exactly
  __device__ static inline float apply(float x, uint32_t bits) {
    if (!isfinite(x)) return Elem<__half>::round(x);
    const float a = fabsf(x);
    if (a < 6.103515625e-05f) {
      const float q = a * 16777216.f;  // a / 2^-24, exact
      const float fl = floorf(q);
      const float up = (float)(bits >> 8) * 5.9604644775390625e-08f < q - fl ? 1.f : 0.f;  // 24 bits
      return copysignf((fl + up) * 5.9604644775390625e-08f, x);
    }
    const uint32_t u = __float_as_uint(x) + (bits & 0x1fffu);
    return __half2float(__float2half_rz(__uint_as_float(u)));
  }
};

// The value a factor element takes when stored: nearest, or stochastic with bits.
template <typename TF>
__device__ __forceinline__ float store_value(float x, int rounding, uint32_t bits) {
  return rounding == kRoundStochastic ? SrRound<TF>::apply(x, bits) : Elem<TF>::round(x);
}


// ---------------------------------------------------------------------------
// 16-bit tensor-core operands: mma.sync m16n8k16 with fp32 accumulation takes
// both operands in the same 16-bit type (bf16 or fp16)
// ---------------------------------------------------------------------------
template <typename TF> struct Mma16;
template <> struct Mma16<__nv_bfloat16> {
  __device__ static inline void mma(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                    uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
  __device__ static inline uint32_t pack(float x, float y) {
    __nv_bfloat162 v = __floats2bfloat162_rn(x, y);
    return *reinterpret_cast<uint32_t *>(&v);
  }
  __device__ static inline float2 unpack(uint32_t u) {
    return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
  }
  __device__ static inline __nv_bfloat16 cvt(float x) { return __float2bfloat16_rn(x); }
  __device__ static inline float back(__nv_bfloat16 x) { return __bfloat162float(x); }
};
template <> struct Mma16<__half> {
  __device__ static inline void mma(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                    uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
  __device__ static inline uint32_t pack(float x, float y) {
    __half2 v = __floats2half2_rn(x, y);
    return *reinterpret_cast<uint32_t *>(&v);
  }
  __device__ static inline float2 unpack(uint32_t u) { return __half22float2(*reinterpret_cast<__half2 *>(&u)); }
  __device__ static inline __half cvt(float x) { return __float2half_rn(x); }
  __device__ static inline float back(__half x) { return __half2float(x); }
};

__device__ static inline float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__device__ static inline float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ static inline bool finite(float x) { return isfinite(x); }

// Named barrier over `nthreads` threads (a multiple of 32) with id 1..15.
__device__ static inline void team_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------------------
// mbarrier + bulk-copy (TMA engine, non-tensor) primitives
// ---------------------------------------------------------------------------

__device__ static inline uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ static inline void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ static inline void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ static inline void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ static inline void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ static inline bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: false if the phase did not complete within the spin limit.
constexpr uint32_t kSpinLimit = 1u << 26;
__device__ static inline bool mbar_wait(uint64_t *bar, uint32_t parity) {
  for (uint32_t it = 0; it < kSpinLimit; ++it)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
// global -> shared bulk copy (size and both addresses multiples of 16 bytes),
// completion counted on `bar` as transaction bytes
__device__ static inline void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// OR of a predicate over the `nthreads` threads of named barrier `id` (also a barrier)
__device__ static inline int team_or(int id, int nthreads, int pred) {
  int r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.s32 p, %1, 0;\n bar.red.or.pred q, %2, %3, p;\n"
      " selp.s32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"(pred), "r"(id), "r"(nthreads)
      : "memory");
  return r;
}

// ---------------------------------------------------------------------------
// per-head geometry shared by the factored kernels
// ---------------------------------------------------------------------------

struct StateView {
  int32_t variant, n_heads, d_k, d_v, T, r, steps;
  int32_t rounding;               // kRoundNearest or kRoundStochastic (16-bit factors)
  uint64_t sr_seed;               // key of the stochastic-rounding bits
  int32_t growth;                 // columns per step
  int32_t cap_uniform;            // r + growth*T when col_offset == NULL
  const int32_t *rank;
  const int64_t *col_offset;
  float *a;
  void *U;
  void *W;
  float *scale;
  const float *vbar;
  const int32_t *vbar_index;
  int32_t *status;
  const int32_t *order;           // heads grouped by column class, or NULL
  int32_t class_end[4];           // with order: where each class ends in it

  __device__ inline int rank_of(int h) const { return rank ? rank[h] : r; }
  __device__ inline int64_t col0(int h) const {
    return col_offset ? col_offset[h] : (int64_t)h * cap_uniform;
  }
  __device__ inline int dir_of(int h) const { return vbar_index ? vbar_index[h] : h; }
};

// Value stored for element `elem` of pool column `col` of U (purpose kSrRebuildU)
// or W (kSrRebuildW) under the state's rounding.  One Philox block serves four
// consecutive elements (word elem % 4); each thread computes its own.
template <typename TF>
__device__ inline float stored_elem(const StateView &sv, float x, int64_t col, int elem, uint32_t purpose) {
  if (sv.rounding != kRoundStochastic) return Elem<TF>::round(x);
  const uint4 b = sr_bits(sv.sr_seed, col, (uint32_t)(elem >> 2), purpose);
  const int q = elem & 3;
  return SrRound<TF>::apply(x, q == 0 ? b.x : q == 1 ? b.y : q == 2 ? b.z : b.w);
}

struct DecodeArgs {
  StateView sv;
  const float *q, *k, *v, *gate, *beta, *A;
  float *o;
  // heads of this launch: sv.order[pos0 .. pos0 + count) when sv.order is set (one
  // column class), else all n_heads heads in index order
  int32_t pos0, count;
};

// Sum of eight per-lane values over the warp: after 9 shuffles lane l holds
// the total of value ((l >> 4) & 1) * 4 + ((l >> 3) & 1) * 2 + ((l >> 2) & 1).
__device__ inline float warp_reduce8(const float (&v)[8], int lane) {
  float a4[4], a2[2];
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float keep = b4 ? v[i + 4] : v[i], send = b4 ? v[i] : v[i + 4];
    a4[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float keep = b3 ? a4[i + 2] : a4[i], send = b3 ? a4[i] : a4[i + 2];
    a2[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
  const float keep = b2 ? a2[1] : a2[0], send = b2 ? a2[0] : a2[1];
  float a = keep + __shfl_xor_sync(0xffffffffu, send, 4);
  a += __shfl_xor_sync(0xffffffffu, a, 2);
  a += __shfl_xor_sync(0xffffffffu, a, 1);
  return a;
}
__device__ inline int reduce8_index(int lane) {
  return ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
}

// Column scales can travel with the bulk copy when their block is 16-byte aligned.
__device__ inline bool scales_in_stage(int64_t c0, int cap) { return ((c0 | cap) & 3) == 0; }

}  // namespace seedk

// Launchers implemented in the kernel files, called by the C-ABI layer.
namespace seedk {
cudaError_t launch_decode(const StateView &sv, int factor_dtype, const float *q, const float *k,
                          const float *v, const float *gate, const float *beta, const float *A,
                          float *o, int cols_max, cudaStream_t s);
cudaError_t launch_decode_mma(const DecodeArgs &a, int factor_dtype, int cols_max, cudaStream_t s);
cudaError_t launch_recompress(const StateView &sv, int factor_dtype, float *trunc_err,
                              int32_t *sweeps, int m_max, cudaStream_t s);
cudaError_t launch_recompress_split(const StateView &sv, int factor_dtype, float *trunc_err,
                                    int32_t *sweeps, int m_max, int r_max, float *ws,
                                    int64_t chunk, cudaStream_t s);
// Workspace floats per head of seed_recompress_ws: the QR route (32-bit factors) or the
// Gram route (16-bit factors).
int64_t split_floats_per_head(int factor_dtype, int m_max, int r_max, int d_v);
int64_t gram_floats_per_head(int m_max, int r_max);
cudaError_t launch_recompress_gram(const StateView &sv, int factor_dtype, float *trunc_err, int32_t *sweeps,
                                   int m_max, int r_max, float *ws, int64_t chunk, cudaStream_t s);
// Fixed device scratch of seed_recompress_noalloc: 64 MiB.
constexpr int64_t kNoAllocScratchFloats = (int64_t)16 << 20;
cudaError_t noalloc_scratch(float **ptr);
cudaError_t launch_compress_dense(const StateView &sv, int factor_dtype, const float *S,
                                  float *trunc_err, cudaStream_t s);
cudaError_t launch_materialize(const StateView &sv, int factor_dtype, float *S_out, int m_max,
                               cudaStream_t s);
cudaError_t launch_dense_decode(int variant, int n_heads, int d_v, float *S, const float *q,
                                const float *k, const float *v, const float *gate,
                                const float *beta, const float *A, const int32_t *dir_index,
                                float *o, cudaStream_t s);
}  // namespace seedk
