// Internal helpers shared by the kernels of libseed.so (not part of the C-ABI).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
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

  __device__ inline int rank_of(int h) const { return rank ? rank[h] : r; }
  __device__ inline int64_t col0(int h) const {
    return col_offset ? col_offset[h] : (int64_t)h * cap_uniform;
  }
  __device__ inline int dir_of(int h) const { return vbar_index ? vbar_index[h] : h; }
};

struct DecodeArgs {
  StateView sv;
  const float *q, *k, *v, *gate, *beta, *A;
  float *o;
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
int sm_count();
cudaError_t launch_decode_mma(const DecodeArgs &a, int cols_max, cudaStream_t s);
cudaError_t launch_recompress(const StateView &sv, int factor_dtype, float *trunc_err,
                              int32_t *sweeps, int m_max, cudaStream_t s);
cudaError_t launch_recompress_split(const StateView &sv, int factor_dtype, float *trunc_err,
                                    int32_t *sweeps, int m_max, int r_max, float *ws,
                                    int64_t chunk, cudaStream_t s);
int64_t split_floats_per_head(int m_max, int r_max, int d_v);
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
