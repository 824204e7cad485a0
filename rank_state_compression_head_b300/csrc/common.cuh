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

// 16-byte global load that bypasses L1 allocation (streamed factor data)
__device__ static inline uint4 ld_stream16(const void *p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

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

}  // namespace seedk

// Launchers implemented in the kernel files, called by the C-ABI layer.
namespace seedk {
cudaError_t launch_decode(const StateView &sv, int factor_dtype, const float *q, const float *k,
                          const float *v, const float *gate, const float *beta, const float *A,
                          float *o, int cols_max, cudaStream_t s);
cudaError_t launch_recompress(const StateView &sv, int factor_dtype, float *trunc_err,
                              int32_t *sweeps, int m_max, cudaStream_t s);
cudaError_t launch_compress_dense(const StateView &sv, int factor_dtype, const float *S,
                                  float *trunc_err, cudaStream_t s);
cudaError_t launch_materialize(const StateView &sv, int factor_dtype, float *S_out, int m_max,
                               cudaStream_t s);
cudaError_t launch_dense_decode(int variant, int n_heads, int d_v, float *S, const float *q,
                                const float *k, const float *v, const float *gate,
                                const float *beta, const float *A, const int32_t *dir_index,
                                float *o, cudaStream_t s);
}  // namespace seedk
