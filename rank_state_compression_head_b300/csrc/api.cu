// C-ABI entry points of libseed.so (declared in include/seed.h).
//
// Every call validates its arguments on the host and launches nothing when
// they are wrong; kernels run asynchronously on the caller's stream.  The
// library allocates no memory and keeps no state between calls: the state
// lives in the caller's seed_state and device buffers.  The one exception is
// the fixed device scratch of seed_recompress_noalloc (recompress_split.cu),
// a file-scope __device__ array that every device loading the library holds.
// Besides that, the decode launchers remember per device which of their kernels
// already had their shared-memory attributes set, and the 16-bit one how many
// CTAs of each kernel the device holds at once (the size of its persistent grid).
#include "common.cuh"

#include <stdint.h>

using namespace seedk;

namespace {

inline bool misaligned(const void *p) { return reinterpret_cast<uintptr_t>(p) % 16 != 0; }
inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? SEED_OK : SEED_ERR_CUDA; }
inline int growth_of(int variant) { return variant == SEED_KDA ? 2 : 1; }

// Shape, pointer and capacity checks shared by the factored-state calls.
int check_state(const seed_state *st) {
  if (!st) return SEED_ERR_INVALID_ARG;
  if (st->variant < SEED_GDN || st->variant > SEED_MAMBA2) return SEED_ERR_INVALID_ARG;
  if (st->factor_dtype != SEED_F32 && st->factor_dtype != SEED_BF16 && st->factor_dtype != SEED_F16)
    return SEED_ERR_INVALID_ARG;
  if (st->rounding != SEED_ROUND_NEAREST && st->rounding != SEED_ROUND_STOCHASTIC) return SEED_ERR_INVALID_ARG;
  if (st->n_heads < 0 || st->T < 1 || st->steps_since_compress < 0) return SEED_ERR_INVALID_ARG;
  if (st->d_k != kDK || (st->d_v != 64 && st->d_v != 128)) return SEED_ERR_UNSUPPORTED_SHAPE;
  const int rmax = st->rank ? st->r_max : st->r;
  if (st->r < 0 || rmax < 0) return SEED_ERR_INVALID_ARG;
  if (!st->rank && st->r_max != st->r && st->r_max != 0) return SEED_ERR_INVALID_ARG;
  const int dmin = st->d_k < st->d_v ? st->d_k : st->d_v;
  if (rmax > dmin) return SEED_ERR_UNSUPPORTED_SHAPE;
  if (rmax + growth_of(st->variant) * st->T > kMaxCols) return SEED_ERR_UNSUPPORTED_SHAPE;
  if (st->n_heads == 0) return SEED_OK;
  if (!st->a || !st->U || !st->W || !st->scale || !st->vbar) return SEED_ERR_INVALID_ARG;
  if (misaligned(st->a) || misaligned(st->U) || misaligned(st->W) || misaligned(st->vbar) ||
      misaligned(st->scale))
    return SEED_ERR_ALIGNMENT;
  if (st->head_order) {
    int prev = 0;
    for (int c = 0; c < 4; ++c) {
      if (st->class_end[c] < prev) return SEED_ERR_INVALID_ARG;
      prev = st->class_end[c];
    }
    if (prev != st->n_heads) return SEED_ERR_INVALID_ARG;
  }
  return SEED_OK;
}

StateView view_of(const seed_state *st) {
  StateView v;
  v.variant = st->variant;
  v.n_heads = st->n_heads;
  v.d_k = st->d_k;
  v.d_v = st->d_v;
  v.T = st->T;
  v.r = st->r;
  v.steps = st->steps_since_compress;
  v.rounding = st->factor_dtype == SEED_F32 ? SEED_ROUND_NEAREST : st->rounding;
  v.sr_seed = st->sr_seed;
  v.growth = growth_of(st->variant);
  v.cap_uniform = (st->rank ? st->r_max : st->r) + v.growth * st->T;
  v.rank = st->rank;
  v.col_offset = st->col_offset;
  v.a = st->a;
  v.U = st->U;
  v.W = st->W;
  v.scale = st->scale;
  v.vbar = st->vbar;
  v.vbar_index = st->vbar_index;
  v.status = st->status;
  // the class order serves 16-bit factors with per-head ranks
  v.order = st->head_order && st->rank && st->factor_dtype != SEED_F32 ? st->head_order : nullptr;
  for (int c = 0; c < 4; ++c) v.class_end[c] = v.order ? st->class_end[c] : 0;
  return v;
}

inline int rmax_of(const seed_state *st) { return st->rank ? st->r_max : st->r; }

}  // namespace

extern "C" int32_t seed_columns_per_head(int32_t variant, int32_t r, int32_t T) {
  return r + growth_of(variant) * T;
}

extern "C" const char *seed_status_string(int status) {
  switch (status) {
    case SEED_OK: return "ok";
    case SEED_ERR_INVALID_ARG: return "invalid argument";
    case SEED_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case SEED_ERR_CAPACITY: return "factor capacity exceeded (recompress first)";
    case SEED_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case SEED_ERR_CUDA: return "CUDA launch failed";
    case SEED_ERR_NOT_CONVERGED: return "Jacobi SVD did not converge";
    case SEED_ERR_NONFINITE: return "non-finite value";
    case SEED_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

extern "C" int seed_compress_dense(const float *S, seed_state *st, float *trunc_err,
                                   seed_stream_t stream) {
  int c = check_state(st);
  if (c) return c;
  if (st->n_heads == 0) { st->steps_since_compress = 0; return SEED_OK; }
  if (!S) return SEED_ERR_INVALID_ARG;
  if (misaligned(S)) return SEED_ERR_ALIGNMENT;
  seed_state tmp = *st;
  tmp.steps_since_compress = 0;
  c = cuda_status(launch_compress_dense(view_of(&tmp), st->factor_dtype, S, trunc_err,
                                        (cudaStream_t)stream));
  if (c == SEED_OK) st->steps_since_compress = 0;
  return c;
}

extern "C" int seed_decode_step(seed_state *st, const float *q, const float *k, const float *v,
                                const float *gate, const float *beta, const float *A, float *o,
                                seed_stream_t stream) {
  int c = check_state(st);
  if (c) return c;
  if (st->steps_since_compress >= st->T) return SEED_ERR_CAPACITY;
  if (st->n_heads == 0) { ++st->steps_since_compress; return SEED_OK; }
  if (!q || !k || !v || !gate || !o) return SEED_ERR_INVALID_ARG;
  if (st->variant != SEED_MAMBA2 && !beta) return SEED_ERR_INVALID_ARG;
  if (st->variant == SEED_MAMBA2 && !A) return SEED_ERR_INVALID_ARG;
  if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(o)) return SEED_ERR_ALIGNMENT;
  if (st->variant == SEED_KDA && misaligned(gate)) return SEED_ERR_ALIGNMENT;
  const int cols = rmax_of(st) + growth_of(st->variant) * st->steps_since_compress;
  c = cuda_status(launch_decode(view_of(st), st->factor_dtype, q, k, v, gate, beta, A, o, cols,
                                (cudaStream_t)stream));
  if (c == SEED_OK) ++st->steps_since_compress;
  return c;
}

extern "C" int seed_recompress_ex(seed_state *st, float *trunc_err, int32_t *sweeps,
                                  seed_stream_t stream) {
  int c = check_state(st);
  if (c) return c;
  if (st->steps_since_compress > st->T) return SEED_ERR_CAPACITY;
  if (st->n_heads == 0) { st->steps_since_compress = 0; return SEED_OK; }
  const int m_max = rmax_of(st) + growth_of(st->variant) * st->steps_since_compress;
  c = cuda_status(launch_recompress(view_of(st), st->factor_dtype, trunc_err, sweeps, m_max,
                                    (cudaStream_t)stream));
  if (c == SEED_OK) st->steps_since_compress = 0;
  return c;
}

extern "C" int seed_recompress_workspace_bytes(const seed_state *st, int32_t heads, int64_t *bytes) {
  const int c = check_state(st);
  if (c) return c;
  if (heads < 1 || !bytes) return SEED_ERR_INVALID_ARG;
  const int rmax = rmax_of(st);
  const int m_cap = rmax + growth_of(st->variant) * st->T;
  *bytes = (int64_t)heads * split_floats_per_head(st->factor_dtype, m_cap, rmax, st->d_v) * (int64_t)sizeof(float);
  return SEED_OK;
}

extern "C" int seed_recompress_ws(seed_state *st, float *trunc_err, int32_t *sweeps, void *workspace,
                                  int64_t workspace_bytes, seed_stream_t stream) {
  int c = check_state(st);
  if (c) return c;
  if (st->steps_since_compress > st->T) return SEED_ERR_CAPACITY;
  if (st->n_heads == 0) { st->steps_since_compress = 0; return SEED_OK; }
  if (!workspace || workspace_bytes < 0) return SEED_ERR_INVALID_ARG;
  if (misaligned(workspace)) return SEED_ERR_ALIGNMENT;
  const int rmax = rmax_of(st);
  const int m_max = rmax + growth_of(st->variant) * st->steps_since_compress;
  const int64_t per_head = split_floats_per_head(st->factor_dtype, m_max, rmax, st->d_v) * (int64_t)sizeof(float);
  const int64_t chunk = workspace_bytes / per_head;
  if (chunk < 1) return SEED_ERR_INVALID_ARG;
  c = cuda_status(launch_recompress_split(view_of(st), st->factor_dtype, trunc_err, sweeps, m_max, rmax,
                                          static_cast<float *>(workspace), chunk, (cudaStream_t)stream));
  if (c == SEED_OK) st->steps_since_compress = 0;
  return c;
}

extern "C" int seed_recompress_noalloc(seed_state *st, float *trunc_err, int32_t *sweeps,
                                       seed_stream_t stream) {
  int c = check_state(st);
  if (c) return c;
  if (st->steps_since_compress > st->T) return SEED_ERR_CAPACITY;
  if (st->n_heads == 0) { st->steps_since_compress = 0; return SEED_OK; }
  const int rmax = rmax_of(st);
  const int m_max = rmax + growth_of(st->variant) * st->steps_since_compress;
  const int64_t need = (int64_t)st->n_heads * split_floats_per_head(st->factor_dtype, m_max, rmax, st->d_v);
  if (need > kNoAllocScratchFloats) return SEED_ERR_UNSUPPORTED_SHAPE;  // checked before any CUDA call
  float *scratch = nullptr;
  if (noalloc_scratch(&scratch) != cudaSuccess) return SEED_ERR_CUDA;
  c = cuda_status(launch_recompress_split(view_of(st), st->factor_dtype, trunc_err, sweeps, m_max, rmax,
                                          scratch, st->n_heads, (cudaStream_t)stream));
  if (c == SEED_OK) st->steps_since_compress = 0;
  return c;
}

extern "C" int seed_recompress(seed_state *st, float *trunc_err, seed_stream_t stream) {
  return seed_recompress_ex(st, trunc_err, nullptr, stream);
}

extern "C" int seed_materialize(const seed_state *st, float *S_out, seed_stream_t stream) {
  int c = check_state(st);
  if (c) return c;
  if (st->steps_since_compress > st->T) return SEED_ERR_CAPACITY;
  if (st->n_heads == 0) return SEED_OK;
  if (!S_out) return SEED_ERR_INVALID_ARG;
  const int m_max = rmax_of(st) + growth_of(st->variant) * st->steps_since_compress;
  return cuda_status(launch_materialize(view_of(st), st->factor_dtype, S_out, m_max > 0 ? m_max : 1,
                                        (cudaStream_t)stream));
}

extern "C" int seed_dense_decode_step(int32_t variant, int32_t n_heads, int32_t d_k, int32_t d_v,
                                      float *S, const float *q, const float *k, const float *v,
                                      const float *gate, const float *beta, const float *A,
                                      const int32_t *dir_index, float *o, seed_stream_t stream) {
  if (variant < SEED_GDN || variant > SEED_MAMBA2 || n_heads < 0) return SEED_ERR_INVALID_ARG;
  if (d_k != kDK || (d_v != 64 && d_v != 128)) return SEED_ERR_UNSUPPORTED_SHAPE;
  if (n_heads == 0) return SEED_OK;
  if (!S || !q || !k || !v || !gate || !o) return SEED_ERR_INVALID_ARG;
  if (variant != SEED_MAMBA2 && !beta) return SEED_ERR_INVALID_ARG;
  if (variant == SEED_MAMBA2 && !A) return SEED_ERR_INVALID_ARG;
  if (misaligned(S) || misaligned(q) || misaligned(k) || misaligned(v) || misaligned(o))
    return SEED_ERR_ALIGNMENT;
  return cuda_status(launch_dense_decode(variant, n_heads, d_v, S, q, k, v, gate, beta, A, dir_index,
                                         o, (cudaStream_t)stream));
}
