/*
 * seed_synth.h — device twin of the seeded synthetic-workload generator
 * (libseed.so).  Not part of the method: it produces the inputs that the
 * benchmark and the tests feed to the calls of seed.h, on the GPU, with the
 * same counter layout as the host generator in the Python module `synth`.
 *
 * Generator: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11).
 *   key     = (seed, (phase << 16) | field)
 *   counter = (block, time, entity, 0)
 * Uniforms u(x) = ((x >> 9) + 0.5) * 2^-23; normals by Box-Muller on word pairs
 * (block b -> values 4b..4b+3).  Raw words match the host bit for bit; floats
 * agree to a few ulp.
 *
 * Workload recipe (one per synthetic workload; heads flattened as
 * h = (request * n_layers + layer) * n_head + head, direction = h mod (n_layers * n_head)):
 *   GDN / KDA:  q, k ~ N(0, I) normalised to unit length;  v = s_dir vbar_dir + noise_std N(0, I);
 *               alpha ~ U[alpha_lo, alpha_hi] (per head, or per channel for KDA);
 *               beta ~ U[beta_lo, beta_hi]
 *   Mamba-2:    C, B ~ N(0, I/N);  x = s_dir xbar_dir + noise_std N(0, I);
 *               dt = softplus(dt_mu + sqrt(dt_var) N(0,1));  A_dir = -U[a_lo, a_hi]
 *   vbar_dir:   normalised N(0, I);  s_dir ~ U[sink_lo, sink_hi]
 *   rank(h):    uniform over rank_choices (or `rank`);  prompt length per request ~
 *               uniform integer in [prefill_lo, prefill_hi] (or `prefill_len`)
 * All pointers are device pointers owned by the caller; calls are asynchronous on
 * `stream` and return seed_status codes (seed.h).
 */
#ifndef SEED_SYNTH_H_
#define SEED_SYNTH_H_

#include <stdint.h>
#include "seed.h"

#ifdef __cplusplus
extern "C" {
#endif

enum { SEED_SYNTH_PHASE_CONST = 0, SEED_SYNTH_PHASE_PREFILL = 1, SEED_SYNTH_PHASE_DECODE = 2 };

typedef struct {
  int32_t variant;                 /* seed_variant */
  int32_t n_req, n_layers, n_head; /* n_heads = n_req * n_layers * n_head */
  int32_t d_k, d_v;
  uint32_t seed;
  int32_t prefill_len;             /* fixed prompt length, or 0: per-request lengths */
  int32_t prefill_lo, prefill_hi;
  int32_t rank;                    /* uniform rank, or 0: rank_choices */
  int32_t n_rank_choices;
  int32_t rank_choices[4];
  float sink_lo, sink_hi, noise_std;
  float alpha_lo, alpha_hi, beta_lo, beta_hi;
  float a_lo, a_hi, dt_mu, dt_var;
} seed_synth_workload;

/* Raw generator words: out[i*4*n_blocks + 4*b + w] for entity = entity0 + i, block b. */
int seed_synth_raw(uint32_t seed, int32_t phase, int32_t field, uint32_t time, uint32_t entity0,
                   int32_t n_entities, int32_t n_blocks, uint32_t *out, seed_stream_t stream);

/*
 * Per-direction and per-head constants.  Any output may be NULL.
 *   vbar        [n_dir][d_v]   unit sink directions
 *   sink_scale  [n_dir]
 *   A           [n_dir]        Mamba-2 A (negative)
 *   rank        [n_heads]
 *   prompt_len  [n_req]
 */
int seed_synth_constants(const seed_synth_workload *w, float *vbar, float *sink_scale, float *A,
                         int32_t *rank, int32_t *prompt_len, seed_stream_t stream);

/*
 * Inputs of one decode step for heads [head0, head0 + n_heads).
 *   q, k [n][d_k], v [n][d_v], gate ([n] or [n][d_k] for KDA; dt for Mamba-2),
 *   beta [n] (NULL allowed for Mamba-2).  Needs vbar and sink_scale from
 *   seed_synth_constants.
 */
int seed_synth_step_inputs(const seed_synth_workload *w, int32_t phase, int32_t time, int64_t head0,
                           int32_t n_heads, const float *vbar, const float *sink_scale, float *q,
                           float *k, float *v, float *gate, float *beta, seed_stream_t stream);

/*
 * Dense fp32 prefill of every head from S = 0 over its request's prompt, with
 * the prompt tokens generated inside the kernel (phase PREFILL, time = token).
 *   prompt_len [n_req] (from seed_synth_constants), vbar, sink_scale, A as above,
 *   S_out [n_heads][d_k][d_v].  Heads [head0, head0 + n_heads) only.
 */
int seed_synth_dense_prefill(const seed_synth_workload *w, int64_t head0, int32_t n_heads,
                             const int32_t *prompt_len, const float *vbar, const float *sink_scale,
                             const float *A, float *S_out, seed_stream_t stream);

/*
 * The same prefill, advanced a chunk of tokens at a time (32 tokens for the
 * scalar gates, 16 for the per-channel gate) in the chunkwise form of the
 * delta rule: within a chunk the corrections u_t solve a unit lower-triangular
 * system built from the chunk's key inner products and gate ratios, and the
 * state takes one rank-C update per chunk (the WY / UT form of Yang et al.,
 * "Parallelizing Linear Transformers with the Delta Rule over Sequence
 * Length", NeurIPS 2024, with the gates carried exactly; for the per-channel
 * gate, which acts after the erase, two update terms per token).  The result is
 * the token-serial recurrence's up to fp32 rounding order.  Arguments, layout,
 * ownership and errors as seed_synth_dense_prefill.  Where the smallest scalar
 * or per-channel gate raised to the chunk length falls below 2^-96 (the
 * cumulative products could leave fp32's normal range), the call runs
 * seed_synth_dense_prefill instead.  Mamba-2 chunks work with the logarithm of
 * the cumulative decay and have no such limit.
 */
int seed_synth_dense_prefill_chunked(const seed_synth_workload *w, int64_t head0, int32_t n_heads,
                                     const int32_t *prompt_len, const float *vbar,
                                     const float *sink_scale, const float *A, float *S_out,
                                     seed_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SEED_SYNTH_H_ */
