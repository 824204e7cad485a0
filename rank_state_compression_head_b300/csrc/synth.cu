// Device twin of the seeded synthetic-workload generator, and the dense fp32
// prefill whose prompt tokens are generated inside the kernel.
//
// Generator: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11), written from
// its published definition, with the counter layout of the host generator:
// key = (seed, phase << 16 | field), counter = (block, time, entity, 0).
//
// The prefill runs the dense recurrence over each request's prompt from S = 0
// ("Shallow Encoding Emits Deep Memories", thelatestinai.com list view,
// Table 1: the states that leave the prefill are then compressed), with the
// state held in registers for the whole prompt and the tokens generated on
// the fly, so no prompt input is ever stored.
#include "common.cuh"
#include "seed_synth.h"

namespace seedk {

enum { F_Q = 1, F_K = 2, F_V = 3, F_ALPHA = 4, F_BETA = 5, F_DT = 6,
       F_VBAR = 16, F_SINK = 17, F_A = 18, F_RANK = 19, F_CTX = 20 };

// philox(): common.cuh

__device__ __forceinline__ uint32_t fkey(int phase, int field) {
  return ((uint32_t)(phase & 0xFFFF) << 16) | (uint32_t)(field & 0xFFFF);
}

__device__ __forceinline__ float uni(uint32_t x) {
  return ((float)(x >> 9) + 0.5f) * 1.1920928955078125e-07f;  // 2^-23
}

// Four standard normals of block `blk` (Box-Muller on word pairs).
__device__ __forceinline__ float4 normal4(uint32_t seed, int phase, int field, uint32_t time,
                                          uint32_t entity, uint32_t blk) {
  const uint4 w = philox(blk, time, entity, 0u, seed, fkey(phase, field));
  const float r01 = sqrtf(-2.f * logf(uni(w.x)));
  const float r23 = sqrtf(-2.f * logf(uni(w.z)));
  float s1, c1, s3, c3;
  sincospif(2.f * uni(w.y), &s1, &c1);
  sincospif(2.f * uni(w.w), &s3, &c3);
  return make_float4(r01 * c1, r01 * s1, r23 * c3, r23 * s3);
}

__device__ __forceinline__ float uniform1(uint32_t seed, int phase, int field, uint32_t time,
                                          uint32_t entity) {
  return uni(philox(0u, time, entity, 0u, seed, fkey(phase, field)).x);
}

__device__ __forceinline__ float softplusf(float x) { return log1pf(expf(x)); }

// ---------------------------------------------------------------------------

__global__ void raw_kernel(uint32_t seed, int phase, int field, uint32_t time, uint32_t entity0,
                           int n_ent, int n_blocks, uint32_t *out) {
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (int64_t)n_ent * n_blocks) return;
  const int i = (int)(idx / n_blocks), b = (int)(idx % n_blocks);
  const uint4 w = philox((uint32_t)b, time, entity0 + (uint32_t)i, 0u, seed, fkey(phase, field));
  reinterpret_cast<uint4 *>(out)[idx] = w;
}

// One warp per direction / head / request (grid-stride).
__global__ void constants_kernel(const seed_synth_workload w, float *vbar, float *sink, float *A,
                                 int32_t *rank, int32_t *plen) {
  const int lane = threadIdx.x & 31;
  const int64_t wid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int n_dir = w.n_layers * w.n_head;
  const int64_t n_heads = (int64_t)n_dir * w.n_req;
  for (int64_t d = wid; d < n_dir; d += nwarps) {
    if (vbar) {
      float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
      if (lane < w.d_v / 4) z = normal4(w.seed, SEED_SYNTH_PHASE_CONST, F_VBAR, 0u, (uint32_t)d, lane);
      const float ss = warp_sum(z.x * z.x + z.y * z.y + z.z * z.z + z.w * z.w);
      const float nrm = sqrtf(ss);
      if (lane < w.d_v / 4)
        reinterpret_cast<float4 *>(vbar + d * w.d_v)[lane] =
            make_float4(z.x / nrm, z.y / nrm, z.z / nrm, z.w / nrm);
    }
    if (lane == 0 && sink) {
      const float u = uniform1(w.seed, SEED_SYNTH_PHASE_CONST, F_SINK, 0u, (uint32_t)d);
      sink[d] = w.sink_lo + (w.sink_hi - w.sink_lo) * u;
    }
    if (lane == 0 && A) {
      const float u = uniform1(w.seed, SEED_SYNTH_PHASE_CONST, F_A, 0u, (uint32_t)d);
      A[d] = -(w.a_lo + (w.a_hi - w.a_lo) * u);
    }
  }
  if (rank) {
    for (int64_t h = wid * 32 + lane; h < n_heads; h += nwarps * 32) {
      if (w.rank > 0) { rank[h] = w.rank; continue; }
      const uint32_t x = philox(0u, 0u, (uint32_t)h, 0u, w.seed, fkey(SEED_SYNTH_PHASE_CONST, F_RANK)).x;
      const uint32_t i = (uint32_t)(((uint64_t)x * (uint64_t)w.n_rank_choices) >> 32);
      rank[h] = w.rank_choices[i];
    }
  }
  if (plen) {
    for (int64_t q = wid * 32 + lane; q < w.n_req; q += nwarps * 32) {
      if (w.prefill_len > 0) { plen[q] = w.prefill_len; continue; }
      const uint32_t x = philox(0u, 0u, (uint32_t)q, 0u, w.seed, fkey(SEED_SYNTH_PHASE_CONST, F_CTX)).x;
      const uint64_t span = (uint64_t)(w.prefill_hi - w.prefill_lo + 1);
      plen[q] = w.prefill_lo + (int32_t)(((uint64_t)x * span) >> 32);
    }
  }
}

// Token inputs of one head, written by warps 0..3 of the calling block.
//   GDN/KDA: out0 = q (unit), out1 = k (unit), out2 = v, gate = alpha, beta
//   Mamba-2: out0 = C, out1 = B, out2 = x, gate = dt
// Returns nothing; the caller synchronises before reading.
__device__ __forceinline__ void gen_token(const seed_synth_workload &w, int phase, uint32_t time,
                                          uint32_t head, int dir, const float *vbar_d, float sink_d,
                                          float *out0, float *out1, float *out2, float *gate,
                                          float *beta, bool need_q) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool m2 = w.variant == SEED_MAMBA2;
  if (warp == 0 || warp == 1) {
    if (warp == 0 && !need_q) return;
    float *out = warp == 0 ? out0 : out1;
    float4 z = normal4(w.seed, phase, warp == 0 ? F_Q : F_K, time, head, lane);  // d_k = 128: 32 blocks
    if (m2) {
      const float sd = 1.f / sqrtf((float)w.d_k);
      z = make_float4(z.x * sd, z.y * sd, z.z * sd, z.w * sd);
    } else {
      const float nrm = sqrtf(warp_sum(z.x * z.x + z.y * z.y + z.z * z.z + z.w * z.w));
      z = make_float4(z.x / nrm, z.y / nrm, z.z / nrm, z.w / nrm);
    }
    reinterpret_cast<float4 *>(out)[lane] = z;
  } else if (warp == 2) {
    if (lane < w.d_v / 4) {
      const float4 z = normal4(w.seed, phase, F_V, time, head, lane);
      const float4 vb = reinterpret_cast<const float4 *>(vbar_d)[lane];
      const float sd = w.noise_std;
      reinterpret_cast<float4 *>(out2)[lane] =
          make_float4(fmaf(sink_d, vb.x, sd * z.x), fmaf(sink_d, vb.y, sd * z.y),
                      fmaf(sink_d, vb.z, sd * z.z), fmaf(sink_d, vb.w, sd * z.w));
    }
  } else if (warp == 3) {
    if (m2) {
      if (lane == 0) {
        const float z = normal4(w.seed, phase, F_DT, time, head, 0u).x;
        gate[0] = softplusf(w.dt_mu + sqrtf(w.dt_var) * z);
      }
    } else if (w.variant == SEED_KDA) {
      const uint4 x = philox((uint32_t)lane, time, head, 0u, w.seed, fkey(phase, F_ALPHA));
      const float sp = w.alpha_hi - w.alpha_lo;
      reinterpret_cast<float4 *>(gate)[lane] =
          make_float4(w.alpha_lo + sp * uni(x.x), w.alpha_lo + sp * uni(x.y),
                      w.alpha_lo + sp * uni(x.z), w.alpha_lo + sp * uni(x.w));
      if (lane == 0)
        beta[0] = w.beta_lo + (w.beta_hi - w.beta_lo) * uniform1(w.seed, phase, F_BETA, time, head);
    } else if (lane == 0) {
      gate[0] = w.alpha_lo + (w.alpha_hi - w.alpha_lo) * uniform1(w.seed, phase, F_ALPHA, time, head);
      beta[0] = w.beta_lo + (w.beta_hi - w.beta_lo) * uniform1(w.seed, phase, F_BETA, time, head);
    }
  }
}

__global__ void __launch_bounds__(128) step_inputs_kernel(const seed_synth_workload w, int phase,
                                                          int time, int64_t head0,
                                                          const float *vbar, const float *sink,
                                                          float *q, float *k, float *v, float *gate,
                                                          float *beta) {
  const int64_t i = blockIdx.x;
  const int64_t h = head0 + i;
  const int n_dir = w.n_layers * w.n_head;
  const int dir = (int)(h % n_dir);
  const bool kda = w.variant == SEED_KDA;
  float *bptr = (beta && w.variant != SEED_MAMBA2) ? beta + i : nullptr;
  float dummy;
  gen_token(w, phase, (uint32_t)time, (uint32_t)h, dir, vbar + (int64_t)dir * w.d_v, sink[dir],
            q + i * w.d_k, k + i * w.d_k, v + i * w.d_v, gate + (kda ? i * w.d_k : i),
            bptr ? bptr : &dummy, true);
}

// Dense prefill: one CTA of 256 threads per head; state rows distributed as in
// the dense decode step (thread holds NL float4 row pieces).
template <int VAR, int DV>
__global__ void __launch_bounds__(256) prefill_kernel(const seed_synth_workload w, int64_t head0,
                                                      const int32_t *plen, const float *vbar,
                                                      const float *sink, const float *A,
                                                      float *S_out) {
  constexpr int DK = kDK;
  constexpr int NW = 8;
  constexpr int LPR = DV / 4;
  constexpr int RPW = 32 / LPR;
  constexpr int NL = DK / (RPW * NW);
  constexpr int NG = NW * RPW;
  constexpr bool M2 = VAR == SEED_MAMBA2;
  constexpr bool KDA = VAR == SEED_KDA;
  __shared__ __align__(16) float kin[2][DK];
  __shared__ __align__(16) float vin[2][DV];
  __shared__ __align__(16) float gin[2][DK];
  __shared__ float bin[2];
  __shared__ __align__(16) float red[NG][DV];

  const int64_t hi = blockIdx.x;
  const int64_t h = head0 + hi;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_dir = w.n_layers * w.n_head;
  const int dir = (int)(h % n_dir);
  const int req = (int)(h / n_dir);
  const int L = plen[req];
  const float *vb = vbar + (int64_t)dir * DV;
  const float sd = sink[dir];
  const float Ad = M2 ? A[dir] : 0.f;
  const int c4 = (lane % LPR) * 4;
  const int grp = warp * RPW + lane / LPR;

  float4 st[NL];
#pragma unroll
  for (int l = 0; l < NL; ++l) st[l] = make_float4(0.f, 0.f, 0.f, 0.f);

  if (L > 0)
    gen_token(w, SEED_SYNTH_PHASE_PREFILL, 0u, (uint32_t)h, dir, vb, sd, nullptr, kin[0], vin[0],
              gin[0], &bin[0], false);
  __syncthreads();
  for (int t = 0; t < L; ++t) {
    const int b = t & 1;
    const float4 v4 = *reinterpret_cast<const float4 *>(&vin[b][c4]);
    if (!M2) {
      float4 u = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int l = 0; l < NL; ++l) {
        const int row = (l * NW + warp) * RPW + lane / LPR;
        const float kr = kin[b][row];
        u.x = fmaf(kr, st[l].x, u.x); u.y = fmaf(kr, st[l].y, u.y);
        u.z = fmaf(kr, st[l].z, u.z); u.w = fmaf(kr, st[l].w, u.w);
      }
      *reinterpret_cast<float4 *>(&red[grp][c4]) = u;
    }
    if (t + 1 < L)
      gen_token(w, SEED_SYNTH_PHASE_PREFILL, (uint32_t)(t + 1), (uint32_t)h, dir, vb, sd, nullptr,
                kin[b ^ 1], vin[b ^ 1], gin[b ^ 1], &bin[b ^ 1], false);
    __syncthreads();
    if (!M2) {
      float4 u = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int gi = 0; gi < NG; ++gi) {
        const float4 x = *reinterpret_cast<const float4 *>(&red[gi][c4]);
        u.x += x.x; u.y += x.y; u.z += x.z; u.w += x.w;
      }
      const float beta = bin[b];
#pragma unroll
      for (int l = 0; l < NL; ++l) {
        const int row = (l * NW + warp) * RPW + lane / LPR;
        const float kr = kin[b][row];
        if (KDA) {
          const float ar = gin[b][row];
          const float bk = beta * kr;
          st[l].x = fmaf(ar, fmaf(-bk, u.x, st[l].x), bk * v4.x);
          st[l].y = fmaf(ar, fmaf(-bk, u.y, st[l].y), bk * v4.y);
          st[l].z = fmaf(ar, fmaf(-bk, u.z, st[l].z), bk * v4.z);
          st[l].w = fmaf(ar, fmaf(-bk, u.w, st[l].w), bk * v4.w);
        } else {
          const float g = gin[b][0];
          st[l].x = fmaf(g, st[l].x, kr * beta * fmaf(-g, u.x, v4.x));
          st[l].y = fmaf(g, st[l].y, kr * beta * fmaf(-g, u.y, v4.y));
          st[l].z = fmaf(g, st[l].z, kr * beta * fmaf(-g, u.z, v4.z));
          st[l].w = fmaf(g, st[l].w, kr * beta * fmaf(-g, u.w, v4.w));
        }
      }
    } else {
      const float dt = gin[b][0];
      const float g = expf(dt * Ad);
#pragma unroll
      for (int l = 0; l < NL; ++l) {
        const int row = (l * NW + warp) * RPW + lane / LPR;
        const float bb = dt * kin[b][row];
        st[l].x = fmaf(g, st[l].x, bb * v4.x); st[l].y = fmaf(g, st[l].y, bb * v4.y);
        st[l].z = fmaf(g, st[l].z, bb * v4.z); st[l].w = fmaf(g, st[l].w, bb * v4.w);
      }
    }
    __syncthreads();
  }
  float *Sh = S_out + hi * DK * DV;
#pragma unroll
  for (int l = 0; l < NL; ++l) {
    const int row = (l * NW + warp) * RPW + lane / LPR;
    *reinterpret_cast<float4 *>(Sh + row * DV + c4) = st[l];
  }
}

// ---------------------------------------------------------------------------
// Chunked (parallel-in-time) dense prefill.
//
// The same recurrence as prefill_kernel, advanced C tokens at a time in the
// chunkwise form of the delta rule (the WY / UT-transform form of Yang, Wang,
// Zhang, Shen, Kim, "Parallelizing Linear Transformers with the Delta Rule over
// Sequence Length", NeurIPS 2024), with the gates carried exactly.  Within a
// chunk from S_0, gamma_t is the product of the gates up to token t (per channel
// for the per-channel gate) and gm_t = gamma_{t-1} (gm_0 = 1).
//
//   scalar gate:  S_t = alpha_t S_{t-1} + k_t u_t^T,  u_t = beta_t (v_t - alpha_t S_{t-1}^T k_t),
//     so (I + A) U = diag(beta) (V - P), P_t = gamma_t k_t^T S_0,
//     A[t][r] = beta_t (gamma_t / gamma_r) k_t . k_r (r < t), forward substitution,
//     and S_C = gamma_C S_0 + sum_t (gamma_C / gamma_t) k_t u_t^T.
//   per-channel gate after the erase (diag(alpha)(I - beta k k^T) S + beta k v^T):
//     S_t = diag(alpha_t) S_{t-1} + (alpha_t * k_t) x_t^T + k_t y_t^T,
//     y_t = beta_t v_t,  x_t = -beta_t S_{t-1}^T k_t, so with P_t = k_t^T diag(gm_t) S_0,
//     Cm[t][r] = sum_i k_t[i] k_r[i] gm_t[i] / gm_r[i],  E[t][r] = sum_i k_t[i] k_r[i] gm_t[i] / gamma_r[i]:
//       x_t = -beta_t (P_t + sum_{r<t} E[t][r] y_r) - beta_t sum_{r<t} Cm[t][r] x_r,
//     S_C = diag(gamma_C) S_0 + sum_r (gamma_C / gm_r * k_r) x_r^T + (gamma_C / gamma_r * k_r) y_r^T.
//   Mamba-2 (no erase): S_C = gamma_C S_0 + sum_t (gamma_C / gamma_t) dt_t B_t x_t^T.
// All arithmetic is fp32 FMA.  One CTA of 256 threads per head; thread
// (q, jp) holds columns 2jp and 2jp + 1 of the state for a quarter (d_v = 128) or
// an eighth (d_v = 64) of its rows in registers, so that each key value it reads
// from shared memory serves two columns; the chunk's tokens are generated in
// parallel (one warp a token); the triangular solve takes one column a thread.
// ---------------------------------------------------------------------------

// One warp generates every input of one prefill token (the values of gen_token).
__device__ __forceinline__ void gen_token_warp(const seed_synth_workload &w, uint32_t time, uint32_t head,
                                               const float *vbar_d, float sink_d, bool live, float *kout,
                                               float *vout, float *gout, float *bout) {
  const int lane = threadIdx.x & 31;
  const bool m2 = w.variant == SEED_MAMBA2, kda = w.variant == SEED_KDA;
  const int phase = SEED_SYNTH_PHASE_PREFILL;
  float4 z = live ? normal4(w.seed, phase, F_K, time, head, lane) : make_float4(0.f, 0.f, 0.f, 0.f);
  if (m2) {
    const float sd = 1.f / sqrtf((float)w.d_k);
    z = make_float4(z.x * sd, z.y * sd, z.z * sd, z.w * sd);
  } else {
    const float nrm = sqrtf(warp_sum(z.x * z.x + z.y * z.y + z.z * z.z + z.w * z.w));
    if (nrm > 0.f) z = make_float4(z.x / nrm, z.y / nrm, z.z / nrm, z.w / nrm);
  }
  reinterpret_cast<float4 *>(kout)[lane] = z;
  if (lane < w.d_v / 4) {
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (live) {
      const float4 n = normal4(w.seed, phase, F_V, time, head, lane);
      const float4 vb = reinterpret_cast<const float4 *>(vbar_d)[lane];
      const float sd = w.noise_std;
      v = make_float4(fmaf(sink_d, vb.x, sd * n.x), fmaf(sink_d, vb.y, sd * n.y), fmaf(sink_d, vb.z, sd * n.z),
                      fmaf(sink_d, vb.w, sd * n.w));
    }
    reinterpret_cast<float4 *>(vout)[lane] = v;
  }
  if (kda) {
    float4 a = make_float4(1.f, 1.f, 1.f, 1.f);
    if (live) {
      const uint4 x = philox((uint32_t)lane, time, head, 0u, w.seed, fkey(phase, F_ALPHA));
      const float sp = w.alpha_hi - w.alpha_lo;
      a = make_float4(w.alpha_lo + sp * uni(x.x), w.alpha_lo + sp * uni(x.y), w.alpha_lo + sp * uni(x.z),
                      w.alpha_lo + sp * uni(x.w));
    }
    reinterpret_cast<float4 *>(gout)[lane] = a;
  }
  if (lane == 0) {
    if (m2) {
      gout[0] = live ? softplusf(w.dt_mu + sqrtf(w.dt_var) * normal4(w.seed, phase, F_DT, time, head, 0u).x) : 0.f;
    } else {
      if (!kda) gout[0] = live ? w.alpha_lo + (w.alpha_hi - w.alpha_lo) * uniform1(w.seed, phase, F_ALPHA, time, head) : 1.f;
      bout[0] = live ? w.beta_lo + (w.beta_hi - w.beta_lo) * uniform1(w.seed, phase, F_BETA, time, head) : 0.f;
    }
  }
}

template <int VAR>
constexpr int chunk_len() { return VAR == SEED_KDA ? 16 : 32; }

template <int VAR, int DV>
struct ChunkSmem {
  static constexpr int DK = kDK, C = chunk_len<VAR>();
  static constexpr int NQ = 512 / DV;                         // row groups of the state (two columns a thread)
  static constexpr bool KDA = VAR == SEED_KDA;
  static constexpr int K_OFF = 0;                             // [C][DK] keys, later update weights
  static constexpr int V_OFF = K_OFF + C * DK;                // [C][DV] values, later U (or y)
  static constexpr int G_OFF = V_OFF + C * DV;                // KDA [C][DK] gates -> gamma, later weights; else [C]
  static constexpr int GI_OFF = G_OFF + (KDA ? C * DK : C);   // KDA [C][DK] 1/gamma; else [C] gamma
  static constexpr int GC_OFF = GI_OFF + (KDA ? C * DK : C);  // KDA [DK] gamma_C
  static constexpr int B_OFF = GC_OFF + (KDA ? DK : 4);       // [C] beta
  static constexpr int A_OFF = B_OFF + C;                     // [C][C + 1] the strictly lower A (or Cm)
  static constexpr int E_OFF = A_OFF + C * (C + 1);           // KDA [C][C + 1] E
  static constexpr int P_OFF = E_OFF + (KDA ? C * (C + 1) : 0);  // [NQ][C][DV] partial P, then x in slice 0
  static constexpr int FLOATS = (P_OFF + NQ * C * DV + 3) & ~3;
};

template <int VAR, int DV>
__global__ void __launch_bounds__(256, 2) prefill_chunk_kernel(const seed_synth_workload w, int64_t head0,
                                                               const int32_t *plen, const float *vbar,
                                                               const float *sink, const float *A, float *S_out) {
  constexpr int DK = kDK;
  using L = ChunkSmem<VAR, DV>;
  constexpr int C = L::C, NQ = L::NQ, RPT = DK / NQ;
  constexpr bool M2 = VAR == SEED_MAMBA2, KDA = VAR == SEED_KDA;
  extern __shared__ __align__(16) float sm[];
  float *Kc = sm + L::K_OFF, *Vc = sm + L::V_OFF, *Gc = sm + L::G_OFF, *Gi = sm + L::GI_OFF;
  float *gCr = sm + L::GC_OFF, *Bc = sm + L::B_OFF, *Am = sm + L::A_OFF, *Em = sm + L::E_OFF, *Pp = sm + L::P_OFF;

  const int64_t h = head0 + blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5;
  // state mapping: thread (q, jp) holds columns j2, j2 + 1 of rows i0 .. i0 + RPT - 1, so that
  // every key value read from shared memory serves two columns
  const int jp = tid % (DV / 2), q = tid / (DV / 2), i0 = q * RPT, j2 = 2 * jp;
  const int j = tid;  // the triangular solve: one column per thread (tid < DV)
  const int n_dir = w.n_layers * w.n_head;
  const int dir = (int)(h % n_dir);
  const int L_tok = plen[h / n_dir];
  const float *vb = vbar + (int64_t)dir * DV;
  const float sd = sink[dir];
  const float Ad = M2 ? A[dir] : 0.f;

  float st[RPT][2];
#pragma unroll
  for (int r = 0; r < RPT; ++r) st[r][0] = st[r][1] = 0.f;

  for (int t0 = 0; t0 < L_tok; t0 += C) {
    // ---- the chunk's tokens (past the prompt: identity steps) ----------------------------------
    for (int t = warp; t < C; t += 8)
      gen_token_warp(w, (uint32_t)(t0 + t), (uint32_t)h, vb, sd, t0 + t < L_tok, Kc + t * DK, Vc + t * DV,
                     KDA ? Gc + t * DK : Gc + t, Bc + t);
    __syncthreads();
    // ---- cumulative gates (products of the per-step gates, as the recurrence) ------------------
    if (KDA) {
      if (tid < DK) {
        float g = 1.f;
        for (int t = 0; t < C; ++t) {
          g *= Gc[t * DK + tid];
          Gc[t * DK + tid] = g;
          Gi[t * DK + tid] = 1.f / g;
        }
        gCr[tid] = g;
      }
    } else if (tid == 0) {
      // gamma_t for the scalar gate; for Mamba-2 its logarithm (sum of dt A), so that
      // no ratio of two underflowing products is ever formed (Gc keeps the step gate or dt)
      float g = M2 ? 0.f : 1.f;
      for (int t = 0; t < C; ++t) {
        if (M2) g = fmaf(Gc[t], Ad, g);
        else g *= Gc[t];
        Gi[t] = g;
      }
    }
    __syncthreads();
    if (!M2) {
      // ---- the strictly lower chunk matrices ------------------------------------------------------
      for (int pr = tid; pr < C * (C - 1) / 2; pr += 256) {
        int t = 1, rem = pr;  // pr -> (t, r), r < t
        while (rem >= t) { rem -= t; ++t; }
        const int r = rem;
        const float4 *kt = reinterpret_cast<const float4 *>(Kc + t * DK);
        const float4 *kr = reinterpret_cast<const float4 *>(Kc + r * DK);
        if (KDA) {
          // gm_t / gm_r and gm_t / gamma_r, with gm_t = gamma_{t-1} and 1/gm_r = 1/gamma_{r-1}
          const float4 *gmt = reinterpret_cast<const float4 *>(Gc + (t - 1) * DK);
          const float4 *igr = reinterpret_cast<const float4 *>(Gi + r * DK);
          const float4 *igmr = reinterpret_cast<const float4 *>(Gi + (r - 1) * DK);
          float cm = 0.f, e = 0.f;
#pragma unroll 4
          for (int i4 = 0; i4 < DK / 4; ++i4) {
            const float4 a = kt[i4], b = kr[i4], g = gmt[i4], ig = igr[i4];
            const float4 igm = r > 0 ? igmr[i4] : make_float4(1.f, 1.f, 1.f, 1.f);
            const float px = a.x * b.x * g.x, py = a.y * b.y * g.y, pz = a.z * b.z * g.z, pw = a.w * b.w * g.w;
            cm = fmaf(px, igm.x, fmaf(py, igm.y, fmaf(pz, igm.z, fmaf(pw, igm.w, cm))));
            e = fmaf(px, ig.x, fmaf(py, ig.y, fmaf(pz, ig.z, fmaf(pw, ig.w, e))));
          }
          Am[t * (C + 1) + r] = cm;
          Em[t * (C + 1) + r] = e;
        } else {
          float acc = 0.f;
#pragma unroll 4
          for (int i4 = 0; i4 < DK / 4; ++i4) {
            const float4 a = kt[i4], b = kr[i4];
            acc = fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, fmaf(a.w, b.w, acc))));
          }
          Am[t * (C + 1) + r] = Bc[t] * (Gi[t] / Gi[r]) * acc;
        }
      }
      // ---- partial P over my rows: P[q][t][j] = sum_i k_t[i] w_t[i] S_0[i][j] ----------------------
      // (w_t = gamma_t for the scalar gate, applied after; gm_t per channel)
      // (tokens in halves of 16 to bound the accumulators)
#pragma unroll
      for (int th = 0; th < C; th += 16) {
        float acc[16][2];
#pragma unroll
        for (int t = 0; t < 16; ++t) acc[t][0] = acc[t][1] = 0.f;
#pragma unroll
        for (int r4 = 0; r4 < RPT / 4; ++r4) {
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            float4 kk = *reinterpret_cast<const float4 *>(Kc + (th + t) * DK + i0 + 4 * r4);
            if (KDA && th + t > 0) {
              const float4 g = *reinterpret_cast<const float4 *>(Gc + (th + t - 1) * DK + i0 + 4 * r4);
              kk = make_float4(kk.x * g.x, kk.y * g.y, kk.z * g.z, kk.w * g.w);
            }
#pragma unroll
            for (int c = 0; c < 2; ++c)
              acc[t][c] = fmaf(kk.x, st[4 * r4][c], fmaf(kk.y, st[4 * r4 + 1][c],
                               fmaf(kk.z, st[4 * r4 + 2][c], fmaf(kk.w, st[4 * r4 + 3][c], acc[t][c]))));
          }
        }
#pragma unroll
        for (int t = 0; t < 16; ++t) {
          const float sc = KDA ? 1.f : Gi[th + t];
          *reinterpret_cast<float2 *>(Pp + (q * C + th + t) * DV + j2) = make_float2(acc[t][0] * sc, acc[t][1] * sc);
        }
      }
      __syncthreads();
      if (tid < DV) {
        // the triangular solve, one column j per thread, with the chunk's solution in
        // registers (fully unrolled: row t's sum runs as soon as its terms are ready)
        if (KDA) {
          // x_t = -beta_t (P_t + sum_{r<t} E[t][r] y_r + sum_{r<t} Cm[t][r] x_r), y_r = beta_r v_r;
          // x_t goes into slice 0 of P, y_t into V
          float x[C], y[C];
#pragma unroll
          for (int t = 0; t < C; ++t) {
            float p = 0.f;
#pragma unroll
            for (int qq = 0; qq < NQ; ++qq) p += Pp[(qq * C + t) * DV + j];
            y[t] = Bc[t] * Vc[t * DV + j];
#pragma unroll
            for (int r = 0; r < t; ++r) p = fmaf(Em[t * (C + 1) + r], y[r], fmaf(Am[t * (C + 1) + r], x[r], p));
            x[t] = -Bc[t] * p;
          }
#pragma unroll
          for (int t = 0; t < C; ++t) {
            Pp[t * DV + j] = x[t];
            Vc[t * DV + j] = y[t];
          }
        } else {
          // u_t = beta_t (v_t - P_t) - sum_{r<t} A[t][r] u_r, then the weight gamma_C / gamma_t
          float u[C];
#pragma unroll
          for (int t = 0; t < C; ++t) {
            float p = 0.f;
#pragma unroll
            for (int qq = 0; qq < NQ; ++qq) p += Pp[(qq * C + t) * DV + j];
            float acc = Bc[t] * (Vc[t * DV + j] - p);
#pragma unroll
            for (int r = 0; r < t; ++r) acc = fmaf(-Am[t * (C + 1) + r], u[r], acc);
            u[t] = acc;
          }
          const float gC = Gi[C - 1];
#pragma unroll
          for (int t = 0; t < C; ++t) Vc[t * DV + j] = u[t] * (gC / Gi[t]);
        }
      } else if (KDA) {
        // meanwhile the update weights: gamma_C / gm_r * k_r (into G) and gamma_C / gamma_r * k_r (into K)
        for (int idx = tid - DV; idx < C * DK; idx += 256 - DV) {
          const int r = idx / DK, i = idx % DK;
          const float k = Kc[idx], g = gCr[i];
          Gc[idx] = k * g * (r > 0 ? Gi[idx - DK] : 1.f);
          Kc[idx] = k * g * Gi[idx];
        }
      }
    } else {
      // Mamba-2: u_t = (gamma_C / gamma_t) dt_t x_t = exp(log gamma_C - log gamma_t) dt_t x_t
      const float lC = Gi[C - 1];
      for (int idx = tid; idx < C * DV; idx += 256) {
        const int t = idx / DV;
        Vc[idx] *= Gc[t] * expf(lC - Gi[t]);
      }
    }
    __syncthreads();
    // ---- S_C = Gamma_C S_0 + sum_t (weights_t) (x) (U or x, y)_t over my rows ---------------------
    {
#pragma unroll
      for (int r = 0; r < RPT; ++r) {
        const float g = KDA ? gCr[i0 + r] : (M2 ? expf(Gi[C - 1]) : Gi[C - 1]);
        st[r][0] *= g;
        st[r][1] *= g;
      }
      for (int t = 0; t < C; ++t) {
        const float2 u = *reinterpret_cast<const float2 *>(Vc + t * DV + j2);
        const float2 x = KDA ? *reinterpret_cast<const float2 *>(Pp + t * DV + j2) : make_float2(0.f, 0.f);
#pragma unroll
        for (int r4 = 0; r4 < RPT / 4; ++r4) {
          const float4 kk = *reinterpret_cast<const float4 *>(Kc + t * DK + i0 + 4 * r4);
          const float ks[4] = {kk.x, kk.y, kk.z, kk.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            st[4 * r4 + e][0] = fmaf(ks[e], u.x, st[4 * r4 + e][0]);
            st[4 * r4 + e][1] = fmaf(ks[e], u.y, st[4 * r4 + e][1]);
          }
          if (KDA) {
            const float4 k1 = *reinterpret_cast<const float4 *>(Gc + t * DK + i0 + 4 * r4);
            const float k1s[4] = {k1.x, k1.y, k1.z, k1.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              st[4 * r4 + e][0] = fmaf(k1s[e], x.x, st[4 * r4 + e][0]);
              st[4 * r4 + e][1] = fmaf(k1s[e], x.y, st[4 * r4 + e][1]);
            }
          }
        }
      }
    }
    __syncthreads();  // the chunk's buffers are free
  }
  float *out = S_out + (int64_t)blockIdx.x * DK * DV;
#pragma unroll
  for (int r = 0; r < RPT; ++r)
    *reinterpret_cast<float2 *>(out + (int64_t)(i0 + r) * DV + j2) = make_float2(st[r][0], st[r][1]);
}

static int check_workload(const seed_synth_workload *w) {
  if (!w) return SEED_ERR_INVALID_ARG;
  if (w->variant < SEED_GDN || w->variant > SEED_MAMBA2) return SEED_ERR_INVALID_ARG;
  if (w->n_req < 0 || w->n_layers <= 0 || w->n_head <= 0) return SEED_ERR_INVALID_ARG;
  if (w->d_k != kDK || (w->d_v != 64 && w->d_v != 128)) return SEED_ERR_UNSUPPORTED_SHAPE;
  if (w->rank <= 0 && (w->n_rank_choices <= 0 || w->n_rank_choices > 4)) return SEED_ERR_INVALID_ARG;
  if (w->prefill_len <= 0 && (w->prefill_lo < 0 || w->prefill_hi < w->prefill_lo)) return SEED_ERR_INVALID_ARG;
  return SEED_OK;
}

}  // namespace seedk

using namespace seedk;

static inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? SEED_OK : SEED_ERR_CUDA; }

extern "C" int seed_synth_raw(uint32_t seed, int32_t phase, int32_t field, uint32_t time,
                              uint32_t entity0, int32_t n_entities, int32_t n_blocks, uint32_t *out,
                              seed_stream_t stream) {
  if (n_entities < 0 || n_blocks < 0) return SEED_ERR_INVALID_ARG;
  if ((int64_t)n_entities * n_blocks == 0) return SEED_OK;
  if (!out) return SEED_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(out) % 16) return SEED_ERR_ALIGNMENT;
  const int64_t n = (int64_t)n_entities * n_blocks;
  raw_kernel<<<(unsigned)((n + 255) / 256), 256, 0, (cudaStream_t)stream>>>(
      seed, phase, field, time, entity0, n_entities, n_blocks, out);
  return cuda_status(cudaGetLastError());
}

extern "C" int seed_synth_constants(const seed_synth_workload *w, float *vbar, float *sink_scale,
                                    float *A, int32_t *rank, int32_t *prompt_len,
                                    seed_stream_t stream) {
  const int c = check_workload(w);
  if (c) return c;
  if (vbar && reinterpret_cast<uintptr_t>(vbar) % 16) return SEED_ERR_ALIGNMENT;
  constants_kernel<<<1184, 256, 0, (cudaStream_t)stream>>>(*w, vbar, sink_scale, A, rank, prompt_len);
  return cuda_status(cudaGetLastError());
}

extern "C" int seed_synth_step_inputs(const seed_synth_workload *w, int32_t phase, int32_t time,
                                      int64_t head0, int32_t n_heads, const float *vbar,
                                      const float *sink_scale, float *q, float *k, float *v,
                                      float *gate, float *beta, seed_stream_t stream) {
  const int c = check_workload(w);
  if (c) return c;
  if (n_heads < 0 || head0 < 0) return SEED_ERR_INVALID_ARG;
  if (n_heads == 0) return SEED_OK;
  if (!vbar || !sink_scale || !q || !k || !v || !gate) return SEED_ERR_INVALID_ARG;
  if (w->variant != SEED_MAMBA2 && !beta) return SEED_ERR_INVALID_ARG;
  for (const void *ptr : {(const void *)vbar, (const void *)q, (const void *)k, (const void *)v,
                          (const void *)gate})
    if (reinterpret_cast<uintptr_t>(ptr) % 16) return SEED_ERR_ALIGNMENT;
  step_inputs_kernel<<<n_heads, 128, 0, (cudaStream_t)stream>>>(*w, phase, time, head0, vbar,
                                                                sink_scale, q, k, v, gate, beta);
  return cuda_status(cudaGetLastError());
}

template <int VAR, int DV>
static cudaError_t launch_chunk_t(const seed_synth_workload &w, int64_t head0, int32_t n_heads, const int32_t *plen,
                                  const float *vbar, const float *sink, const float *A, float *S_out,
                                  cudaStream_t s) {
  const int bytes = ChunkSmem<VAR, DV>::FLOATS * 4;
  auto kern = prefill_chunk_kernel<VAR, DV>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  kern<<<n_heads, 256, bytes, s>>>(w, head0, plen, vbar, sink, A, S_out);
  return cudaGetLastError();
}

extern "C" int seed_synth_dense_prefill(const seed_synth_workload *w, int64_t head0, int32_t n_heads,
                                        const int32_t *prompt_len, const float *vbar,
                                        const float *sink_scale, const float *A, float *S_out,
                                        seed_stream_t stream) {
  const int c = check_workload(w);
  if (c) return c;
  if (n_heads < 0 || head0 < 0) return SEED_ERR_INVALID_ARG;
  if (n_heads == 0) return SEED_OK;
  if (!prompt_len || !vbar || !sink_scale || !S_out) return SEED_ERR_INVALID_ARG;
  if (w->variant == SEED_MAMBA2 && !A) return SEED_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(S_out) % 16 || reinterpret_cast<uintptr_t>(vbar) % 16)
    return SEED_ERR_ALIGNMENT;
  cudaStream_t s = (cudaStream_t)stream;
  const bool d64 = w->d_v == 64;
  switch (w->variant) {
    case SEED_GDN:
      if (d64) prefill_kernel<SEED_GDN, 64><<<n_heads, 256, 0, s>>>(*w, head0, prompt_len, vbar, sink_scale, A, S_out);
      else prefill_kernel<SEED_GDN, 128><<<n_heads, 256, 0, s>>>(*w, head0, prompt_len, vbar, sink_scale, A, S_out);
      break;
    case SEED_KDA:
      if (d64) prefill_kernel<SEED_KDA, 64><<<n_heads, 256, 0, s>>>(*w, head0, prompt_len, vbar, sink_scale, A, S_out);
      else prefill_kernel<SEED_KDA, 128><<<n_heads, 256, 0, s>>>(*w, head0, prompt_len, vbar, sink_scale, A, S_out);
      break;
    default:
      if (d64) prefill_kernel<SEED_MAMBA2, 64><<<n_heads, 256, 0, s>>>(*w, head0, prompt_len, vbar, sink_scale, A, S_out);
      else prefill_kernel<SEED_MAMBA2, 128><<<n_heads, 256, 0, s>>>(*w, head0, prompt_len, vbar, sink_scale, A, S_out);
      break;
  }
  return cuda_status(cudaGetLastError());
}

extern "C" int seed_synth_dense_prefill_chunked(const seed_synth_workload *w, int64_t head0, int32_t n_heads,
                                                const int32_t *prompt_len, const float *vbar,
                                                const float *sink_scale, const float *A, float *S_out,
                                                seed_stream_t stream) {
  // The delta-rule chunks divide by cumulative gate products; where the smallest
  // gate raised to the chunk length could leave fp32's normal range, the
  // token-serial kernel (the same result) runs instead.
  if (w && w->variant != SEED_MAMBA2) {
    const int clen = w->variant == SEED_KDA ? chunk_len<SEED_KDA>() : chunk_len<SEED_GDN>();
    if (!(w->alpha_lo > 0.f) || (double)clen * log2((double)w->alpha_lo) < -96.0)
      return seed_synth_dense_prefill(w, head0, n_heads, prompt_len, vbar, sink_scale, A, S_out, stream);
  }
  const int c = check_workload(w);
  if (c) return c;
  if (n_heads < 0 || head0 < 0) return SEED_ERR_INVALID_ARG;
  if (n_heads == 0) return SEED_OK;
  if (!prompt_len || !vbar || !sink_scale || !S_out) return SEED_ERR_INVALID_ARG;
  if (w->variant == SEED_MAMBA2 && !A) return SEED_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(S_out) % 16 || reinterpret_cast<uintptr_t>(vbar) % 16)
    return SEED_ERR_ALIGNMENT;
  cudaStream_t s = (cudaStream_t)stream;
  const bool d64 = w->d_v == 64;
  cudaError_t e;
  switch (w->variant) {
    case SEED_GDN:
      e = d64 ? launch_chunk_t<SEED_GDN, 64>(*w, head0, n_heads, prompt_len, vbar, sink_scale, A, S_out, s)
              : launch_chunk_t<SEED_GDN, 128>(*w, head0, n_heads, prompt_len, vbar, sink_scale, A, S_out, s);
      break;
    case SEED_KDA:
      e = d64 ? launch_chunk_t<SEED_KDA, 64>(*w, head0, n_heads, prompt_len, vbar, sink_scale, A, S_out, s)
              : launch_chunk_t<SEED_KDA, 128>(*w, head0, n_heads, prompt_len, vbar, sink_scale, A, S_out, s);
      break;
    default:
      e = d64 ? launch_chunk_t<SEED_MAMBA2, 64>(*w, head0, n_heads, prompt_len, vbar, sink_scale, A, S_out, s)
              : launch_chunk_t<SEED_MAMBA2, 128>(*w, head0, n_heads, prompt_len, vbar, sink_scale, A, S_out, s);
      break;
  }
  return cuda_status(e);
}
