// Compression of factors (every T steps) and of dense states (end of prefill).
//
// "Shallow Encoding Emits Deep Memories", thelatestinai.com list view, Table 1:
// the states that leave the prefill are compressed to the sink plus rank-R
// factors, and the decode compresses back to rank R every W steps.  picx.dev
// summary, Theoretical and Practical Implications > Lemma 1: the sink split
// a = S vbar / |vbar|^2, C = S - a vbar^T, never recomputed afterwards.
//
// recompress (one CTA of 128 threads per head):
//   A = U_eff, B = W (fp32 in shared memory, column-major, padded columns)
//   Householder QR of A and of B, concurrently in two 64-thread teams
//   K = R_a R_b^T (m x m)
//   one-sided Jacobi SVD of K: rotate pairs of columns of K until every pair
//     is orthogonal; then K J = X Sigma, K = X Sigma J^T
//   order columns by |K_j| (= sigma_j), keep the rank(h) largest
//   Q_a, Q_b formed in place from the reflectors
//   U_new = Q_a X_r,  W_new = Q_b K^T X_r = Q_b Y_r Sigma_r   (X_r: normalised
//   kept columns of K J; the singular values go with W, and K^T X_r is the
//   projection of the core onto the kept directions, so no rotation is kept)
// compress_dense (one CTA of 256 threads per head): the same with A = C and
// B = I (so K = R_a and W_new = R_a^T X_r).
//
// The arithmetic is fp32 FMA: the QR and Jacobi steps are sequences of small
// dependent reductions that do not map onto tensor-core tiles.
#include "common.cuh"

#include <float.h>

namespace seedk {

constexpr int kMaxSweeps = 30;
// After the core is scaled to a largest entry in [1/2, 1), a column whose squared
// norm is below this is under fp32 resolution of the largest one: rotating it only
// stirs rounding noise, so it is left alone (its singular value is negligible).
constexpr float kNegligible = 1e-14f;

struct CompressArgs {
  StateView sv;
  float *trunc_err;
  int32_t *sweeps;  // Jacobi sweeps per head (or -1: limit reached), optional
  const float *S;   // dense input (compress_dense) or nullptr (recompress)
  int m_max;        // smem sizing: largest column count of any head
  int cs_alloc;     // column stride of the core buffers in the allocation
};

// x . y over rows [i0, nrows) of two columns (16-byte aligned column starts,
// nrows a multiple of 4): scalar head up to a multiple of 4, then float4 body.
__device__ static inline float col_dot(const float *__restrict__ x, const float *__restrict__ y, int i0,
                                       int nrows) {
  float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
  int i = i0;
  for (; (i & 3) && i < nrows; ++i) s0 = fmaf(x[i], y[i], s0);
  for (; i < nrows; i += 4) {
    const float4 a = *reinterpret_cast<const float4 *>(x + i);
    const float4 b = *reinterpret_cast<const float4 *>(y + i);
    s0 = fmaf(a.x, b.x, s0); s1 = fmaf(a.y, b.y, s1); s2 = fmaf(a.z, b.z, s2); s3 = fmaf(a.w, b.w, s3);
  }
  return (s0 + s1) + (s2 + s3);
}
// y[i] -= a x[i] over rows [i0, nrows), same layout rules.
__device__ static inline void col_axpy(float a, const float *__restrict__ x, float *__restrict__ y, int i0,
                                       int nrows) {
  int i = i0;
  for (; (i & 3) && i < nrows; ++i) y[i] = fmaf(-a, x[i], y[i]);
  for (; i < nrows; i += 4) {
    const float4 b = *reinterpret_cast<const float4 *>(x + i);
    float4 c = *reinterpret_cast<const float4 *>(y + i);
    c.x = fmaf(-a, b.x, c.x); c.y = fmaf(-a, b.y, c.y); c.z = fmaf(-a, b.z, c.z); c.w = fmaf(-a, b.w, c.w);
    *reinterpret_cast<float4 *>(y + i) = c;
  }
}

// Householder QR in place on a column-major nrows x ncols panel (leading
// dimension ld, a multiple of 4; nrows a multiple of 4).  On exit the upper
// triangle holds R; below the diagonal of column j sits the reflector's vector
// v_j (v_j[j] = 1 implicit), tau[j] its coefficient: H_j = I - tau_j v_j v_j^T,
// A = H_0 H_1 ... H_{n-1} R.  Each reflector is formed from the column scaled
// by its largest magnitude, so that columns far below 1 (long products of
// gates) do not underflow in their squared norm: an inaccurate norm would give
// a reflector that is not orthogonal, which then corrupts the larger columns
// it is applied to.  Columns below the smallest normal float are treated as zero.
__device__ static void householder_qr(float *A, int ld, int nrows, int ncols, float *tau,
                                      int ttid, int tsize, int bar) {
  const int lane = ttid & 31;
  const int nref = ncols < nrows ? ncols : nrows;
  for (int j = 0; j < nref; ++j) {
    float *cj = A + j * ld;
    if (ttid < 32) {
      float amax = 0.f;
      for (int i = j + lane; i < nrows; i += 32) amax = fmaxf(amax, fabsf(cj[i]));
      amax = warp_max(amax);
      const float alpha = cj[j];
      float tj = 0.f, beta = alpha;
      if (amax >= FLT_MIN) {
        const float inv = 1.f / amax;
        float ss = 0.f;
        for (int i = j + 1 + lane; i < nrows; i += 32) {
          const float x = cj[i] * inv;
          ss = fmaf(x, x, ss);
        }
        ss = warp_sum(ss);
        if (ss > 0.f) {
          const float as = alpha * inv;
          const float nrm = sqrtf(fmaf(as, as, ss));
          const float bs = as >= 0.f ? -nrm : nrm;
          tj = (bs - as) / bs;
          const float sc = 1.f / ((as - bs) * amax);  // v_i = x_i / (alpha - beta), |v_i| <= 1
          for (int i = j + 1 + lane; i < nrows; i += 32) cj[i] *= sc;
          beta = bs * amax;
        }
      } else {
        for (int i = j + 1 + lane; i < nrows; i += 32) cj[i] = 0.f;
      }
      __syncwarp();
      if (lane == 0) { cj[j] = beta; tau[j] = tj; }
    }
    team_sync(bar, tsize);
    const float tj = tau[j];
    if (tj != 0.f) {
      for (int l = j + 1 + ttid; l < ncols; l += tsize) {
        float *cl = A + l * ld;
        const float sv = tj * (cl[j] + col_dot(cj, cl, j + 1, nrows));
        cl[j] -= sv;
        col_axpy(sv, cj, cl, j + 1, nrows);
      }
    }
    team_sync(bar, tsize);
  }
}

// Overwrite the reflectors with the first ncols columns of Q = H_0 ... H_{n-1}.
__device__ static void form_q(float *A, int ld, int nrows, int ncols, const float *tau, int ttid,
                              int tsize, int bar) {
  for (int j = ncols - 1; j >= 0; --j) {
    const float *cj = A + j * ld;
    const float tj = tau[j];
    if (tj != 0.f) {
      for (int l = j + 1 + ttid; l < ncols; l += tsize) {
        float *cl = A + l * ld;  // rows < l of a finished column are zero, so cl[j] == 0
        const float sv = tj * col_dot(cj, cl, j + 1, nrows);
        cl[j] = -sv;
        col_axpy(sv, cj, cl, j + 1, nrows);
      }
    }
    team_sync(bar, tsize);
    float *cw = A + j * ld;
    for (int i = ttid; i < nrows; i += tsize) {
      if (i < j) cw[i] = 0.f;
      else if (i == j) cw[i] = 1.f - tj;
      else cw[i] = -tj * cw[i];
    }
    team_sync(bar, tsize);
  }
}

// Geometry of the core K (n x n) in shared memory for the Jacobi rounds: the
// threads of a column pair own contiguous chunks of R = ld / tpp rows (R a
// multiple of 4, rows n..ld-1 are zero), columns are cs = ld + 4 floats apart
// so that 16-byte accesses of different columns spread over the banks.
struct JacobiGeom {
  int tpp, ld, cs;
};
__host__ __device__ inline JacobiGeom jacobi_geom(int n, int nthreads) {
  const int P = (n + 1) / 2 > 0 ? (n + 1) / 2 : 1;
  const int n4 = (n + 3) & ~3;
  int tpp = 1;
  while (tpp * 2 * P <= nthreads && tpp < 32 && 8 * tpp <= n4) tpp *= 2;
  const int ld = (n + 4 * tpp - 1) / (4 * tpp) * (4 * tpp);
  return JacobiGeom{tpp, ld, ld + 4};
}
__host__ inline int jacobi_cs_alloc(int m_max, int nthreads) {
  int cs = 4;
  for (int n = 0; n <= m_max; ++n) {
    const int c = jacobi_geom(n, nthreads).cs;
    cs = c > cs ? c : cs;
  }
  return cs;
}

// One-sided (Hestenes) Jacobi on the n columns of K: rotate pairs of columns
// until every pair is orthogonal, K <- K J, so that the columns of K J are
// X Sigma.  The rotations J are not kept: the rebuild uses the original core.
// Round-robin pair order: n' = n rounded up to even seats, seat 0 fixed, the
// others move one seat each round; pair i joins seats i and n'-1-i.  A pair is
// rotated when |k_p . k_q| > tol |k_p| |k_q| and both columns are above fp32
// resolution of the core (scaled to a largest entry in [1/2, 1)).  Each thread
// keeps its chunk of both columns in registers through a round.  Whole block.
// Returns the number of sweeps, or -1 if the sweep limit was reached.
template <int NT, int RMAX>
__device__ static int jacobi_svd(float *K, int n, const JacobiGeom &g, float tol) {
  if (n < 2) return 0;
  const int tid = threadIdx.x;
  const int nn = n + (n & 1);
  const int P = nn / 2;
  const int tpp = g.tpp, cs = g.cs;
  const int R = g.ld / tpp, R4 = R / 4;
  const int pair = tid / tpp, sub = tid % tpp;
  const bool active = pair < P;
  for (int sweep = 0; sweep < kMaxSweeps; ++sweep) {
    int rotated = 0;
    for (int round = 0; round < nn - 1; ++round) {
      int p = 0, q = 0;
      if (active) {
        const int sp = pair, sq = nn - 1 - pair;
        p = sp == 0 ? 0 : 1 + (sp - 1 + round) % (nn - 1);
        q = 1 + (sq - 1 + round) % (nn - 1);
      }
      const bool real = active && p < n && q < n;
      float4 xp[RMAX / 4], xq[RMAX / 4];
      float al = 0.f, be = 0.f, ga = 0.f;
      float4 *kp = reinterpret_cast<float4 *>(K + p * cs + sub * R);
      float4 *kq = reinterpret_cast<float4 *>(K + q * cs + sub * R);
      if (real) {
#pragma unroll
        for (int v = 0; v < RMAX / 4; ++v) {
          if (v < R4) {
            xp[v] = kp[v];
            xq[v] = kq[v];
            al = fmaf(xp[v].x, xp[v].x, fmaf(xp[v].y, xp[v].y, fmaf(xp[v].z, xp[v].z, fmaf(xp[v].w, xp[v].w, al))));
            be = fmaf(xq[v].x, xq[v].x, fmaf(xq[v].y, xq[v].y, fmaf(xq[v].z, xq[v].z, fmaf(xq[v].w, xq[v].w, be))));
            ga = fmaf(xp[v].x, xq[v].x, fmaf(xp[v].y, xq[v].y, fmaf(xp[v].z, xq[v].z, fmaf(xp[v].w, xq[v].w, ga))));
          }
        }
      }
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        if (o < tpp) {
          al += __shfl_xor_sync(0xffffffffu, al, o);
          be += __shfl_xor_sync(0xffffffffu, be, o);
          ga += __shfl_xor_sync(0xffffffffu, ga, o);
        }
      }
      if (real && al > kNegligible && be > kNegligible && fabsf(ga) > tol * sqrtf(al) * sqrtf(be)) {
        // Any t gives an exact rotation (c^2 + s^2 = 1 to rounding), so the angle
        // may use fast reciprocals; |zeta| large (tiny ga) gives t ~ 1/(2 zeta).
        const float zeta = (be - al) * __frcp_rn(2.f * ga);
        const float az = fabsf(zeta);
        const float root = az < 1e18f ? az + fmaf(az, az, 1.f) * rsqrtf(fmaf(az, az, 1.f)) : 2.f * az;
        const float t = copysignf(__frcp_rn(root), zeta);
        const float c = rsqrtf(fmaf(t, t, 1.f));
        const float s = c * t;
#pragma unroll
        for (int v = 0; v < RMAX / 4; ++v) {
          if (v < R4) {
            const float4 a = xp[v], b = xq[v];
            kp[v] = make_float4(fmaf(c, a.x, -s * b.x), fmaf(c, a.y, -s * b.y), fmaf(c, a.z, -s * b.z),
                                fmaf(c, a.w, -s * b.w));
            kq[v] = make_float4(fmaf(s, a.x, c * b.x), fmaf(s, a.y, c * b.y), fmaf(s, a.z, c * b.z),
                                fmaf(s, a.w, c * b.w));
          }
        }
        rotated = 1;
      }
      __syncthreads();
    }
    if (!__syncthreads_or(rotated)) return sweep + 1;
  }
  return -1;
}

// Dynamic shared-memory layout of the compression kernels (offsets in floats,
// multiples of 4).
struct Smem {
  int lda, ldb;
  int offA, offB, offK, offK0, offTa, offTb, offS, offI, offO, offR;
  int total_floats;
  __host__ __device__ Smem(int m, int dk, int dv, bool dense, int cs) {
    lda = dk + 4;  // 16-byte aligned columns, 4 banks apart
    ldb = dv + 4;
    auto up4 = [](int x) { return (x + 3) & ~3; };
    offA = 0;
    offB = up4(offA + m * lda);
    offK = up4(offB + (dense ? 0 : m * ldb));
    offK0 = up4(offK + m * cs);
    offTa = up4(offK0 + m * cs);
    offTb = offTa + up4(m);
    offS = offTb + up4(m);
    offI = offS + up4(m);
    offO = offI + up4(m);
    offR = offO + up4(m);     // 8 floats of reduction scratch
    total_floats = offR + 8;
  }
};

template <int VAR, typename TF, int DV, bool DENSE>
__global__ void __launch_bounds__(DENSE ? 256 : 128) compress_kernel(const CompressArgs p) {
  constexpr int DK = kDK;
  constexpr int NT = DENSE ? 256 : 128;
  constexpr int RMAX = DENSE ? 32 : 16;
  extern __shared__ __align__(16) float smem[];
  const int h = blockIdx.x;
  const int tid = threadIdx.x;
  const StateView &sv = p.sv;
  const int r = sv.rank_of(h);
  const int m = DENSE ? DV : r + sv.growth * sv.steps;
  if (r < 0 || (!DENSE && m > p.m_max)) {  // rank table disagrees with r_max: touch nothing
    if (tid == 0 && sv.status) sv.status[h] = SEED_ERR_INVALID_ARG;
    return;
  }
  const int64_t c0 = sv.col0(h);
  const Smem L(DENSE ? DV : p.m_max, DK, DV, DENSE, p.cs_alloc);
  const JacobiGeom jg = jacobi_geom(m, NT);
  const int cs = jg.cs, ldr = jg.ld;
  float *A = smem + L.offA, *B = smem + L.offB, *K = smem + L.offK, *K0 = smem + L.offK0;
  float *tauA = smem + L.offTa, *tauB = smem + L.offTb, *sig2 = smem + L.offS, *inv = smem + L.offI;
  int *order = reinterpret_cast<int *>(smem + L.offO);
  float *red = smem + L.offR;
  const int lda = L.lda, ldb = L.ldb;
  TF *Uh = reinterpret_cast<TF *>(sv.U) + c0 * DK;
  TF *Wh = reinterpret_cast<TF *>(sv.W) + c0 * DV;

  // ---- load -------------------------------------------------------------------
  if (DENSE) {
    // A[j][i] = S[i][j]; then a = S vbar / |vbar|^2 and C = S - a vbar^T in place
    const float *Sh = p.S + (int64_t)h * DK * DV;
    for (int idx = tid; idx < DK * DV; idx += NT) {
      const int i = idx / DV, j = idx % DV;
      A[j * lda + i] = Sh[idx];
    }
    __syncthreads();
    const float *vb = sv.vbar + (int64_t)sv.dir_of(h) * DV;
    float vv = 0.f;
    for (int j = 0; j < DV; ++j) vv = fmaf(vb[j], vb[j], vv);
    if (tid < DK) {
      float acc = 0.f;
      for (int j = 0; j < DV; ++j) acc = fmaf(A[j * lda + tid], vb[j], acc);
      const float ai = acc / vv;
      sv.a[(int64_t)h * DK + tid] = ai;
      for (int j = 0; j < DV; ++j) A[j * lda + tid] = fmaf(-ai, vb[j], A[j * lda + tid]);
    }
  } else {
    for (int idx = tid; idx < m * DK; idx += NT) {
      const int j = idx / DK, i = idx % DK;
      const float u = Elem<TF>::load(Uh + idx);
      const float f = VAR == SEED_KDA ? sv.scale[(int64_t)h * DK + i] : sv.scale[c0 + j];
      A[j * lda + i] = u * f;
    }
    for (int idx = tid; idx < m * DV; idx += NT) {
      const int j = idx / DV, i = idx % DV;
      B[j * ldb + i] = Elem<TF>::load(Wh + idx);
    }
  }
  __syncthreads();

  // ---- QR ---------------------------------------------------------------------
  if (DENSE) {
    householder_qr(A, lda, DK, m, tauA, tid, NT, 1);
  } else {
    const int team = tid / 64, ttid = tid % 64;
    if (team == 0) householder_qr(A, lda, DK, m, tauA, ttid, 64, 1);
    else householder_qr(B, ldb, DV, m, tauB, ttid, 64, 2);
  }
  __syncthreads();

  // ---- core K = R_a R_b^T (or R_a), rows padded with zeros to ld; K0 keeps a copy --------
  for (int idx = tid; idx < m * ldr; idx += NT) {
    const int j = idx / ldr, i = idx % ldr;  // K[j][i]: column j, row i
    float acc = 0.f;
    if (i < m) {
      if (DENSE) {
        acc = i <= j ? A[j * lda + i] : 0.f;
      } else {
        for (int l = max(i, j); l < m; ++l) acc = fmaf(A[l * lda + i], B[l * ldb + j], acc);
      }
    }
    K[j * cs + i] = acc;
    K0[j * cs + i] = acc;
  }
  __syncthreads();

  // ---- Q factors in place -----------------------------------------------------------
  if (DENSE) {
    form_q(A, lda, DK, m, tauA, tid, NT, 1);
  } else {
    const int team = tid / 64, ttid = tid % 64;
    if (team == 0) form_q(A, lda, DK, m, tauA, ttid, 64, 1);
    else form_q(B, ldb, DV, m, tauB, ttid, 64, 2);
  }

  // ---- SVD of the core, scaled by a power of two to a largest entry in [1/2, 1) ----------
  float kmax = 0.f;
  for (int idx = tid; idx < m * ldr; idx += NT) kmax = fmaxf(kmax, fabsf(K[(idx / ldr) * cs + idx % ldr]));
  kmax = warp_max(kmax);
  if ((tid & 31) == 0) red[tid >> 5] = kmax;
  __syncthreads();
  kmax = 0.f;
  for (int w = 0; w < NT / 32; ++w) kmax = fmaxf(kmax, red[w]);
  int kexp = 0;
  if (kmax > 0.f) frexpf(kmax, &kexp);
  const float kscale = ldexpf(1.f, -kexp), kunscale = ldexpf(1.f, kexp);
  for (int idx = tid; idx < m * ldr; idx += NT) K[(idx / ldr) * cs + idx % ldr] *= kscale;
  __syncthreads();
  const float tol = sizeof(TF) == 2 ? 1e-5f : (float)(m > 16 ? m : 16) * FLT_EPSILON;
  const int sweeps = jacobi_svd<NT, RMAX>(K, m, jg, tol);

  // ---- order by sigma, truncation error -----------------------------------------------
  for (int j = tid; j < m; j += NT) {
    float acc = 0.f;
    for (int i = 0; i < m; ++i) acc = fmaf(K[j * cs + i], K[j * cs + i], acc);
    sig2[j] = acc;
    inv[j] = acc > kNegligible ? rsqrtf(acc) : 0.f;  // x_j = (K J)_j / sigma_j
  }
  __syncthreads();
  for (int j = tid; j < m; j += NT) {
    int rank = 0;
    const float sj = sig2[j];
    for (int i = 0; i < m; ++i) {
      const float si = sig2[i];
      rank += (si > sj) || (si == sj && i < j);
    }
    order[rank] = j;
  }
  __syncthreads();
  if (tid == 0) {
    float e = 0.f;
    for (int k = r; k < m; ++k) e += sig2[order[k]];
    if (p.trunc_err) p.trunc_err[h] = sqrtf(e) * kunscale;
    if (p.sweeps) p.sweeps[h] = sweeps;
    if (sv.status) sv.status[h] = sweeps < 0 ? SEED_ERR_NOT_CONVERGED : SEED_OK;
  }

  // ---- rebuild the kept columns: U = Q_a X_r,  W = Q_b K0^T X_r ----------------------------
  const int rk = r < m ? r : m;
  if (tid < DK) {
    for (int k = 0; k < rk; ++k) {
      const int col = order[k];
      const float *z = K + col * cs;
      float acc = 0.f;
      for (int l = 0; l < m; ++l) acc = fmaf(A[l * lda + tid], z[l], acc);
      Elem<TF>::store(Uh + (int64_t)k * DK + tid, acc * inv[col]);
    }
  }
  if (DENSE) {
    // Q_b = I: W[:, k] = K0^T x_k
    for (int i = tid; i < DV; i += NT) {
      for (int k = 0; k < rk; ++k) {
        const int col = order[k];
        const float *z = K + col * cs;
        float acc = 0.f;
        for (int l = 0; l < m; ++l) acc = fmaf(K0[i * cs + l], z[l], acc);
        Elem<TF>::store(Wh + (int64_t)k * DV + i, acc * inv[col]);
      }
    }
  } else {
    __syncthreads();  // A (Q_a) is no longer needed: Y = K0^T X_r goes there
    float *Y = A;
    for (int idx = tid; idx < rk * m; idx += NT) {
      const int k = idx / m, l = idx % m;
      const int col = order[k];
      const float *z = K + col * cs;
      float acc = 0.f;
      for (int i = 0; i < m; ++i) acc = fmaf(K0[l * cs + i], z[i], acc);
      Y[k * cs + l] = acc * inv[col];
    }
    __syncthreads();
    if (tid < DV) {
      for (int k = 0; k < rk; ++k) {
        float acc = 0.f;
        for (int l = 0; l < m; ++l) acc = fmaf(B[l * ldb + tid], Y[k * cs + l], acc);
        Elem<TF>::store(Wh + (int64_t)k * DV + tid, acc);
      }
    }
  }
  if (VAR == SEED_KDA) {
    for (int i = tid; i < DK; i += NT) sv.scale[(int64_t)h * DK + i] = 1.f;
  } else {
    for (int k = tid; k < rk; k += NT) sv.scale[c0 + k] = 1.f;
  }
}

template <int VAR, typename TF, int DV, bool DENSE>
static cudaError_t launch_compress_t(const CompressArgs &a, cudaStream_t s) {
  CompressArgs args = a;
  const int m_alloc = DENSE ? DV : a.m_max;
  args.cs_alloc = jacobi_cs_alloc(m_alloc, DENSE ? 256 : 128);
  const Smem L(m_alloc, kDK, DV, DENSE, args.cs_alloc);
  const size_t bytes = (size_t)L.total_floats * sizeof(float);
  auto kern = compress_kernel<VAR, TF, DV, DENSE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  kern<<<a.sv.n_heads, DENSE ? 256 : 128, bytes, s>>>(args);
  return cudaGetLastError();
}

template <int VAR, typename TF, bool DENSE>
static cudaError_t launch_compress_d(const CompressArgs &a, cudaStream_t s) {
  if (a.sv.d_v == 64) return launch_compress_t<VAR, TF, 64, DENSE>(a, s);
  return launch_compress_t<VAR, TF, 128, DENSE>(a, s);
}

template <typename TF, bool DENSE>
static cudaError_t launch_compress_v(const CompressArgs &a, cudaStream_t s) {
  // Only the scale layout differs between variants here.
  if (a.sv.variant == SEED_KDA) return launch_compress_d<SEED_KDA, TF, DENSE>(a, s);
  return launch_compress_d<SEED_GDN, TF, DENSE>(a, s);
}

cudaError_t launch_recompress(const StateView &sv, int factor_dtype, float *trunc_err,
                              int32_t *sweeps, int m_max, cudaStream_t s) {
  CompressArgs a{sv, trunc_err, sweeps, nullptr, m_max, 0};
  if (factor_dtype == SEED_BF16) return launch_compress_v<__nv_bfloat16, false>(a, s);
  return launch_compress_v<float, false>(a, s);
}

cudaError_t launch_compress_dense(const StateView &sv, int factor_dtype, const float *S,
                                  float *trunc_err, cudaStream_t s) {
  CompressArgs a{sv, trunc_err, nullptr, S, sv.d_v, 0};
  if (factor_dtype == SEED_BF16) return launch_compress_v<__nv_bfloat16, true>(a, s);
  return launch_compress_v<float, true>(a, s);
}

}  // namespace seedk
