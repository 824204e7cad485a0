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
//   one-sided Jacobi SVD of K: rotate pairs of columns of K (and of Y = I)
//     until every pair is orthogonal; then K Y = X Sigma, K = X Sigma Y^T
//   order columns by |K_j| (= sigma_j), keep the rank(h) largest
//   Q_a, Q_b formed in place from the reflectors
//   U_new = Q_a (K)[:, kept] = Q_a X_r Sigma_r,  W_new = Q_b Y[:, kept]
// compress_dense (one CTA of 256 threads per head): the same with A = C and
// B = I (so K = R_a and W_new = Y[:, kept]).
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
};

// Householder QR in place on a column-major nrows x ncols panel (leading
// dimension ld).  On exit the upper triangle holds R; below the diagonal of
// column j sits the reflector's vector v_j (v_j[j] = 1 implicit), tau[j] its
// coefficient: H_j = I - tau_j v_j v_j^T, A = H_0 H_1 ... H_{n-1} R.
// Each reflector is formed from the column scaled by its largest magnitude,
// so that columns far below 1 (long products of gates) do not underflow in
// their squared norm: an inaccurate norm would give a reflector that is not
// orthogonal, which then corrupts the larger columns it is applied to.
// Columns below the smallest normal float are treated as zero.
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
          const float sc = 1.f / ((as - bs) * amax);   // v_i = x_i / (alpha - beta), |v_i| <= 1
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
        float s0 = cl[j], s1 = 0.f, s2 = 0.f, s3 = 0.f;
        int i = j + 1;
        for (; i + 3 < nrows; i += 4) {
          s0 = fmaf(cj[i], cl[i], s0);
          s1 = fmaf(cj[i + 1], cl[i + 1], s1);
          s2 = fmaf(cj[i + 2], cl[i + 2], s2);
          s3 = fmaf(cj[i + 3], cl[i + 3], s3);
        }
        for (; i < nrows; ++i) s0 = fmaf(cj[i], cl[i], s0);
        const float sv = tj * ((s0 + s1) + (s2 + s3));
        cl[j] -= sv;
        for (i = j + 1; i < nrows; ++i) cl[i] = fmaf(-sv, cj[i], cl[i]);
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
        float *cl = A + l * ld;  // rows < l of a finished column are zero
        float s0 = 0.f, s1 = 0.f;
        int i = j + 1;
        for (; i + 1 < nrows; i += 2) {
          s0 = fmaf(cj[i], cl[i], s0);
          s1 = fmaf(cj[i + 1], cl[i + 1], s1);
        }
        for (; i < nrows; ++i) s0 = fmaf(cj[i], cl[i], s0);
        const float sv = tj * (s0 + s1);   // cl[j] == 0 here
        cl[j] = -sv;
        for (i = j + 1; i < nrows; ++i) cl[i] = fmaf(-sv, cj[i], cl[i]);
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

// One-sided (Hestenes) Jacobi on the n columns of K (ld x n, rows 0..n-1),
// accumulating the rotations in Y (starts as I).  Round-robin pair order: n'
// = n rounded up to even seats, seat 0 fixed, the others rotate each round;
// pair i joins seats i and n'-1-i.  A pair is rotated when
// |k_p . k_q| > tol |k_p| |k_q|.  Whole block (NT threads).  Returns the
// number of sweeps, or -1 if the sweep limit was reached while still rotating.
template <int NT>
__device__ static int jacobi_svd(float *K, float *Y, int ld, int n, float tol) {
  const int tid = threadIdx.x;
  for (int idx = tid; idx < n * ld; idx += NT) {
    const int c = idx / ld, r = idx % ld;
    Y[idx] = (r == c) ? 1.f : 0.f;
  }
  if (n < 2) { __syncthreads(); return 0; }
  const int nn = n + (n & 1);
  const int P = nn / 2;
  int tpp = 1;
  while (tpp * 2 * P <= NT && tpp < 32) tpp *= 2;
  const int pair = tid / tpp, sub = tid % tpp;
  const bool active = pair < P;
  __syncthreads();
  for (int sweep = 0; sweep < kMaxSweeps; ++sweep) {
    int rotated = 0;
    for (int round = 0; round < nn - 1; ++round) {
      int p = -1, q = -1;
      if (active) {
        const int sp = pair, sq = nn - 1 - pair;
        p = sp == 0 ? 0 : 1 + (sp - 1 + round) % (nn - 1);
        q = 1 + (sq - 1 + round) % (nn - 1);
      }
      const bool real = active && p < n && q < n;
      float al = 0.f, be = 0.f, ga = 0.f;
      if (real) {
        const float *kp = K + p * ld, *kq = K + q * ld;
        for (int r = sub; r < n; r += tpp) {
          const float x = kp[r], y = kq[r];
          al = fmaf(x, x, al); be = fmaf(y, y, be); ga = fmaf(x, y, ga);
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
        const float zeta = (be - al) / (2.f * ga);
        const float t = copysignf(1.f, zeta) / (fabsf(zeta) + sqrtf(fmaf(zeta, zeta, 1.f)));
        const float c = rsqrtf(fmaf(t, t, 1.f));
        const float s = c * t;
        float *kp = K + p * ld, *kq = K + q * ld, *yp = Y + p * ld, *yq = Y + q * ld;
        for (int r = sub; r < n; r += tpp) {
          const float x = kp[r], y = kq[r];
          kp[r] = fmaf(c, x, -s * y);
          kq[r] = fmaf(s, x, c * y);
          const float u = yp[r], w = yq[r];
          yp[r] = fmaf(c, u, -s * w);
          yq[r] = fmaf(s, u, c * w);
        }
        rotated = 1;
      }
      __syncthreads();
    }
    if (!__syncthreads_or(rotated)) return sweep + 1;
  }
  return -1;
}

// Dynamic shared-memory layout of the compression kernels.
struct Smem {
  int lda, ldb, ldk;
  int offA, offB, offK, offY, offTa, offTb, offS, offO, offR;
  int total_floats;
  __host__ __device__ Smem(int m, int dk, int dv, bool dense) {
    lda = dk + 1;
    ldb = dv + 1;
    ldk = m + 1;
    offA = 0;
    offB = offA + m * lda;
    offK = offB + (dense ? 0 : m * ldb);
    offY = offK + m * ldk;
    offTa = offY + m * ldk;
    offTb = offTa + m;
    offS = offTb + m;
    offO = offS + m;
    offR = offO + m;          // 8 floats of reduction scratch
    total_floats = offR + 8;
  }
};

template <int VAR, typename TF, int DV, bool DENSE>
__global__ void __launch_bounds__(DENSE ? 256 : 128) compress_kernel(const CompressArgs p) {
  constexpr int DK = kDK;
  constexpr int NT = DENSE ? 256 : 128;
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
  const Smem L(DENSE ? DV : p.m_max, DK, DV, DENSE);
  float *A = smem + L.offA, *B = smem + L.offB, *K = smem + L.offK, *Y = smem + L.offY;
  float *tauA = smem + L.offTa, *tauB = smem + L.offTb, *sig2 = smem + L.offS;
  int *order = reinterpret_cast<int *>(smem + L.offO);
  const int lda = L.lda, ldb = L.ldb, ldk = L.ldk;
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

  // ---- core K = R_a R_b^T (or R_a) ----------------------------------------------
  for (int idx = tid; idx < m * m; idx += NT) {
    const int j = idx / m, i = idx % m;  // K[j][i]: column j, row i
    float acc = 0.f;
    if (DENSE) {
      acc = i <= j ? A[j * lda + i] : 0.f;
    } else {
      for (int l = max(i, j); l < m; ++l) acc = fmaf(A[l * lda + i], B[l * ldb + j], acc);
    }
    K[j * ldk + i] = acc;
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
  __syncthreads();

  // ---- SVD of the core, scaled by a power of two to a largest entry in [1/2, 1) ----------
  float kmax = 0.f;
  for (int idx = tid; idx < m * m; idx += NT) kmax = fmaxf(kmax, fabsf(K[(idx / m) * ldk + idx % m]));
  kmax = warp_max(kmax);
  float *red = smem + L.offR;
  if ((tid & 31) == 0) red[tid >> 5] = kmax;
  __syncthreads();
  kmax = 0.f;
  for (int w = 0; w < NT / 32; ++w) kmax = fmaxf(kmax, red[w]);
  int kexp = 0;
  if (kmax > 0.f) frexpf(kmax, &kexp);
  const float kscale = ldexpf(1.f, -kexp), kunscale = ldexpf(1.f, kexp);
  __syncthreads();
  for (int idx = tid; idx < m * m; idx += NT) K[(idx / m) * ldk + idx % m] *= kscale;
  __syncthreads();
  const float tol = (float)(m > 16 ? m : 16) * FLT_EPSILON;
  const int sweeps = jacobi_svd<NT>(K, Y, ldk, m, tol);

  // ---- order by sigma, truncation error -----------------------------------------------
  for (int j = tid; j < m; j += NT) {
    float acc = 0.f;
    for (int i = 0; i < m; ++i) acc = fmaf(K[j * ldk + i], K[j * ldk + i], acc);
    sig2[j] = acc;
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

  // ---- rebuild the kept columns -----------------------------------------------------
  const int rk = r < m ? r : m;
  if (tid < DK) {
    for (int k = 0; k < rk; ++k) {
      const float *z = K + order[k] * ldk;
      float acc = 0.f;
      for (int l = 0; l < m; ++l) acc = fmaf(A[l * lda + tid], z[l], acc);
      Elem<TF>::store(Uh + (int64_t)k * DK + tid, acc * kunscale);
    }
  }
  if (tid >= NT - DV) {
    const int i = tid - (NT - DV);
    for (int k = 0; k < rk; ++k) {
      const float *y = Y + order[k] * ldk;
      float acc;
      if (DENSE) {
        acc = y[i];
      } else {
        acc = 0.f;
        for (int l = 0; l < m; ++l) acc = fmaf(B[l * ldb + i], y[l], acc);
      }
      Elem<TF>::store(Wh + (int64_t)k * DV + i, acc);
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
  const Smem L(DENSE ? DV : a.m_max, kDK, DV, DENSE);
  const size_t bytes = (size_t)L.total_floats * sizeof(float);
  auto kern = compress_kernel<VAR, TF, DV, DENSE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  kern<<<a.sv.n_heads, DENSE ? 256 : 128, bytes, s>>>(a);
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
  CompressArgs a{sv, trunc_err, sweeps, nullptr, m_max};
  if (factor_dtype == SEED_BF16) return launch_compress_v<__nv_bfloat16, false>(a, s);
  return launch_compress_v<float, false>(a, s);
}

cudaError_t launch_compress_dense(const StateView &sv, int factor_dtype, const float *S,
                                  float *trunc_err, cudaStream_t s) {
  CompressArgs a{sv, trunc_err, nullptr, S, sv.d_v};
  if (factor_dtype == SEED_BF16) return launch_compress_v<__nv_bfloat16, true>(a, s);
  return launch_compress_v<float, true>(a, s);
}

}  // namespace seedk
