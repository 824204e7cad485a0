// Device building blocks of the compression kernels: Householder QR of a
// factor panel in shared memory, the explicit Q, pivoted QR and the
// seat-indexed one-sided Jacobi SVD of the core.  Used whole by the single-kernel
// recompression and the dense compression (recompress.cu); the three-phase
// recompression (recompress_split.cu) takes the constants, the seat geometry
// and the column helpers from here and lays the same steps out in registers
// (qr_registers.cuh) and per warp (svd_warp.cuh).
#pragma once

#include "common.cuh"

#include <float.h>

namespace seedk {

constexpr int kMaxSweeps = 30;
// After the core is scaled to a largest entry in [1/2, 1), a column whose squared
// norm is below this is under fp32 resolution of the largest one: rotating it only
// stirs rounding noise, so it is left alone (its singular value is negligible).
constexpr float kNegligible = 1e-14f;

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
// Run by a team of tsize threads (ttid its index) synchronised on named barrier bar.
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

// Thread geometry of the Jacobi rounds on an n x n core: tpp threads per column
// pair (as many as fit in nthreads, at most 32, at least 8 rows each), each
// owning R = ld / tpp rows (R a multiple of 4, rows n..ld-1 zero); cs is the
// column stride (refined by seat_geom).
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



// ---------------------------------------------------------------------------
// Preconditioned Jacobi on the core: K P = Q R (Householder QR with column
// pivoting), then one-sided Jacobi on the columns of R^T.  The pivoted R is
// graded (decreasing diagonal), so the rotations converge in about half the
// sweeps needed on K itself.  The columns of R^T J are V Sigma with V the right
// singular vectors of R; those of K are P V, and K (P v_k) = sigma_k x_k.
// ---------------------------------------------------------------------------

// y[i] -= a x[i] over rows [i0, nrows) (layout rules of col_axpy); returns the
// sum of squares of the updated y[i0..nrows).
__device__ static inline float col_axpy_ss(float a, const float *__restrict__ x, float *__restrict__ y,
                                           int i0, int nrows) {
  float ss = 0.f;
  int i = i0;
  for (; (i & 3) && i < nrows; ++i) {
    const float c = fmaf(-a, x[i], y[i]);
    y[i] = c;
    ss = fmaf(c, c, ss);
  }
  for (; i < nrows; i += 4) {
    const float4 b = *reinterpret_cast<const float4 *>(x + i);
    float4 c = *reinterpret_cast<const float4 *>(y + i);
    c.x = fmaf(-a, b.x, c.x); c.y = fmaf(-a, b.y, c.y); c.z = fmaf(-a, b.z, c.z); c.w = fmaf(-a, b.w, c.w);
    *reinterpret_cast<float4 *>(y + i) = c;
    ss = fmaf(c.x, c.x, fmaf(c.y, c.y, fmaf(c.z, c.z, fmaf(c.w, c.w, ss))));
  }
  return ss;
}

// Householder QR with column pivoting of the nrows x ncols matrix A (nrows >=
// ncols; column-major, column stride cs a multiple of 4, rows nrows..n4-1 zero
// with n4 = nrows rounded up to 4).  Each step moves the remaining column of
// largest trailing norm to the front (ties: the lower index); the trailing norms
// are recomputed from the updated columns rather than downdated.  On exit the
// upper triangle holds R and piv[j] is the original index of column j:
// A[:, piv] = Q R.  Warp 0 forms the pivot and the reflector, all NT threads
// update the trailing columns.  vn (ncols floats) and red (2 floats) are
// shared scratch.
template <int NT>
__device__ static void qrcp_rect(float *A, int nrows, int ncols, int cs, int *piv, float *vn, float *red) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int n4 = (nrows + 3) & ~3;
  for (int l = tid; l < ncols; l += NT) {
    vn[l] = col_dot(A + l * cs, A + l * cs, 0, n4);
    piv[l] = l;
  }
  __syncthreads();
  for (int j = 0; j < ncols; ++j) {
    float *cj = A + j * cs;
    if (tid < 32) {
      float best = -1.f;
      int bi = ncols;
      for (int l = j + lane; l < ncols; l += 32)
        if (vn[l] > best) { best = vn[l]; bi = l; }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ob = __shfl_xor_sync(0xffffffffu, best, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ob > best || (ob == best && oi < bi)) { best = ob; bi = oi; }
      }
      if (bi != j && bi < ncols) {
        float *cb = A + bi * cs;
        for (int i = lane; i < nrows; i += 32) {
          const float t = cj[i];
          cj[i] = cb[i];
          cb[i] = t;
        }
        if (lane == 0) {
          const int t = piv[j];
          piv[j] = piv[bi];
          piv[bi] = t;
          vn[bi] = vn[j];
        }
      }
      __syncwarp();
      float amax = 0.f;
      for (int i = j + lane; i < n4; i += 32) amax = fmaxf(amax, fabsf(cj[i]));
      amax = warp_max(amax);
      const float alpha = cj[j];
      float tj = 0.f, beta = alpha;
      if (amax >= FLT_MIN) {
        const float inv = 1.f / amax;
        float ss = 0.f;
        for (int i = j + 1 + lane; i < n4; i += 32) {
          const float x = cj[i] * inv;
          ss = fmaf(x, x, ss);
        }
        ss = warp_sum(ss);
        if (ss > 0.f) {
          const float as = alpha * inv;
          const float nrm = sqrtf(fmaf(as, as, ss));
          const float bs = as >= 0.f ? -nrm : nrm;
          tj = (bs - as) / bs;
          const float sc = 1.f / ((as - bs) * amax);
          for (int i = j + 1 + lane; i < n4; i += 32) cj[i] *= sc;
          beta = bs * amax;
        }
      } else {
        for (int i = j + 1 + lane; i < n4; i += 32) cj[i] = 0.f;
      }
      __syncwarp();
      if (lane == 0) { cj[j] = beta; red[0] = tj; }
    }
    __syncthreads();
    const float tj = red[0];
    for (int l = j + 1 + tid; l < ncols; l += NT) {
      float *cl = A + l * cs;
      if (tj != 0.f) {
        const float sv = tj * (cl[j] + col_dot(cj, cl, j + 1, n4));
        cl[j] -= sv;
        vn[l] = col_axpy_ss(sv, cj, cl, j + 1, n4);
      } else {
        vn[l] = col_dot(cl, cl, j + 1, n4);
      }
    }
    __syncthreads();
  }
}

template <int NT>
__device__ static void qrcp(float *A, int m, int cs, int *piv, float *vn, float *red) {
  qrcp_rect<NT>(A, m, m, cs, piv, vn, red);
}

// Geometry of the seat-indexed Jacobi: as jacobi_geom, with the seat stride cs
// the smallest value >= ld with cs = 16 (mod 32) floats, so that two adjacent
// seats start four 16-byte bank groups apart.
__host__ __device__ inline JacobiGeom seat_geom(int n, int nthreads) {
  JacobiGeom g = jacobi_geom(n, nthreads);
  g.cs = g.ld + (((16 - g.ld) % 32) + 32) % 32;
  return g;
}
__host__ inline int seat_cs_alloc(int m_max, int nthreads) {
  int cs = 16;
  for (int n = 0; n <= m_max; ++n) {
    const int c = seat_geom(n, nthreads).cs;
    cs = c > cs ? c : cs;
  }
  return cs;
}

// One-sided Jacobi with the columns moving between seats (round-robin with seat
// 0 fixed: after each round the column at seat s >= 1 moves to seat s + 1, the
// one at seat n'-1 to seat 1; pair i rotates seats i and n'-1-i).  Columns are
// read from one buffer and written, rotated, to their next seats in the other,
// so the 16-byte chunks that the threads of two adjacent pairs touch always
// fall in distinct bank groups (chunk c of a pair's column goes to thread
// c mod tpp).  A pair is rotated when (k_p . k_q)^2 > tol^2 |k_p|^2 |k_q|^2 and
// both columns are above fp32 resolution of the core (scaled to a largest entry
// in [1/2, 1)); the angle comes from fast reciprocals, which is exact enough
// because any t gives an orthogonal rotation (c^2 + s^2 = 1 to rounding), and
// |zeta| large (tiny k_p . k_q) gives t ~ 1/(2 zeta).  The sweeps stop
// after the first one in which no pair was further from orthogonal than
// tol_stop (|cos| of the pair's angle): rotations converge quadratically, so
// what is left after such a sweep is of order tol_stop^2 (tol_stop = sqrt(tol)
// leaves about tol), and the sweep that would only confirm it is saved.  buf0 holds column j
// at seat j (seat stride g.cs, rows padded with zeros to g.ld; an odd n gets a
// zero column at seat n).  After whole sweeps every column is back at its
// seat; *out points to the buffer that holds them.  Whole block of NT threads.
// Returns the number of sweeps, or -1 if the sweep limit was reached.
template <int NT, int RMAX>
__device__ static int jacobi_seats(float *buf0, float *buf1, int n, const JacobiGeom &g, float tol,
                                   float tol_stop, float **out) {
  *out = buf0;
  if (n < 2) return 0;
  const int tid = threadIdx.x;
  const int nn = n + (n & 1);
  const int P = nn / 2;
  const int tpp = g.tpp, cs = g.cs;
  const int R4 = g.ld / tpp / 4;
  const int pair = tid / tpp, sub = tid % tpp;
  const bool active = pair < P;
  const float tol2 = tol * tol, stop2 = tol_stop * tol_stop;
  const int st = active ? pair : 0, sb = active ? nn - 1 - pair : 1;
  const int nt = st == 0 ? 0 : (st == nn - 1 ? 1 : st + 1);
  const int nb = sb == nn - 1 ? 1 : sb + 1;
  int p = st, q = sb;  // columns at my seats; column at seat s >= 1 steps down by one per round
  float *cur = buf0, *nxt = buf1;
  for (int sweep = 0; sweep < kMaxSweeps; ++sweep) {
    int far = 0;  // a pair in this sweep was further from orthogonal than tol_stop
    for (int round = 0; round < nn - 1; ++round) {
      float4 xp[RMAX / 4], xq[RMAX / 4];
      float al = 0.f, be = 0.f, ga = 0.f;
      if (active) {
        const float4 *kp = reinterpret_cast<const float4 *>(cur + st * cs) + sub;
        const float4 *kq = reinterpret_cast<const float4 *>(cur + sb * cs) + sub;
#pragma unroll
        for (int v = 0; v < RMAX / 4; ++v) {
          if (v < R4) {
            xp[v] = kp[v * tpp];
            xq[v] = kq[v * tpp];
            al = fmaf(xp[v].x, xp[v].x, fmaf(xp[v].y, xp[v].y, fmaf(xp[v].z, xp[v].z, fmaf(xp[v].w, xp[v].w, al))));
            be = fmaf(xq[v].x, xq[v].x, fmaf(xq[v].y, xq[v].y, fmaf(xq[v].z, xq[v].z, fmaf(xq[v].w, xq[v].w, be))));
            ga = fmaf(xp[v].x, xq[v].x, fmaf(xp[v].y, xq[v].y, fmaf(xp[v].z, xq[v].z, fmaf(xp[v].w, xq[v].w, ga))));
          }
        }
      }
      // every lane of the warp takes part (a warp may hold active and idle pairs)
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        if (o < tpp) {
          al += __shfl_xor_sync(0xffffffffu, al, o);
          be += __shfl_xor_sync(0xffffffffu, be, o);
          ga += __shfl_xor_sync(0xffffffffu, ga, o);
        }
      }
      if (active) {
        float4 *wp = reinterpret_cast<float4 *>(nxt + nt * cs) + sub;
        float4 *wq = reinterpret_cast<float4 *>(nxt + nb * cs) + sub;
        if (p < n && q < n && al > kNegligible && be > kNegligible && ga * ga > tol2 * al * be) {
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
              wp[v * tpp] = make_float4(fmaf(c, a.x, -s * b.x), fmaf(c, a.y, -s * b.y), fmaf(c, a.z, -s * b.z),
                                        fmaf(c, a.w, -s * b.w));
              wq[v * tpp] = make_float4(fmaf(s, a.x, c * b.x), fmaf(s, a.y, c * b.y), fmaf(s, a.z, c * b.z),
                                        fmaf(s, a.w, c * b.w));
            }
          }
          far |= ga * ga > stop2 * al * be;
        } else {
#pragma unroll
          for (int v = 0; v < RMAX / 4; ++v) {
            if (v < R4) {
              wp[v * tpp] = xp[v];
              wq[v * tpp] = xq[v];
            }
          }
        }
        if (st != 0) p = p == 1 ? nn - 1 : p - 1;
        q = q == 1 ? nn - 1 : q - 1;
      }
      float *t = cur;
      cur = nxt;
      nxt = t;
      if (round < nn - 2) __syncthreads();
    }
    if (!__syncthreads_or(far)) {
      *out = cur;
      return sweep + 1;
    }
  }
  *out = cur;
  return -1;
}

// The core stage shared by both recompression schedules.  In: Kb holds the
// scaled core (column j at j * g.cs, rows m..m4-1 zero), Tb a second buffer of
// the same size (n' seats).  Pivoted QR of K in Kb, R^T into Tb, Jacobi between
// the two; then the squared column norms sig2 (= sigma^2 of the core), their
// inverse square roots inv (0 below fp32 resolution), and order (column
// indices by decreasing sigma, ties by index); the Jacobi stops after a sweep
// with no pair beyond tol_stop from orthogonal.  *fin is the buffer that holds
// the columns V Sigma of R^T J; piv the column pivots of the QR.  Returns the
// Jacobi sweeps (or -1).  Whole block of NT threads; ends with a barrier.
template <int NT>
__device__ static int core_factor(float *Kb, float *Tb, int m, const JacobiGeom &g, float tol, float tol_stop,
                                  int *piv, float *vn, float *sig2, float *inv, int *order, float *red,
                                  float **fin) {
  const int tid = threadIdx.x;
  const int cs = g.cs, ld = g.ld;
  qrcp<NT>(Kb, m, cs, piv, vn, red);
  const int nn = m + (m & 1);
  for (int idx = tid; idx < nn * ld; idx += NT) {
    const int j = idx / ld, i = idx % ld;  // seat j of R^T = row j of R
    Tb[j * cs + i] = (j < m && i < m && i >= j) ? Kb[i * cs + j] : 0.f;
  }
  __syncthreads();
  const int sweeps = jacobi_seats<NT, 16>(Tb, Kb, m, g, tol, tol_stop, fin);
  const float *F = *fin;
  for (int j = tid; j < m; j += NT) {
    float acc = 0.f;
    for (int i = 0; i < m; ++i) acc = fmaf(F[j * cs + i], F[j * cs + i], acc);
    sig2[j] = acc;
    inv[j] = acc > kNegligible ? rsqrtf(acc) : 0.f;
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
  return sweeps;
}

}  // namespace seedk
