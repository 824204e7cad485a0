// SVD of the recompression core with one warp per head and the core in
// registers: pivoted Householder QR K P = Q R, then one-sided Jacobi on the
// columns of R^T (the algorithm of core_factor in recompress_core.cuh, laid
// out for a warp instead of a CTA, so that no block barrier is needed).
//
// Pivoted QR: lane l holds columns l and l + 32 of K (all rows, in
// registers).  Each step the warp picks the remaining column of largest
// trailing norm (shuffle argmax, ties to the lower index), its owner lays it
// out in a shared row, the 32 lanes form the reflector there (scaled by the
// column's largest magnitude, as householder_qr), and every lane applies it to
// its remaining columns, refreshing their trailing norms.  Columns keep their
// lanes; only the pivot order is recorded.
//
// Jacobi: lane i (i < P = n'/2) holds two seats in registers, A and B:
// lane 0 has seat n'-1 in A and the fixed seat 0 in B, lane i >= 1 has seat i
// in A and seat n'-1-i in B.  After each round the column at seat s >= 1 moves
// to seat s + 1 (n'-1 to 1); with this assignment that is one shuffle up of A
// and one shuffle down of B per element, plus the ends of the chain.  Rotation
// rule, tolerance and stopping rule as jacobi_seats.
#pragma once

#include "recompress_core.cuh"

namespace seedk {

constexpr int kSvdWarps = 2;  // heads (warps) per CTA

// Per-warp shared layout (floats): a row-pitch-(MR+1) square for transposes,
// the reflector row, sigma^2, 1/sigma, the column order and the pivots.
template <int MR>
struct SvdWarpSmem {
  static constexpr int TP = MR + 1;
  static constexpr int T_OFF = 0;
  static constexpr int V_OFF = (MR * TP + 3) & ~3;
  static constexpr int S_OFF = V_OFF + MR;
  static constexpr int I_OFF = S_OFF + MR;
  static constexpr int O_OFF = I_OFF + MR;
  static constexpr int P_OFF = O_OFF + MR;
  static constexpr int FLOATS = P_OFF + MR;
};

// One warp: pivoted QR of the scaled core (columns c0 = K[:, lane], c1 =
// K[:, lane + 32]), then Jacobi on R^T.  Leaves in the warp's shared square F
// (row pitch TP) the columns of R^T J by seat (F[seat * TP + s]), sig2/inv by
// seat, order, piv.  Returns the sweeps (or -1).
template <int MR>
__device__ int svd_warp_core(float (&c0)[MR], float (&c1)[MR], int m, float tol, float *sw) {
  using L = SvdWarpSmem<MR>;
  constexpr bool TWO = MR > 32;
  constexpr int RPL = (MR + 31) / 32;  // rows per lane in the reflector
  const int lane = threadIdx.x & 31;
  const unsigned full = 0xffffffffu;
  float *T = sw + L::T_OFF, *vrow = sw + L::V_OFF, *sig2 = sw + L::S_OFF, *inv = sw + L::I_OFF;
  int *order = reinterpret_cast<int *>(sw + L::O_OFF);
  int *piv = reinterpret_cast<int *>(sw + L::P_OFF);

  // ---- pivoted QR ------------------------------------------------------------------------
  float vn0 = 0.f, vn1 = 0.f;
#pragma unroll
  for (int r = 0; r < MR; ++r) {
    vn0 = fmaf(c0[r], c0[r], vn0);
    if (TWO) vn1 = fmaf(c1[r], c1[r], vn1);
  }
  bool done0 = lane >= m, done1 = !TWO || lane + 32 >= m;
  int s0 = 0, s1 = 0;  // step at which my column was chosen (its column index in R)
  for (int j = 0; j < m; ++j) {
    float best = -1.f;
    int bi = 1 << 20;
    if (!done0) { best = vn0; bi = lane; }
    if (!done1 && vn1 > best) { best = vn1; bi = lane + 32; }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ob = __shfl_xor_sync(full, best, o);
      const int oi = __shfl_xor_sync(full, bi, o);
      if (ob > best || (ob == best && oi < bi)) { best = ob; bi = oi; }
    }
    const int pc = bi, owner = pc & 31;
    const bool hi = pc >= 32;
    if (lane == owner) {
#pragma unroll
      for (int r = 0; r < MR; ++r) vrow[r] = hi ? c1[r] : c0[r];
    }
    __syncwarp();
    float a[RPL];
#pragma unroll
    for (int e = 0; e < RPL; ++e) a[e] = lane + 32 * e < MR ? vrow[lane + 32 * e] : 0.f;
    const float alpha = vrow[j];
    float tj = 0.f, beta = alpha, sc = 0.f;
    // one reduction for the norm unless it nears the ends of the fp32 range
    // (then scaled by the largest magnitude, as householder_qr)
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < RPL; ++e) {
      const float x = lane + 32 * e > j ? a[e] : 0.f;
      ss = fmaf(x, x, ss);
    }
    ss = warp_sum(ss);
    float amax = 1.f;
    if (!(ss >= 1e-30f && ss <= 1e30f)) {
      amax = 0.f;
#pragma unroll
      for (int e = 0; e < RPL; ++e)
        if (lane + 32 * e >= j) amax = fmaxf(amax, fabsf(a[e]));
      amax = warp_max(amax);
      ss = 0.f;
      if (amax >= FLT_MIN) {
        const float rinv = 1.f / amax;
#pragma unroll
        for (int e = 0; e < RPL; ++e) {
          const float xs = lane + 32 * e > j ? a[e] * rinv : 0.f;
          ss = fmaf(xs, xs, ss);
        }
        ss = warp_sum(ss);
      }
    }
    if (ss > 0.f && amax >= FLT_MIN) {
      const float as = alpha / amax;
      const float nrm = sqrtf(fmaf(as, as, ss));
      const float bs = as >= 0.f ? -nrm : nrm;
      tj = (bs - as) / bs;
      sc = 1.f / ((as - bs) * amax);
      beta = bs * amax;
    }
    __syncwarp();
#pragma unroll
    for (int e = 0; e < RPL; ++e) {
      const int r = lane + 32 * e;
      if (r < MR) vrow[r] = r < j ? 0.f : r == j ? 1.f : a[e] * sc;
    }
    if (lane == 0) piv[j] = pc;
    __syncwarp();
    // the chosen column becomes column j of R (rows above j were finished by
    // the earlier steps, row j is beta, rows below are zero)
    if (lane == owner) {
#pragma unroll
      for (int r = 0; r < MR; ++r) {
        if (hi) { if (r == j) c1[r] = beta; else if (r > j) c1[r] = 0.f; }
        else { if (r == j) c0[r] = beta; else if (r > j) c0[r] = 0.f; }
      }
      if (hi) { done1 = true; s1 = j; } else { done0 = true; s0 = j; }
    }
    // the remaining columns: a -= tau (v . a) v, then their norms below row j
    const float4 *v4 = reinterpret_cast<const float4 *>(vrow);
    if (!done0 || !done1) {
      float d0 = 0.f, d1 = 0.f;
#pragma unroll
      for (int q = 0; q < MR / 4; ++q) {
        const float4 v = v4[q];
        d0 = fmaf(v.x, c0[4 * q], fmaf(v.y, c0[4 * q + 1], fmaf(v.z, c0[4 * q + 2], fmaf(v.w, c0[4 * q + 3], d0))));
        if (TWO) d1 = fmaf(v.x, c1[4 * q], fmaf(v.y, c1[4 * q + 1], fmaf(v.z, c1[4 * q + 2], fmaf(v.w, c1[4 * q + 3], d1))));
      }
      const float t0 = done0 ? 0.f : tj * d0, t1 = done1 ? 0.f : tj * d1;
      float n0 = 0.f, n1 = 0.f;
#pragma unroll
      for (int q = 0; q < MR / 4; ++q) {
        const float4 v = v4[q];
        const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int r = 4 * q + e;
          c0[r] = fmaf(-t0, vv[e], c0[r]);
          const float y0 = r > j ? c0[r] : 0.f;
          n0 = fmaf(y0, y0, n0);
          if (TWO) {
            c1[r] = fmaf(-t1, vv[e], c1[r]);
            const float y1 = r > j ? c1[r] : 0.f;
            n1 = fmaf(y1, y1, n1);
          }
        }
      }
      if (!done0) vn0 = n0;
      if (!done1) vn1 = n1;
    }
    __syncwarp();
  }

  // ---- R^T to the seats of the Jacobi: seat i = row i of R --------------------------------
  if (lane < m) {
#pragma unroll
    for (int r = 0; r < MR; ++r) T[s0 * L::TP + r] = c0[r];
  }
  if (TWO && lane + 32 < m) {
#pragma unroll
    for (int r = 0; r < MR; ++r) T[s1 * L::TP + r] = c1[r];
  }
  __syncwarp();
  const int nn = m + (m & 1), P = nn / 2;
  const bool active = lane < P;
  const int seatA = lane == 0 ? nn - 1 : lane, seatB = lane == 0 ? 0 : nn - 1 - lane;
  float A[MR], B[MR];
#pragma unroll
  for (int s = 0; s < MR; ++s) {
    A[s] = (active && s < m && seatA < m) ? T[s * L::TP + seatA] : 0.f;
    B[s] = (active && s < m && seatB < m) ? T[s * L::TP + seatB] : 0.f;
  }
  __syncwarp();

  // ---- Jacobi -------------------------------------------------------------------------------
  int sweeps = 0;
  if (m >= 2) {
    const float tol2 = tol * tol, stop2 = tol;  // tol_stop = sqrt(tol)
    int colA = seatA, colB = seatB;            // column indices at my seats (>= m: the zero seat)
    sweeps = -1;
    for (int sweep = 0; sweep < kMaxSweeps; ++sweep) {
      int far = 0;
      for (int round = 0; round < nn - 1; ++round) {
        float al0 = 0.f, al1 = 0.f, be0 = 0.f, be1 = 0.f, ga0 = 0.f, ga1 = 0.f;
#pragma unroll
        for (int s = 0; s < MR; s += 2) {
          al0 = fmaf(A[s], A[s], al0); be0 = fmaf(B[s], B[s], be0); ga0 = fmaf(A[s], B[s], ga0);
          al1 = fmaf(A[s + 1], A[s + 1], al1); be1 = fmaf(B[s + 1], B[s + 1], be1);
          ga1 = fmaf(A[s + 1], B[s + 1], ga1);
        }
        const float al = al0 + al1, be = be0 + be1, ga = ga0 + ga1;
        if (active && colA < m && colB < m && al > kNegligible && be > kNegligible && ga * ga > tol2 * al * be) {
          const float zeta = (be - al) * __frcp_rn(2.f * ga);
          const float az = fabsf(zeta);
          const float root = az < 1e18f ? az + fmaf(az, az, 1.f) * rsqrtf(fmaf(az, az, 1.f)) : 2.f * az;
          const float t = copysignf(__frcp_rn(root), zeta);
          const float c = rsqrtf(fmaf(t, t, 1.f));
          const float sn = c * t;
#pragma unroll
          for (int s = 0; s < MR; ++s) {
            const float a = A[s], b = B[s];
            A[s] = fmaf(c, a, -sn * b);
            B[s] = fmaf(sn, a, c * b);
          }
          far |= ga * ga > stop2 * al * be;
        }
        if (P > 1) {
          // seat s >= 1 moves to s + 1 (n'-1 to 1): A up one lane, B down one lane;
          // lane 0 takes lane 1's B into A, lane P-1 keeps its A as B
#pragma unroll
          for (int s = 0; s < MR; ++s) {
            const float up = __shfl_up_sync(full, A[s], 1);
            const float dn = __shfl_down_sync(full, B[s], 1);
            const float a = A[s];
            A[s] = lane == 0 ? dn : up;
            if (lane == P - 1) B[s] = a;
            else if (lane != 0) B[s] = dn;
          }
          const int cu = __shfl_up_sync(full, colA, 1), cd = __shfl_down_sync(full, colB, 1);
          const int ca = colA;
          colA = lane == 0 ? cd : cu;
          if (lane == P - 1) colB = ca;
          else if (lane != 0) colB = cd;
        }
      }
      if (!__any_sync(full, far)) {
        sweeps = sweep + 1;
        break;
      }
    }
  }

  // ---- columns of R^T J by seat, sigma^2, order -----------------------------------------------
  float sa = 0.f, sb = 0.f;
#pragma unroll
  for (int s = 0; s < MR; ++s) {
    sa = fmaf(A[s], A[s], sa);
    sb = fmaf(B[s], B[s], sb);
  }
  if (active) {
    if (seatA < m) {
#pragma unroll
      for (int s = 0; s < MR; ++s) T[seatA * L::TP + s] = A[s];
      sig2[seatA] = sa;
      inv[seatA] = sa > kNegligible ? rsqrtf(sa) : 0.f;
    }
    if (seatB < m) {
#pragma unroll
      for (int s = 0; s < MR; ++s) T[seatB * L::TP + s] = B[s];
      sig2[seatB] = sb;
      inv[seatB] = sb > kNegligible ? rsqrtf(sb) : 0.f;
    }
  }
  __syncwarp();
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int j = lane + 32 * e;
    if (j < m) {
      int rank = 0;
      const float sj = sig2[j];
      for (int i = 0; i < m; ++i) {
        const float si = sig2[i];
        rank += (si > sj) || (si == sj && i < j);
      }
      order[rank] = j;
    }
  }
  __syncwarp();
  return sweeps;
}

}  // namespace seedk
