// SVD of the recompression core with one warp per head and the core in
// registers: pivoted Householder QR K P = Q R, then one-sided Jacobi on the
// columns of R^T (the algorithm of core_factor in recompress_core.cuh, laid
// out for a warp instead of a CTA, so that no block barrier is needed).
//
// Pivoted QR: the core sits in the warp's shared square, column c at
// c * TP (TP = MR + 4: the 16-byte chunks of eight consecutive columns fall in
// distinct bank groups); lane l looks after columns l and l + 32.  Each step
// the warp picks the remaining column of largest trailing norm (shuffle argmax,
// ties to the lower index), the 32 lanes form the reflector from it (norm in one
// reduction, max-scaled near the fp32 range ends, as householder_qr), and every
// lane applies it to its remaining columns with 16-byte loads, refreshing their
// trailing norms.  Columns stay in place; only the pivot order is recorded.
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

// Per-warp shared layout (floats): the square (pitch MR + 4) that holds the
// core, then R^T's seats' results, the reflector row, sigma^2, 1/sigma, the
// column order and the pivots.
template <int MR>
struct SvdWarpSmem {
  static constexpr int TP = MR + 4;
  static constexpr int T_OFF = 0;
  static constexpr int V_OFF = (MR * TP + 3) & ~3;
  static constexpr int S_OFF = V_OFF + MR;
  static constexpr int I_OFF = S_OFF + MR;
  static constexpr int O_OFF = I_OFF + MR;
  static constexpr int P_OFF = O_OFF + MR;
  static constexpr int FLOATS = P_OFF + MR;
};

// One warp: pivoted QR of the scaled core held in the square T (column c at
// T[c * TP], rows m..MR-1 zero), then Jacobi on R^T.  Leaves in T the columns
// of R^T J by seat (T[seat * TP + s]), sig2/inv by seat, order, piv.  Returns
// the sweeps (or -1).
template <int MR>
__device__ int svd_warp_core(int m, float tol, float *sw) {
  using L = SvdWarpSmem<MR>;
  constexpr bool TWO = MR > 32;
  constexpr int RPL = (MR + 31) / 32;  // rows per lane in the reflector
  constexpr int TP = L::TP;
  const int lane = threadIdx.x & 31;
  const unsigned full = 0xffffffffu;
  float *T = sw + L::T_OFF, *vrow = sw + L::V_OFF, *sig2 = sw + L::S_OFF, *inv = sw + L::I_OFF;
  int *order = reinterpret_cast<int *>(sw + L::O_OFF);
  int *piv = reinterpret_cast<int *>(sw + L::P_OFF);
  const float4 *v4 = reinterpret_cast<const float4 *>(vrow);

  // ---- pivoted QR ------------------------------------------------------------------------
  auto colnorm = [&](int c, int from) {  // sum of squares of rows >= from of column c
    const float4 *x4 = reinterpret_cast<const float4 *>(T + c * TP);
    float a = 0.f;
#pragma unroll
    for (int q = 0; q < MR / 4; ++q) {
      const float4 x = x4[q];
      const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float y = 4 * q + e >= from ? xs[e] : 0.f;
        a = fmaf(y, y, a);
      }
    }
    return a;
  };
  bool done0 = lane >= m, done1 = !TWO || lane + 32 >= m;
  float vn0 = done0 ? 0.f : colnorm(lane, 0), vn1 = done1 ? 0.f : colnorm(lane + 32, 0);
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
    const int pc = bi;
    float *cp = T + pc * TP;
    float a[RPL];
#pragma unroll
    for (int e = 0; e < RPL; ++e) a[e] = lane + 32 * e < MR ? cp[lane + 32 * e] : 0.f;
    const float alpha = cp[j];
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
    // v_j into the reflector row; the chosen column becomes column j of R (rows
    // above j were finished by the earlier steps, row j is beta, rows below zero)
#pragma unroll
    for (int e = 0; e < RPL; ++e) {
      const int r = lane + 32 * e;
      if (r < MR) {
        vrow[r] = r < j ? 0.f : r == j ? 1.f : a[e] * sc;
        if (r >= j) cp[r] = r == j ? beta : 0.f;
      }
    }
    if (lane == 0) piv[j] = pc;
    if (lane == (pc & 31)) {
      if (pc >= 32) done1 = true;
      else done0 = true;
    }
    __syncwarp();
    // the remaining columns: a -= tau (v . a) v, then their norms below row j
#pragma unroll
    for (int h = 0; h < (TWO ? 2 : 1); ++h) {
      if (h == 0 ? done0 : done1) continue;
      float4 *x4 = reinterpret_cast<float4 *>(T + (lane + 32 * h) * TP);
      float d = 0.f;
#pragma unroll
      for (int q = 0; q < MR / 4; ++q) {
        const float4 v = v4[q], x = x4[q];
        d = fmaf(v.x, x.x, fmaf(v.y, x.y, fmaf(v.z, x.z, fmaf(v.w, x.w, d))));
      }
      const float t = tj * d;
      float nrm = 0.f;
#pragma unroll
      for (int q = 0; q < MR / 4; ++q) {
        const float4 v = v4[q];
        float4 x = x4[q];
        x.x = fmaf(-t, v.x, x.x); x.y = fmaf(-t, v.y, x.y); x.z = fmaf(-t, v.z, x.z); x.w = fmaf(-t, v.w, x.w);
        x4[q] = x;
        const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float y = 4 * q + e > j ? xs[e] : 0.f;
          nrm = fmaf(y, y, nrm);
        }
      }
      if (h == 0) vn0 = nrm;
      else vn1 = nrm;
    }
    __syncwarp();
  }

  // ---- R^T to the seats of the Jacobi: seat i = row i of R = T[s * TP + i] over s ----------
  // (R column s is the column chosen at step s: T[piv[s] * TP + i])
  const int nn = m + (m & 1), P = nn / 2;
  const bool active = lane < P;
  const int seatA = lane == 0 ? nn - 1 : lane, seatB = lane == 0 ? 0 : nn - 1 - lane;
  float A[MR], B[MR];
#pragma unroll
  for (int s = 0; s < MR; ++s) {
    const int c = s < m ? piv[s] : 0;
    A[s] = (active && s < m && seatA < m) ? T[c * TP + seatA] : 0.f;
    B[s] = (active && s < m && seatB < m) ? T[c * TP + seatB] : 0.f;
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
      for (int s = 0; s < MR; ++s) T[seatA * TP + s] = A[s];
      sig2[seatA] = sa;
      inv[seatA] = sa > kNegligible ? rsqrtf(sa) : 0.f;
    }
    if (seatB < m) {
#pragma unroll
      for (int s = 0; s < MR; ++s) T[seatB * TP + s] = B[s];
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
