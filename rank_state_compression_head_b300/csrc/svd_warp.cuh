// SVD of the recompression core with one lane group per head: pivoted
// Householder QR K P = Q R, then one-sided Jacobi on the columns of R^T (the
// algorithm of core_factor in recompress_core.cuh, laid out for a group of HW
// lanes instead of a CTA, so that no block barrier is needed).  A group is a
// warp, or a half warp for cores of at most 32 columns (two heads per warp:
// such a core has at most 16 column pairs); every shuffle, vote and warp
// barrier names only the group's lanes.
//
// Pivoted QR: the core sits in the warp's shared square, column c at
// c * TP (TP = MR + 4: the 16-byte chunks of eight consecutive columns fall in
// distinct bank groups); lane l looks after columns l and l + HW.  Each step
// the group picks the remaining column of largest trailing norm (shuffle argmax,
// ties to the lower index), its lanes form the reflector from it (norm in one
// reduction, max-scaled near the fp32 range ends, as householder_qr), and every
// lane applies it to its remaining columns with 16-byte loads and downdates
// their trailing norms (summed in full again once cancellation has eaten most
// of them).  Columns stay in place; only the pivot order is recorded.
//
// Jacobi: lane i (i < P = n'/2) looks after two seats, A and B: lane 0 has
// seat n'-1 in A and the fixed seat 0 in B, lane i >= 1 has seat i in A and
// seat n'-1-i in B.  The columns of R^T stay in the square (column i at
// i * TP); a lane reads the two columns on its seats this round, rotates them in
// registers and writes them back in place (only if it rotated them), one warp
// barrier a round.  Rotation rule, tolerance and stopping rule as jacobi_seats;
// the rotation is applied to scaled columns and the norms are carried from
// round to round (see the loop).
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

template <int MR, int HW>
__device__ int jacobi_warp(int m, float tol, float tol_stop, float *sw);

// One lane group: pivoted QR of the scaled core held in the square T (column c at
// T[c * TP], rows m..MR-1 zero), then Jacobi on R^T.  Leaves in T the columns
// of R^T J by seat (T[seat * TP + s]), sig2/inv by seat, order, piv.  Returns
// the sweeps (or -1).
template <int MR, int HW>
__device__ int svd_warp_core(int m, float tol, float tol_stop, float *sw) {
  using L = SvdWarpSmem<MR>;
  static_assert(HW == 16 || HW == 32, "a lane group is a half warp or a warp");
  static_assert(MR <= 2 * HW, "two columns per lane at most");
  constexpr bool TWO = MR > HW;
  constexpr int RPL = (MR + HW - 1) / HW;  // rows per lane in the reflector
  constexpr int TP = L::TP;
  const int lane = threadIdx.x & (HW - 1);
  const unsigned full = HW == 32 ? 0xffffffffu : 0xffffu << (threadIdx.x & 16);  // my group
  auto gsum = [&](float x) {
#pragma unroll
    for (int o = HW / 2; o > 0; o >>= 1) x += __shfl_xor_sync(full, x, o);
    return x;
  };
  auto gmax = [&](float x) {
#pragma unroll
    for (int o = HW / 2; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(full, x, o));
    return x;
  };
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
  bool done0 = lane >= m, done1 = !TWO || lane + HW >= m;
  float vn0 = done0 ? 0.f : colnorm(lane, 0), vn1 = done1 ? 0.f : colnorm(lane + HW, 0);
  float vr0 = vn0, vr1 = vn1;  // each column's trailing norm when last summed in full
  for (int j = 0; j < m; ++j) {
    float best = -1.f;
    int bi = 1 << 20;
    if (!done0) { best = vn0; bi = lane; }
    if (!done1 && vn1 > best) { best = vn1; bi = lane + HW; }
#pragma unroll
    for (int o = HW / 2; o > 0; o >>= 1) {
      const float ob = __shfl_xor_sync(full, best, o);
      const int oi = __shfl_xor_sync(full, bi, o);
      if (ob > best || (ob == best && oi < bi)) { best = ob; bi = oi; }
    }
    const int pc = bi;
    float *cp = T + pc * TP;
    float a[RPL];
#pragma unroll
    for (int e = 0; e < RPL; ++e) a[e] = lane + HW * e < MR ? cp[lane + HW * e] : 0.f;
    const float alpha = cp[j];
    float tj = 0.f, beta = alpha, sc = 0.f;
    // one reduction for the norm unless it nears the ends of the fp32 range
    // (then scaled by the largest magnitude, as householder_qr)
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < RPL; ++e) {
      const float x = lane + HW * e > j ? a[e] : 0.f;
      ss = fmaf(x, x, ss);
    }
    ss = gsum(ss);
    float amax = 1.f;
    if (!(ss >= 1e-30f && ss <= 1e30f)) {
      amax = 0.f;
#pragma unroll
      for (int e = 0; e < RPL; ++e)
        if (lane + HW * e >= j) amax = fmaxf(amax, fabsf(a[e]));
      amax = gmax(amax);
      ss = 0.f;
      if (amax >= FLT_MIN) {
        const float rinv = 1.f / amax;
#pragma unroll
        for (int e = 0; e < RPL; ++e) {
          const float xs = lane + HW * e > j ? a[e] * rinv : 0.f;
          ss = fmaf(xs, xs, ss);
        }
        ss = gsum(ss);
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
    __syncwarp(full);
    // v_j into the reflector row; the chosen column becomes column j of R (rows
    // above j were finished by the earlier steps, row j is beta, rows below zero)
#pragma unroll
    for (int e = 0; e < RPL; ++e) {
      const int r = lane + HW * e;
      if (r < MR) {
        vrow[r] = r < j ? 0.f : r == j ? 1.f : a[e] * sc;
        if (r >= j) cp[r] = r == j ? beta : 0.f;
      }
    }
    if (lane == 0) piv[j] = pc;
    if (lane == (pc & (HW - 1))) {
      if (pc >= HW) done1 = true;
      else done0 = true;
    }
    __syncwarp(full);
    // the remaining columns: a -= tau (v . a) v, then their norms below row j
#pragma unroll
    for (int h = 0; h < (TWO ? 2 : 1); ++h) {
      if (h == 0 ? done0 : done1) continue;
      float4 *x4 = reinterpret_cast<float4 *>(T + (lane + HW * h) * TP);
      float d = 0.f;
#pragma unroll
      for (int q = 0; q < MR / 4; ++q) {
        const float4 v = v4[q], x = x4[q];
        d = fmaf(v.x, x.x, fmaf(v.y, x.y, fmaf(v.z, x.z, fmaf(v.w, x.w, d))));
      }
      const float t = tj * d;
#pragma unroll
      for (int q = 0; q < MR / 4; ++q) {
        const float4 v = v4[q];
        float4 x = x4[q];
        x.x = fmaf(-t, v.x, x.x); x.y = fmaf(-t, v.y, x.y); x.z = fmaf(-t, v.z, x.z); x.w = fmaf(-t, v.w, x.w);
        x4[q] = x;
      }
      // trailing norm below row j: take row j's square off the old one, and sum
      // it in full again once that has cancelled to below sqrt(eps) of the last
      // full sum (the column downdate of Businger and Golub's pivoted QR)
      const int c = lane + HW * h;
      const float xj = T[c * TP + j];
      float nrm = (h == 0 ? vn0 : vn1) - xj * xj;
      if (nrm <= 3.5e-4f * (h == 0 ? vr0 : vr1)) {
        nrm = colnorm(c, j + 1);
        if (h == 0) vr0 = nrm;
        else vr1 = nrm;
      }
      if (h == 0) vn0 = nrm;
      else vn1 = nrm;
    }
    __syncwarp(full);
  }

  // ---- R^T to the seats of the Jacobi: seat i = row i of R, R column s = T[piv[s] * TP] -------
  const int nn = m + (m & 1), P = nn / 2;
  const bool active = lane < P;
  const int seatA = lane == 0 ? nn - 1 : lane, seatB = lane == 0 ? 0 : nn - 1 - lane;
  {
    float A[MR], B[MR];
#pragma unroll
    for (int s = 0; s < MR; ++s) {
      const int c = s < m ? piv[s] : 0;
      A[s] = (active && s < m && seatA < m) ? T[c * TP + seatA] : 0.f;
      B[s] = (active && s < m && seatB < m) ? T[c * TP + seatB] : 0.f;
    }
    __syncwarp(full);
    if (active) {  // seat s at T[s * TP] from here on (the core is no longer needed)
#pragma unroll
      for (int q = 0; q < MR / 4; ++q) {
        reinterpret_cast<float4 *>(T + seatA * TP)[q] = make_float4(A[4 * q], A[4 * q + 1], A[4 * q + 2], A[4 * q + 3]);
        reinterpret_cast<float4 *>(T + seatB * TP)[q] = make_float4(B[4 * q], B[4 * q + 1], B[4 * q + 2], B[4 * q + 3]);
      }
    }
    __syncwarp(full);
  }

  return jacobi_warp<MR, HW>(m, tol, tol_stop, sw);
}

// One-sided Jacobi with one lane group per head on the seats of the warp's
// square: seat i (i < n', n' = m rounded up to even) holds column i at
// T[i * TP], zero for i >= m.  Leaves the columns of (seats) J in place, their
// squared norms sig2 and reciprocal norms inv by seat, and the seats in order of
// decreasing sigma.  Returns the sweeps run, or -1 at the sweep limit.
template <int MR, int HW>
__device__ int jacobi_warp(int m, float tol, float tol_stop, float *sw) {
  using L = SvdWarpSmem<MR>;
  constexpr int TP = L::TP;
  const int lane = threadIdx.x & (HW - 1);
  const unsigned full = HW == 32 ? 0xffffffffu : 0xffffu << (threadIdx.x & 16);  // my group
  float *T = sw + L::T_OFF, *sig2 = sw + L::S_OFF, *inv = sw + L::I_OFF;
  int *order = reinterpret_cast<int *>(sw + L::O_OFF);
  const int nn = m + (m & 1), P = nn / 2;
  const bool active = lane < P;
  const int seatA = lane == 0 ? nn - 1 : lane, seatB = lane == 0 ? 0 : nn - 1 - lane;

  // ---- Jacobi: the columns of R^T stay where they are (column i at T[i * TP]);
  // each round lane i takes the pair that the round-robin puts on its two seats
  // (the column at seat s >= 1 moves on to s + 1, n'-1 to 1, seat 0 stays) and
  // writes the pair back only if it rotated it.  A column is kept scaled, true
  // column = d * stored, with d and its squared norm in the row's pad
  // (T[i * TP + MR], MR + 1): a rotation [c -s; s c] becomes
  // a' = a - t (d_b / d_a) b, b' = b + t (d_a / d_b) a with both scales times c
  // (one FMA an element instead of two), and the norms move as alpha - t gamma,
  // beta + t gamma (Rutishauser's update).  Norms are summed in full on a
  // sweep's first round and for a norm marked stale (negative) because its
  // update lost more than two bits to cancellation; a pair with a column whose
  // norm is known to be negligible is not read at all.
  int sweeps = 0;
  if (m >= 2) {
    const float tol2 = tol * tol, stop2 = tol_stop * tol_stop;
    int colA = seatA, colB = seatB;  // the pair on my seats this round (>= m: the zero column)
    if (active) {
      *reinterpret_cast<float2 *>(T + seatA * TP + MR) = make_float2(1.f, -1.f);
      *reinterpret_cast<float2 *>(T + seatB * TP + MR) = make_float2(1.f, -1.f);
    }
    __syncwarp(full);
    sweeps = -1;
    for (int sweep = 0; sweep < kMaxSweeps; ++sweep) {
      int far = 0;
      for (int round = 0; round < nn - 1; ++round) {
        if (active) {
          float *ca = T + colA * TP, *cb = T + colB * TP;
          const float2 sa = *reinterpret_cast<const float2 *>(ca + MR);
          const float2 sb = *reinterpret_cast<const float2 *>(cb + MR);
          const bool nega = sa.y >= 0.f && sa.y <= kNegligible, negb = sb.y >= 0.f && sb.y <= kNegligible;
          if (colA < m && colB < m && !nega && !negb) {
            float4 a4[MR / 4], b4[MR / 4];
            const float4 *pa = reinterpret_cast<const float4 *>(ca);
            const float4 *pb = reinterpret_cast<const float4 *>(cb);
            float ga0 = 0.f, ga1 = 0.f;
#pragma unroll
            for (int q = 0; q < MR / 4; ++q) {
              a4[q] = pa[q];
              b4[q] = pb[q];
              ga0 = fmaf(a4[q].x, b4[q].x, fmaf(a4[q].y, b4[q].y, ga0));
              ga1 = fmaf(a4[q].z, b4[q].z, fmaf(a4[q].w, b4[q].w, ga1));
            }
            const float da = sa.x, db = sb.x;
            float al = sa.y, be = sb.y;
            const bool fresh_a = round == 0 || al < 0.f, fresh_b = round == 0 || be < 0.f;
            if (fresh_a) {
              float s0 = 0.f, s1 = 0.f;
#pragma unroll
              for (int q = 0; q < MR / 4; ++q) {
                s0 = fmaf(a4[q].x, a4[q].x, fmaf(a4[q].y, a4[q].y, s0));
                s1 = fmaf(a4[q].z, a4[q].z, fmaf(a4[q].w, a4[q].w, s1));
              }
              al = (s0 + s1) * (da * da);
            }
            if (fresh_b) {
              float s0 = 0.f, s1 = 0.f;
#pragma unroll
              for (int q = 0; q < MR / 4; ++q) {
                s0 = fmaf(b4[q].x, b4[q].x, fmaf(b4[q].y, b4[q].y, s0));
                s1 = fmaf(b4[q].z, b4[q].z, fmaf(b4[q].w, b4[q].w, s1));
              }
              be = (s0 + s1) * (db * db);
            }
            const float ga = (ga0 + ga1) * (da * db);
            if (al > kNegligible && be > kNegligible && ga * ga > tol2 * al * be) {
              const float zeta = (be - al) * __frcp_rn(2.f * ga);
              const float az = fabsf(zeta);
              const float root = az < 1e18f ? az + fmaf(az, az, 1.f) * rsqrtf(fmaf(az, az, 1.f)) : 2.f * az;
              const float t = copysignf(__frcp_rn(root), zeta);
              const float c = rsqrtf(fmaf(t, t, 1.f));
              const float ta = t * db * __frcp_rn(da), tb = t * da * __frcp_rn(db);
              const float tg = t * ga;  // > 0: alpha shrinks, < 0: beta shrinks
              float nal = al - tg, nbe = be + tg;
              if (tg > 0.f && nal < 0.25f * al) nal = -1.f;
              if (tg < 0.f && nbe < 0.25f * be) nbe = -1.f;
              far |= ga * ga > stop2 * al * be;
              float4 *wa = reinterpret_cast<float4 *>(ca);
              float4 *wb = reinterpret_cast<float4 *>(cb);
#pragma unroll
              for (int q = 0; q < MR / 4; ++q) {
                const float4 a = a4[q], b = b4[q];
                wa[q] = make_float4(fmaf(-ta, b.x, a.x), fmaf(-ta, b.y, a.y), fmaf(-ta, b.z, a.z), fmaf(-ta, b.w, a.w));
                wb[q] = make_float4(fmaf(tb, a.x, b.x), fmaf(tb, a.y, b.y), fmaf(tb, a.z, b.z), fmaf(tb, a.w, b.w));
              }
              *reinterpret_cast<float2 *>(ca + MR) = make_float2(c * da, nal);
              *reinterpret_cast<float2 *>(cb + MR) = make_float2(c * db, nbe);
            } else {
              if (fresh_a) ca[MR + 1] = al;
              if (fresh_b) cb[MR + 1] = be;
            }
          }
          if (seatA != 0) colA = colA == 1 ? nn - 1 : colA - 1;
          if (seatB != 0) colB = colB == 1 ? nn - 1 : colB - 1;
        }
        __syncwarp(full);  // the next round's pairs were written by other lanes
      }
      const bool conv = !__any_sync(full, far);
      // fold the scales into the columns: at the end, or once one has shrunk
      // below 2^-20 (each rotation takes at most a factor 1/sqrt(2) off it);
      // after a whole sweep my pair is (seatA, seatB) again
      if (active) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float *col = T + (e == 0 ? seatA : seatB) * TP;
          const float d = col[MR];
          if (conv || sweep + 1 == kMaxSweeps || d < 9.5367e-7f) {
            float4 *c4 = reinterpret_cast<float4 *>(col);
#pragma unroll
            for (int q = 0; q < MR / 4; ++q) {
              const float4 x = c4[q];
              c4[q] = make_float4(x.x * d, x.y * d, x.z * d, x.w * d);
            }
            col[MR] = 1.f;
          }
        }
      }
      __syncwarp(full);
      if (conv) {
        sweeps = sweep + 1;
        break;
      }
    }
  }

  // ---- columns of R^T J (in place: column i at T[i * TP]), sigma^2 ---------------------------
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int j = lane + HW * e;
    if (j < m) {
      const float4 *f4 = reinterpret_cast<const float4 *>(T + j * TP);
      float acc = 0.f;
#pragma unroll
      for (int q = 0; q < MR / 4; ++q) {
        const float4 f = f4[q];
        acc = fmaf(f.x, f.x, fmaf(f.y, f.y, fmaf(f.z, f.z, fmaf(f.w, f.w, acc))));
      }
      sig2[j] = acc;
      inv[j] = acc > kNegligible ? rsqrtf(acc) : 0.f;
    }
  }
  __syncwarp(full);
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int j = lane + HW * e;
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
  __syncwarp(full);
  return sweeps;
}

// ---------------------------------------------------------------------------------------
// One-sided Jacobi with the columns in registers.
//
// Same rotation rule, tolerance, stopping rule, scaled columns and carried norms as
// jacobi_warp; only the pair order and where the columns live differ.  Lane i
// (i < P = n'/2) holds two columns, A and B, in registers.  The order is the
// odd-even transposition order on the n' positions with an exchange after every
// pair (each pair of columns meets exactly once in n' rounds): even rounds pair
// positions (2i, 2i+1), both held by lane i; odd rounds pair (2i+1, 2i+2), one
// column of lane i with one of lane i+1.  An exchange within a lane is only a
// relabelling (which register holds the left position flips every even round),
// so columns move between lanes only in odd rounds, where the left lane of a
// pair decides the rotation and both build the rotated column that lands on
// their own position (jac_round_pair).
// ---------------------------------------------------------------------------------------

struct JacCol {     // metadata of a column held in registers
  float d;          // scale: true column = d * stored
  float n2;         // squared norm of the true column (carried)
};

// Rotation of the pair (x, y) (true columns dx x, dy y with squared norms al, be),
// decided as in jacobi_warp, without branches: a pair left as it is gets the
// coefficients of the identity (ta = tb = tg = 0, c = 1).  Returns whether it rotates.
__device__ inline bool jac_rotation(float dot_xy, const JacCol &x, const JacCol &y, float tol2,
                                    float stop2, float &ta, float &tb, float &c, float &tg, int &far) {
  const float ga = dot_xy * (x.d * y.d);
  const float al = x.n2, be = y.n2;
  const bool rot = al > kNegligible && be > kNegligible && ga * ga > tol2 * al * be;
  // Approximate quotients (about 2^-22 relative): a rotating pair has |2 ga| above
  // 1e-4 kNegligible and the scales lie in [2^-20, 1], far inside their range.  An
  // error of that size in t makes each rotation orthogonal to about 2^-22; over the
  // few hundred rotations a column takes part in, that stays near 1e-6, far below
  // the convergence tolerance.
  // t = sign(zeta) / (|zeta| + sqrt(1 + zeta^2)) with zeta = (be - al) / (2 ga), written
  // as 2 ga sign(be - al) / (|be - al| + sqrt((be - al)^2 + 4 ga^2)): the same root with
  // one quotient fewer on the chain (ga^2 > 0 when the pair rotates; the other branch
  // is discarded by the select)
  const float dba = be - al, dd = fabsf(dba), g2 = 2.f * ga;
  const float r2 = fmaf(dd, dd, g2 * g2);
  const float t = rot ? __fdividef(copysignf(1.f, dba) * g2, dd + r2 * rsqrtf(r2)) : 0.f;
  c = rsqrtf(fmaf(t, t, 1.f));
  ta = t * __fdividef(y.d, x.d);
  tb = t * __fdividef(x.d, y.d);
  tg = t * ga;
  far |= rot && ga * ga > stop2 * al * be;
  return rot;
}

// The register arrays hold a column as MR / 2 pairs of consecutive elements, so that
// the element loops run on the packed two-lane fp32 instructions of sm_100 and later
// (each lane of a packed FMA rounds as a scalar FMA does, in half the issue slots).
// Elements 2k, 2k+1 sit in pair k.
__device__ inline float2 f2(float v) { return make_float2(v, v); }

// Sums of products over a column in four packed accumulators (pair k into k % 4:
// eight chains of element k % 8), so that the dependent chains are short.
template <int MR>
__device__ inline float jac_sum8(float2 (&s)[4]) {
  return ((s[0].x + s[0].y) + (s[1].x + s[1].y)) + ((s[2].x + s[2].y) + (s[3].x + s[3].y));
}

template <int MR>
__device__ inline float jac_norm2(const float2 (&x)[MR / 2], float d) {
  float2 s[4] = {f2(0.f), f2(0.f), f2(0.f), f2(0.f)};
#pragma unroll
  for (int k = 0; k < MR / 2; ++k) s[k & 3] = __ffma2_rn(x[k], x[k], s[k & 3]);
  return jac_sum8<MR>(s) * (d * d);
}

template <int MR>
__device__ inline float jac_dot(const float2 (&x)[MR / 2], const float2 (&y)[MR / 2]) {
  float2 s[4] = {f2(0.f), f2(0.f), f2(0.f), f2(0.f)};
#pragma unroll
  for (int k = 0; k < MR / 2; ++k) s[k & 3] = __ffma2_rn(x[k], y[k], s[k & 3]);
  return jac_sum8<MR>(s);
}

// One even round (the lane's own pair) and one odd round (pairs with the
// neighbours).  RIGHT_A: after the even round the right-facing column is A.
//
// Odd round, pair (x = my right-facing column, y = the right neighbour's
// left-facing one): I receive y into Y and decide the rotation; the neighbour
// receives my decision (ta, c, tg, whether it rotated) and x's metadata by
// shuffles instead of deciding it again, then each side builds the rotated column
// that lands on its own position from the other's old column (y' = y + tb x stays
// on my right, x' = x - ta y goes to the neighbour's left), which needs the old
// columns to cross once more.  So a lane holds three columns, and the pair's dot
// product and coefficients are formed once.
template <int MR, int HW, bool RIGHT_A>
__device__ inline void jac_round_pair(float2 (&A)[MR / 2], float2 (&B)[MR / 2], float2 (&Y)[MR / 2], JacCol &ca,
                                      JacCol &cb, bool has_left, bool has_right, unsigned full, float tol2,
                                      float stop2, int &far) {
  constexpr int NP = MR / 2;
  // ---- even round ----
  {
    float ta, tb, c, tg;
    const bool rot = jac_rotation(jac_dot<MR>(A, B), ca, cb, tol2, stop2, ta, tb, c, tg, far);
    const float2 mta = f2(-ta), ptb = f2(tb);
#pragma unroll
    for (int k = 0; k < NP; ++k) {
      const float2 a = A[k], b = B[k];
      A[k] = __ffma2_rn(mta, b, a);
      B[k] = __ffma2_rn(ptb, a, b);
    }
    const float na = ca.n2 - tg, nb = cb.n2 + tg;
    ca.d *= c;
    cb.d *= c;
    if (rot && na < 0.25f * ca.n2) ca.n2 = jac_norm2<MR>(A, ca.d); else ca.n2 = na;
    if (rot && nb < 0.25f * cb.n2) cb.n2 = jac_norm2<MR>(B, cb.d); else cb.n2 = nb;
  }
  // ---- odd round ----
  float2 (&Xr)[NP] = RIGHT_A ? A : B;   // my right-facing column
  float2 (&Xl)[NP] = RIGHT_A ? B : A;   // my left-facing column
  JacCol &cxr = RIGHT_A ? ca : cb;
  JacCol &cxl = RIGHT_A ? cb : ca;
  float2 s[4] = {f2(0.f), f2(0.f), f2(0.f), f2(0.f)};
#pragma unroll
  for (int k = 0; k < NP; ++k) {
    Y[k].x = __shfl_down_sync(full, Xl[k].x, 1, HW);   // right neighbour's left-facing column
    Y[k].y = __shfl_down_sync(full, Xl[k].y, 1, HW);
    s[k & 3] = __ffma2_rn(Xr[k], Y[k], s[k & 3]);
  }
  JacCol cr;
  cr.d = __shfl_down_sync(full, cxl.d, 1, HW);
  cr.n2 = __shfl_down_sync(full, cxl.n2, 1, HW);
  float ta1, tb1, c1, tg1;
  int far1 = 0;
  const bool rot1 = jac_rotation(jac_sum8<MR>(s), cxr, cr, tol2, stop2, ta1, tb1, c1, tg1, far1);
  far |= has_right && far1;
  // the left neighbour's decision on the pair (its x, my left-facing y), and its x's metadata
  const float ta2 = __shfl_up_sync(full, ta1, 1, HW);
  const float c2 = __shfl_up_sync(full, c1, 1, HW);
  const float tg2 = __shfl_up_sync(full, tg1, 1, HW);
  const bool rot2 = __shfl_up_sync(full, (int)rot1, 1, HW) != 0;
  JacCol cl;
  cl.d = __shfl_up_sync(full, cxr.d, 1, HW);
  cl.n2 = __shfl_up_sync(full, cxr.n2, 1, HW);
  // (lane-predicated, so element by element: a packed update under a per-lane
  // condition costs more registers than it saves)
#pragma unroll
  for (int k = 0; k < NP; ++k) {
    float2 lw;  // left neighbour's old right-facing column
    lw.x = __shfl_up_sync(full, Xr[k].x, 1, HW);
    lw.y = __shfl_up_sync(full, Xr[k].y, 1, HW);
    if (has_right) {
      Xr[k].x = fmaf(tb1, Xr[k].x, Y[k].x);
      Xr[k].y = fmaf(tb1, Xr[k].y, Y[k].y);
    }
    if (has_left) {
      Xl[k].x = fmaf(-ta2, Xl[k].x, lw.x);
      Xl[k].y = fmaf(-ta2, Xl[k].y, lw.y);
    }
  }
  if (has_right) {
    const float ny = cr.n2 + tg1;
    cxr.d = cr.d * c1;
    cxr.n2 = (rot1 && ny < 0.25f * cr.n2) ? jac_norm2<MR>(Xr, cxr.d) : ny;
  }
  if (has_left) {
    const float nx = cl.n2 - tg2;
    cxl.d = cl.d * c2;
    cxl.n2 = (rot2 && nx < 0.25f * cl.n2) ? jac_norm2<MR>(Xl, cxl.d) : nx;
  }
}

// Leaves what jacobi_warp leaves, over all n' seats (the zero column of an odd m
// among them, ranked last): the columns of (seats) J in the square, sig2, inv and
// the order of decreasing sigma.  Returns the sweeps run, or -1 at the sweep limit.
template <int MR, int HW>
__device__ int jacobi_warp_reg(int m, float tol, float tol_stop, float *sw) {
  using L = SvdWarpSmem<MR>;
  constexpr int TP = L::TP;
  static_assert(MR % 4 == 0 && MR <= 2 * HW, "two columns a lane, in registers");
  const int lane = threadIdx.x & (HW - 1);
  const unsigned full = HW == 32 ? 0xffffffffu : 0xffffu << (threadIdx.x & 16);
  float *T = sw + L::T_OFF, *sig2 = sw + L::S_OFF, *inv = sw + L::I_OFF;
  int *order = reinterpret_cast<int *>(sw + L::O_OFF);
  const int nn = m + (m & 1), P = nn / 2;
  const bool active = lane < P;
  const bool has_right = lane + 1 < P, has_left = lane > 0 && active;
  const float tol2 = tol * tol, stop2 = tol_stop * tol_stop;

  float2 A[MR / 2], B[MR / 2], Y[MR / 2];
  {
    const float4 *a4 = reinterpret_cast<const float4 *>(T + (2 * lane) * TP);
    const float4 *b4 = reinterpret_cast<const float4 *>(T + (2 * lane + 1) * TP);
#pragma unroll
    for (int q = 0; q < MR / 4; ++q) {
      const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
      const float4 a = active ? a4[q] : z, b = active ? b4[q] : z;
      A[2 * q] = make_float2(a.x, a.y); A[2 * q + 1] = make_float2(a.z, a.w);
      B[2 * q] = make_float2(b.x, b.y); B[2 * q + 1] = make_float2(b.z, b.w);
    }
  }
  JacCol ca{1.f, 0.f}, cb{1.f, 0.f};
  int sweeps = 0;
  if (m >= 2) {
    sweeps = -1;
    for (int sweep = 0; sweep < kMaxSweeps; ++sweep) {
      ca.n2 = jac_norm2<MR>(A, ca.d);  // norms summed afresh every sweep
      cb.n2 = jac_norm2<MR>(B, cb.d);
      int far = 0;
      // rounds in pairs (even, odd); after an even round at parity 0 the right-facing
      // register is A, at parity 1 it is B: two copies of the pair, fixed at compile time
      for (int rr = 0; rr < P; ++rr) {
        if ((rr & 1) == 0) jac_round_pair<MR, HW, true>(A, B, Y, ca, cb, has_left, has_right, full, tol2, stop2, far);
        else jac_round_pair<MR, HW, false>(A, B, Y, ca, cb, has_left, has_right, full, tol2, stop2, far);
      }
      const bool conv = !__any_sync(full, far);
      // fold the scales into the columns: at the end, or once one has shrunk below 2^-20
      if (conv || sweep + 1 == kMaxSweeps || ca.d < 9.5367e-7f) {
#pragma unroll
        for (int k = 0; k < MR / 2; ++k) A[k] = __fmul2_rn(A[k], f2(ca.d));
        ca.d = 1.f;
      }
      if (conv || sweep + 1 == kMaxSweeps || cb.d < 9.5367e-7f) {
#pragma unroll
        for (int k = 0; k < MR / 2; ++k) B[k] = __fmul2_rn(B[k], f2(cb.d));
        cb.d = 1.f;
      }
      if (conv) {
        sweeps = sweep + 1;
        break;
      }
    }
  }
  // ---- the columns to the seats (lane i: seats 2i, 2i+1), sigma^2, order ---------------------
  if (active) {
#pragma unroll
    for (int q = 0; q < MR / 4; ++q) {
      reinterpret_cast<float4 *>(T + (2 * lane) * TP)[q] = make_float4(A[2 * q].x, A[2 * q].y, A[2 * q + 1].x, A[2 * q + 1].y);
      reinterpret_cast<float4 *>(T + (2 * lane + 1) * TP)[q] = make_float4(B[2 * q].x, B[2 * q].y, B[2 * q + 1].x, B[2 * q + 1].y);
    }
    const float a2 = jac_norm2<MR>(A, 1.f), b2 = jac_norm2<MR>(B, 1.f);
    sig2[2 * lane] = a2;
    sig2[2 * lane + 1] = b2;
    inv[2 * lane] = a2 > kNegligible ? rsqrtf(a2) : 0.f;
    inv[2 * lane + 1] = b2 > kNegligible ? rsqrtf(b2) : 0.f;
  }
  __syncwarp(full);
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int j = lane + HW * e;
    if (j < nn) {
      int rank = 0;
      const float sj = sig2[j];
      for (int i = 0; i < nn; ++i) {
        const float si = sig2[i];
        rank += (si > sj) || (si == sj && i < j);
      }
      order[rank] = j;
    }
  }
  __syncwarp(full);
  return sweeps;
}

}  // namespace seedk
