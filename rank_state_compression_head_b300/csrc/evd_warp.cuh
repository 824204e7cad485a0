// Eigenvectors of a small symmetric positive semi-definite matrix with one lane
// group per head: pivoted Cholesky M = Rt^T Rt, then one-sided Jacobi on the
// columns of Rt^T (the rows of Rt).
//
// Why it gives the eigenvectors: with Rt^T J = V Sigma (Jacobi, J orthogonal),
// M = Rt^T Rt = (Rt^T J)(Rt^T J)^T = V Sigma^2 V^T, so the normalized columns of
// Rt^T J are eigenvectors of M and Sigma^2 its eigenvalues.  The pivoted
// Cholesky plays the part that the column-pivoted QR plays for a core matrix:
// if M = K^T K, then P^T M P = R^T R is the R of K P, and the Jacobi on its graded
// rows needs about half the sweeps that it needs on K itself.
//
// Layout: M (symmetric) comes from global memory, row c at Mg + c * mp (16-byte
// rows): lane l loads rows l and l + HW, which are its columns, straight into
// registers with 16-byte loads, scaled by mscale, zero from m on; the warp's
// shared square (SvdWarpSmem) takes the rows of Rt.  The Schur complement stays in the original index order,
// nothing is swapped: step j picks the remaining index p of largest diagonal;
// the pivot's lane forms row j of Rt (Rt[j][x] = S[x][p] / sqrt(S[p][p]) for the
// remaining x, zero for the pivoted ones) and stores it where column p was, and
// every lane reads it back and updates its remaining columns S[.][c] -=
// Rt[j][.] Rt[j][c].  So Rt's rows are kept in the original column order, and
// the Jacobi's columns give the eigenvectors directly in that order (no
// permutation back).  A diagonal that has fallen to zero or below (rounding)
// gives a zero row.
#pragma once

#include "svd_warp.cuh"

namespace seedk {

// Returns the Jacobi sweeps (or -1); leaves what jacobi_warp leaves, with the
// eigenvector of seat s in T[s * TP + x], x in the original order, and piv.
template <int MR, int HW>
__device__ int evd_warp_core(int m, float tol, float tol_stop, float *sw, const float *Mg, int mp, float mscale) {
  using L = SvdWarpSmem<MR>;
  static_assert(HW == 16 || HW == 32, "a lane group is a half warp or a warp");
  static_assert(MR <= 2 * HW, "two indices per lane at most");
  constexpr bool TWO = MR > HW;
  constexpr int TP = L::TP;
  const int lane = threadIdx.x & (HW - 1);
  const unsigned full = HW == 32 ? 0xffffffffu : 0xffffu << (threadIdx.x & 16);
  float *T = sw + L::T_OFF;
  int *piv = reinterpret_cast<int *>(sw + L::P_OFF);
  const int c0 = lane, c1 = lane + HW;

  // My columns in registers (rows 0..MR-1; rows and columns from m on are zero), as
  // pairs of consecutive rows for the packed fp32 instructions (svd_warp.cuh); all
  // the loads are issued before any is used
  float2 colA[MR / 2], colB[TWO ? MR / 2 : 1];
  bool done0 = c0 >= m, done1 = !TWO || c1 >= m;
  {
    const float4 *a4 = reinterpret_cast<const float4 *>(Mg + (int64_t)(done0 ? 0 : c0) * mp);
    const float4 *b4 = reinterpret_cast<const float4 *>(Mg + (int64_t)(done1 ? 0 : c1) * mp);
    float4 xa[MR / 4], xb[TWO ? MR / 4 : 1];
#pragma unroll
    for (int q = 0; q < MR / 4; ++q) {
      const bool in = 4 * q < mp;
      xa[q] = !done0 && in ? a4[q] : make_float4(0.f, 0.f, 0.f, 0.f);
      if constexpr (TWO) xb[q] = !done1 && in ? b4[q] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    auto keep = [&](float v, int x) { return x < m ? v * mscale : 0.f; };
#pragma unroll
    for (int q = 0; q < MR / 4; ++q) {
      colA[2 * q] = make_float2(keep(xa[q].x, 4 * q), keep(xa[q].y, 4 * q + 1));
      colA[2 * q + 1] = make_float2(keep(xa[q].z, 4 * q + 2), keep(xa[q].w, 4 * q + 3));
      if constexpr (TWO) {
        colB[2 * q] = make_float2(keep(xb[q].x, 4 * q), keep(xb[q].y, 4 * q + 1));
        colB[2 * q + 1] = make_float2(keep(xb[q].z, 4 * q + 2), keep(xb[q].w, 4 * q + 3));
      }
    }
  }
  float dg0 = done0 ? 0.f : Mg[(int64_t)c0 * mp + c0] * mscale;
  float dg1 = done1 ? 0.f : Mg[(int64_t)(TWO ? c1 : 0) * mp + (TWO ? c1 : 0)] * mscale;
  // rows already pivoted (and rows from m on), the same in every lane
  uint64_t gone = m >= 64 ? 0ull : ~0ull << m;
  __syncwarp(full);
  // order-preserving integer key of a finite float (larger float, larger key; 0 = none)
  auto okey = [](float f) {
    const unsigned u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  };
  const int gbase = threadIdx.x & (32 - HW);  // first lane of my group in the warp
  for (int j = 0; j < m; ++j) {
    // the remaining index of largest diagonal (ties to the lower index): one warp
    // reduction of the keys, then the lowest lane holding the maximum, first among the
    // lower indices l, then among l + HW
    const unsigned k0 = done0 ? 0u : okey(dg0), k1 = done1 ? 0u : okey(dg1);
    const unsigned kmax = __reduce_max_sync(full, k0 > k1 ? k0 : k1);
    const unsigned b0 = (__ballot_sync(full, !done0 && k0 == kmax) >> gbase) & (HW == 32 ? 0xffffffffu : 0xffffu);
    const unsigned b1 = (__ballot_sync(full, !done1 && k1 == kmax) >> gbase) & (HW == 32 ? 0xffffffffu : 0xffffu);
    const int p = b0 ? __ffs(b0) - 1 : HW + __ffs(b1) - 1;
    const float best = __uint_as_float((kmax & 0x80000000u) ? (kmax ^ 0x80000000u) : ~kmax);
    const float d = fmaxf(best, 0.f);
    const float inv = d > 0.f ? rsqrtf(d) : 0.f;  // 1 / r_jj (a couple of ulp)
    float *row = T + p * TP;  // row j of Rt goes where column p was
    // The pivot's lane stores its column as it stands; then every lane turns its own
    // two entries into those of row j of Rt: Rt[j][x] = S[x][p] / r_jj for the rows not
    // yet pivoted (r_jj at x = p), zero for the others.
    if (lane == (p & (HW - 1))) {
      if (TWO && p >= HW) {
#pragma unroll
        for (int q = 0; q < MR / 4; ++q)
          reinterpret_cast<float4 *>(row)[q] =
              make_float4(colB[TWO ? 2 * q : 0].x, colB[TWO ? 2 * q : 0].y, colB[TWO ? 2 * q + 1 : 0].x, colB[TWO ? 2 * q + 1 : 0].y);
        done1 = true;
      } else {
#pragma unroll
        for (int q = 0; q < MR / 4; ++q)
          reinterpret_cast<float4 *>(row)[q] = make_float4(colA[2 * q].x, colA[2 * q].y, colA[2 * q + 1].x, colA[2 * q + 1].y);
        done0 = true;
      }
    }
    __syncwarp(full);
    if (c0 < MR) row[c0] = (gone >> c0) & 1ull ? 0.f : row[c0] * inv;
    if (TWO && c1 < MR) row[c1] = (gone >> c1) & 1ull ? 0.f : row[c1] * inv;
    gone |= 1ull << p;
    __syncwarp(full);
    // Schur update of my remaining columns: S[x][c] -= Rt[j][x] Rt[j][c]
    const float4 *r4 = reinterpret_cast<const float4 *>(row);
    const float t0 = done0 ? 0.f : row[c0];
    const float t1 = done1 ? 0.f : row[TWO ? c1 : 0];
    // (v (-t) rounds as (-v) t: the sign is exact)
    const float2 mt0 = make_float2(-t0, -t0), mt1 = make_float2(-t1, -t1);
#pragma unroll
    for (int q = 0; q < MR / 4; ++q) {
      const float4 v = r4[q];
      const float2 v01 = make_float2(v.x, v.y), v23 = make_float2(v.z, v.w);
      colA[2 * q] = __ffma2_rn(v01, mt0, colA[2 * q]);
      colA[2 * q + 1] = __ffma2_rn(v23, mt0, colA[2 * q + 1]);
      if constexpr (TWO) {
        colB[2 * q] = __ffma2_rn(v01, mt1, colB[2 * q]);
        colB[2 * q + 1] = __ffma2_rn(v23, mt1, colB[2 * q + 1]);
      }
    }
    dg0 = fmaf(-t0, t0, dg0);
    if (TWO) dg1 = fmaf(-t1, t1, dg1);
    if (lane == 0) piv[j] = p;
    __syncwarp(full);  // row j has been read by every lane
  }

  // ---- rows of Rt to the Jacobi seats: seat s = column piv[s] -----------------------------
  const int nn = m + (m & 1), P = nn / 2;
  const bool active = lane < P;
  const int seatA = lane == 0 ? nn - 1 : lane, seatB = lane == 0 ? 0 : nn - 1 - lane;
  {
    float4 A[MR / 4], B[MR / 4];
    const float4 *sa = reinterpret_cast<const float4 *>(T + (seatA < m ? piv[seatA] : 0) * TP);
    const float4 *sb = reinterpret_cast<const float4 *>(T + (seatB < m ? piv[seatB] : 0) * TP);
#pragma unroll
    for (int q = 0; q < MR / 4; ++q) {
      const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
      A[q] = (active && seatA < m) ? sa[q] : z;
      B[q] = (active && seatB < m) ? sb[q] : z;
    }
    __syncwarp(full);
    if (active) {
#pragma unroll
      for (int q = 0; q < MR / 4; ++q) {
        reinterpret_cast<float4 *>(T + seatA * TP)[q] = A[q];
        reinterpret_cast<float4 *>(T + seatB * TP)[q] = B[q];
      }
    }
    __syncwarp(full);
  }
  // the columns in registers (three MR-float arrays a lane)
  return jacobi_warp_reg<MR, HW>(m, tol, tol_stop, sw);
}

}  // namespace seedk
