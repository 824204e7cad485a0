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
// Layout: M sits in the warp's shared square (SvdWarpSmem), column c at
// T[c * TP], rows and columns m..MR-1 zero; lane l looks after indices l and
// l + HW.  The Schur complement stays in the original index order, nothing is
// swapped: step j picks the remaining index p of largest diagonal, forms row j
// of Rt (Rt[j][x] = S[x][p] / sqrt(S[p][p]) for the remaining x, zero for the
// pivoted ones), updates the remaining columns S[.][c] -= Rt[j][.] Rt[j][c], and
// then stores row j of Rt in column p, which is no longer needed.  So Rt's rows
// are kept in the original column order, and the Jacobi's columns give the
// eigenvectors directly in that order (no permutation back).  A diagonal that
// has fallen to zero or below (rounding) gives a zero row.
#pragma once

#include "svd_warp.cuh"

namespace seedk {

// Returns the Jacobi sweeps (or -1); leaves what jacobi_warp leaves, with the
// eigenvector of seat s in T[s * TP + x], x in the original order, and piv.
template <int MR, int HW>
__device__ int evd_warp_core(int m, float tol, float tol_stop, float *sw) {
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

  bool done0 = c0 >= m, done1 = !TWO || c1 >= m;
  float dg0 = done0 ? 0.f : T[c0 * TP + c0];
  float dg1 = done1 ? 0.f : T[c1 * TP + c1];
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
    float *cp = T + p * TP;
    if (lane == (p & (HW - 1))) {
      if (p >= HW) done1 = true;
      else done0 = true;
    }
    // Schur update of my remaining columns: S[.][c] -= (S[.][p] / rjj) (S[c][p] / rjj)
    const float4 *p4 = reinterpret_cast<const float4 *>(cp);
#pragma unroll
    for (int e = 0; e < (TWO ? 2 : 1); ++e) {
      if (e == 0 ? done0 : done1) continue;
      const int c = e == 0 ? c0 : c1;
      const float t = cp[c] * inv * inv;
      float4 *x4 = reinterpret_cast<float4 *>(T + c * TP);
#pragma unroll
      for (int q = 0; q < MR / 4; ++q) {
        const float4 v = p4[q];
        float4 x = x4[q];
        x.x = fmaf(-t, v.x, x.x); x.y = fmaf(-t, v.y, x.y); x.z = fmaf(-t, v.z, x.z); x.w = fmaf(-t, v.w, x.w);
        x4[q] = x;
      }
      if (e == 0) dg0 = T[c * TP + c];
      else dg1 = T[c * TP + c];
    }
    __syncwarp(full);  // column p has been read by every lane
    // column p becomes row j of Rt: my two entries of it (zero where already pivoted,
    // including p itself before this step's flag; Rt[j][p] = S[p][p] / rjj = rjj)
#pragma unroll
    for (int e = 0; e < (TWO ? 2 : 1); ++e) {
      const int x = e == 0 ? c0 : c1;
      if (x < MR) {
        const bool was_done = x == p ? false : (e == 0 ? done0 : done1);
        cp[x] = was_done ? 0.f : cp[x] * inv;
      }
    }
    if (lane == 0) piv[j] = p;
    __syncwarp(full);
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
