// Householder QR of a factor panel with the panel held in registers.
//
// TPC threads per column (TPC = 4 here): thread part p < TPC of column l holds
// rows 4c..4c+3 of the column for the chunks c = p + TPC i, i < rows / (4 TPC).
//
// Factorization (one barrier per step j): the warp that holds column j turns
// it into the reflector together - the owners lay the column out in V[j]
// (shared), the 32 lanes form amax, the scaled norm and v_j (v_j[j] = 1, zeros
// above) in place and keep beta = R[j][j] beside it.
// After the barrier every later column takes v_j . a_l over its rows (two
// shuffles join the parts) and subtracts tau_j (v_j . a_l) v_j in its
// registers.  The panel itself never goes through shared memory; V keeps all
// reflectors, so that they can be applied to other vectors afterwards
// (rr_apply, rr_apply2).
//
// The reflector is the one of householder_qr (zero below the smallest normal
// float); its norm is taken unscaled unless the sum of squares nears the ends
// of the fp32 range, where it is scaled by the column's largest magnitude as in
// householder_qr.  The result differs from householder_qr only in rounding.
#pragma once

#include "common.cuh"

#include <float.h>

namespace seedk {

constexpr int kTPC = 4;                   // threads per column
constexpr int kRRChunks = 128 / (4 * kTPC);  // float4 chunks per thread for a 128-row panel

// My part of a column: chunks i < nch (nch = rows / (4 TPC)) are in use.
struct RRCol {
  float4 x[kRRChunks];
  int nch;
};

__device__ inline int rr_row(int p, int i, int e) { return 4 * (p + kTPC * i) + e; }
__device__ inline float f4get(const float4 &v, int e) { return e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w; }

// Step j of the factorization, run by every lane of the warp that holds column
// j (owner: the kTPC lanes of column j).  vj: V[j] (rows floats); on exit it holds
// v_j, *tau = tau_j and *beta_out = beta (R[j][j]).  The owners' registers are
// left as they were: rows above j already hold R, and nothing reads the rest.
__device__ inline void rr_reflector_warp(const RRCol &c, bool owner, int p, int j, int rows, float *vj,
                                         float *tau, float *beta_out) {
  const int lane = threadIdx.x & 31;
  if (owner) {
#pragma unroll
    for (int i = 0; i < kRRChunks; ++i) {
      if (i >= c.nch) break;
      reinterpret_cast<float4 *>(vj)[p + kTPC * i] = c.x[i];
    }
  }
  __syncwarp();
  // lane k holds rows [k * rpl, (k + 1) * rpl), rpl = rows / 32 (4 or 2)
  const int rpl = rows >> 5;
  float a[4] = {0.f, 0.f, 0.f, 0.f};
  if (rpl == 4) {  // one 16-byte (or 8-byte) access per lane: no bank conflicts
    const float4 t = reinterpret_cast<const float4 *>(vj)[lane];
    a[0] = t.x; a[1] = t.y; a[2] = t.z; a[3] = t.w;
  } else {
    const float2 t = reinterpret_cast<const float2 *>(vj)[lane];
    a[0] = t.x; a[1] = t.y;
  }
  const float alpha = vj[j];
  float tj = 0.f, beta = alpha, sc = 0.f;
  // The sum of squares below row j in one reduction; only where it leaves
  // [1e-30, 1e30] (entries near the ends of the fp32 range) is it formed again
  // from the column scaled by its largest magnitude.
  float ss = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float x = (e < rpl && lane * rpl + e > j) ? a[e] : 0.f;
    ss = fmaf(x, x, ss);
  }
  ss = warp_sum(ss);
  float amax = 1.f;
  if (!(ss >= 1e-30f && ss <= 1e30f)) {
    amax = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (e < rpl && lane * rpl + e >= j) amax = fmaxf(amax, fabsf(a[e]));
    amax = warp_max(amax);
    ss = 0.f;
    if (amax >= FLT_MIN) {
      const float inv = 1.f / amax;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float xs = (e < rpl && lane * rpl + e > j) ? a[e] * inv : 0.f;
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
    sc = 1.f / ((as - bs) * amax);  // v_i = x_i / (alpha - beta), |v_i| <= 1
    beta = bs * amax;
  }
  __syncwarp();
  float w[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int row = lane * rpl + e;
    w[e] = row < j ? 0.f : row == j ? 1.f : a[e] * sc;
  }
  if (rpl == 4) reinterpret_cast<float4 *>(vj)[lane] = make_float4(w[0], w[1], w[2], w[3]);
  else reinterpret_cast<float2 *>(vj)[lane] = make_float2(w[0], w[1]);
  if (lane == 0) {
    *tau = tj;
    *beta_out = beta;
  }
}

// a_l -= tau (v . a_l) v over my rows.  All kTPC lanes of the column call it
// (pmask: those lanes).
__device__ inline void rr_apply(RRCol &c, int p, const float *v, float tau, unsigned pmask) {
  const float4 *v4 = reinterpret_cast<const float4 *>(v);
  float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
  for (int i = 0; i < kRRChunks; ++i) {
    if (i >= c.nch) break;
    const float4 w = v4[p + kTPC * i];
    s0 = fmaf(w.x, c.x[i].x, s0); s1 = fmaf(w.y, c.x[i].y, s1);
    s2 = fmaf(w.z, c.x[i].z, s2); s3 = fmaf(w.w, c.x[i].w, s3);
  }
  float dot = (s0 + s1) + (s2 + s3);
#pragma unroll
  for (int o = 1; o < kTPC; o <<= 1) dot += __shfl_xor_sync(pmask, dot, o);
  const float sv = tau * dot;
  // read v again rather than keeping a second copy of the chunk in registers
  asm volatile("" ::: "memory");
#pragma unroll
  for (int i = 0; i < kRRChunks; ++i) {
    if (i >= c.nch) break;
    const float4 w = v4[p + kTPC * i];
    c.x[i].x = fmaf(-sv, w.x, c.x[i].x); c.x[i].y = fmaf(-sv, w.y, c.x[i].y);
    c.x[i].z = fmaf(-sv, w.z, c.x[i].z); c.x[i].w = fmaf(-sv, w.w, c.x[i].w);
  }
}

// a_l <- H_a H_b a_l for two reflectors at once (H = I - tau v v^T, g = v_a . v_b):
// with d_b = v_b . a_l and d_a = v_a . a_l, H_b first takes x_b = tau_b d_b of
// v_b off, which leaves v_a . a_l = d_a - x_b g, so H_a takes x_a = tau_a (d_a -
// x_b g) of v_a.  The two dot products and their reductions run side by side.
__device__ inline void rr_apply2(RRCol &c, int p, const float *va, const float *vb, float tau_a, float tau_b,
                                 float g, unsigned pmask) {
  const float4 *a4 = reinterpret_cast<const float4 *>(va);
  const float4 *b4 = reinterpret_cast<const float4 *>(vb);
  float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
#pragma unroll
  for (int i = 0; i < kRRChunks; ++i) {
    if (i >= c.nch) break;
    const float4 wa = a4[p + kTPC * i], wb = b4[p + kTPC * i];
    a0 = fmaf(wa.x, c.x[i].x, fmaf(wa.y, c.x[i].y, a0)); a1 = fmaf(wa.z, c.x[i].z, fmaf(wa.w, c.x[i].w, a1));
    b0 = fmaf(wb.x, c.x[i].x, fmaf(wb.y, c.x[i].y, b0)); b1 = fmaf(wb.z, c.x[i].z, fmaf(wb.w, c.x[i].w, b1));
  }
  float da = a0 + a1, db = b0 + b1;
#pragma unroll
  for (int o = 1; o < kTPC; o <<= 1) {
    da += __shfl_xor_sync(pmask, da, o);
    db += __shfl_xor_sync(pmask, db, o);
  }
  const float xb = tau_b * db;
  const float xa = tau_a * fmaf(-xb, g, da);
  asm volatile("" ::: "memory");
#pragma unroll
  for (int i = 0; i < kRRChunks; ++i) {
    if (i >= c.nch) break;
    const float4 wa = a4[p + kTPC * i], wb = b4[p + kTPC * i];
    c.x[i].x = fmaf(-xa, wa.x, fmaf(-xb, wb.x, c.x[i].x)); c.x[i].y = fmaf(-xa, wa.y, fmaf(-xb, wb.y, c.x[i].y));
    c.x[i].z = fmaf(-xa, wa.z, fmaf(-xb, wb.z, c.x[i].z)); c.x[i].w = fmaf(-xa, wa.w, fmaf(-xb, wb.w, c.x[i].w));
  }
}

}  // namespace seedk
