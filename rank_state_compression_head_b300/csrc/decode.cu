// Fused read-out + exact factored update (one decode step of every head).
//
// "Shallow Encoding Emits Deep Memories", picx.dev summary, Methodology >
// Exact Update (Lemma 2): the sink + low-rank form is closed under the Gated
// DeltaNet, Kimi Delta Attention and Mamba-2 updates; each step appends
// columns to the factors.  thelatestinai.com list view, Table 1 (decode
// column): every step reads out and updates each recurrent state.
//
// One CTA per head.  The kernel streams the head's m stored columns of U and
// W from HBM exactly once (16-byte loads, all issued up front so that a head's
// whole factor block is in flight), computes
//     x_k = U_eff^T k  and  x_q = U_eff^T q           (one pass over U)
//     W x_k and W x_q                                   (one pass over W)
// reduces through shared memory, and writes the appended column(s), the new
// sink coefficient, the column (or row) scales and the read-out.  Existing
// columns are never rewritten: the gate of existing columns lives in fp32
// scales, so each stored bf16 column is rounded exactly once.
#include "common.cuh"

namespace seedk {

struct DecodeArgs {
  StateView sv;
  const float *q, *k, *v, *gate, *beta, *A;
  float *o;
};

template <int VAR, typename TF, int DV, int MAXC, int NW>
__global__ void __launch_bounds__(NW * 32) decode_kernel(const DecodeArgs p) {
  constexpr int DK = kDK;
  constexpr int NT = NW * 32;
  constexpr int EPL = Elem<TF>::kPer16B;   // elements in one 16-byte chunk
  constexpr int LPC_U = DK / EPL;          // lanes covering one U column
  constexpr int CPL_U = 32 / LPC_U;        // U columns per warp-wide load
  constexpr int LPC_W = DV / EPL;
  constexpr int CPL_W = 32 / LPC_W;
  constexpr int NLU = (MAXC + CPL_U * NW - 1) / (CPL_U * NW);
  constexpr int NLW = (MAXC + CPL_W * NW - 1) / (CPL_W * NW);
  constexpr int NGW = NW * CPL_W;          // partial groups of the W pass
  constexpr bool KDA = VAR == SEED_KDA;
  constexpr bool M2 = VAR == SEED_MAMBA2;
  constexpr int NX = M2 ? 1 : 2;           // mat-vecs per pass: (x_k, x_q) or x_q alone
  constexpr int NS = 8;                    // block-reduced scalars
  static_assert(NT >= DK && NT >= DV, "one thread per state row / column");
  static_assert(NX * MAXC <= NT, "one thread per (column, mat-vec) in the U reduction");

  __shared__ __align__(16) float part[MAXC][LPC_U][NX];
  __shared__ __align__(16) float xs[NX][MAXC];
  __shared__ __align__(16) float red[NGW][NX][DV];
  __shared__ float scal[NW][NS];

  const int h = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const StateView &sv = p.sv;
  const int r_h = sv.rank_of(h);
  const int m = r_h + sv.growth * sv.steps;
  if (r_h < 0 || m > MAXC) {  // rank table disagrees with r_max: touch nothing
    if (tid == 0 && sv.status) sv.status[h] = SEED_ERR_INVALID_ARG;
    return;
  }
  const int64_t c0 = sv.col0(h);
  const int dir = sv.dir_of(h);
  const TF *Uh = reinterpret_cast<const TF *>(sv.U) + c0 * DK;
  const TF *Wh = reinterpret_cast<const TF *>(sv.W) + c0 * DV;

  // ---- 1. put the whole factor block of this head in flight ----------------
  uint4 ureg[NLU], wreg[NLW];
#pragma unroll
  for (int L = 0; L < NLU; ++L) {
    const int col = (L * NW + warp) * CPL_U + lane / LPC_U;
    ureg[L] = make_uint4(0, 0, 0, 0);
    if (col < m) ureg[L] = ld_stream16(Uh + (int64_t)col * DK + (lane % LPC_U) * EPL);
  }
#pragma unroll
  for (int L = 0; L < NLW; ++L) {
    const int col = (L * NW + warp) * CPL_W + lane / LPC_W;
    wreg[L] = make_uint4(0, 0, 0, 0);
    if (col < m) wreg[L] = ld_stream16(Wh + (int64_t)col * DV + (lane % LPC_W) * EPL);
  }

  // ---- 2. per-thread inputs -------------------------------------------------
  const float *qh = p.q + (int64_t)h * DK;   // Mamba-2: C
  const float *kh = p.k + (int64_t)h * DK;   // Mamba-2: B
  const float *vh = p.v + (int64_t)h * DV;   // Mamba-2: x
  const float *vb = sv.vbar + (int64_t)dir * DV;
  float *ah = sv.a + (int64_t)h * DK;

  // gates
  float g = 0.f, beta = 0.f, dt = 0.f;
  if (VAR == SEED_GDN) { g = p.gate[h]; beta = p.beta[h]; }
  if (KDA) { beta = p.beta[h]; }
  if (M2) { dt = p.gate[h]; g = expf(dt * p.A[dir]); }

  // row slice [r0, r0 + EPL) of the U pass, with the vectors it contracts against
  const int r0 = (lane % LPC_U) * EPL;
  float kx[EPL], qx[EPL];
#pragma unroll
  for (int e = 0; e < EPL; e += 4) {
    const float4 q4 = *reinterpret_cast<const float4 *>(qh + r0 + e);
    const float4 k4 = *reinterpret_cast<const float4 *>(kh + r0 + e);
    qx[e] = q4.x; qx[e + 1] = q4.y; qx[e + 2] = q4.z; qx[e + 3] = q4.w;
    kx[e] = k4.x; kx[e + 1] = k4.y; kx[e + 2] = k4.z; kx[e + 3] = k4.w;
  }
  if (KDA) {  // x_k = U^T (D k), x_q = U^T (D' q) with D' = alpha D
    const float *Dh = sv.scale + (int64_t)h * DK;
    const float *al = p.gate + (int64_t)h * DK;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      const float d = Dh[r0 + e];
      kx[e] *= d;
      qx[e] *= al[r0 + e] * d;
    }
  }

  // element phase inputs: thread t owns row t (< DK) and value column t (< DV)
  float kt = 0.f, qt = 0.f, at = 0.f, vt = 0.f, vbt = 0.f, alt = 0.f, Dt = 0.f;
  float unew0 = 0.f, unew1 = 0.f;  // stored (rounded) values of the appended U column(s) at row t
  float s[NS];
#pragma unroll
  for (int i = 0; i < NS; ++i) s[i] = 0.f;
  if (tid < DK) {
    kt = kh[tid]; qt = qh[tid]; at = ah[tid];
    if (VAR == SEED_GDN) {
      unew0 = Elem<TF>::round(kt);
      s[0] = kt * at; s[1] = qt * at; s[2] = kt * qt; s[3] = unew0 * qt;
    } else if (KDA) {
      alt = p.gate[(int64_t)h * DK + tid];
      Dt = sv.scale[(int64_t)h * DK + tid];
      const float Dn = alt * Dt;
      unew0 = Elem<TF>::round(kt / Dt);
      unew1 = Elem<TF>::round(kt / Dn);
      s[0] = kt * at; s[1] = alt * at * qt; s[2] = alt * kt * qt; s[3] = kt * qt;
      s[6] = unew0 * Dn * qt; s[7] = unew1 * Dn * qt;
    } else {
      unew0 = Elem<TF>::round(dt * kt);
      s[0] = at * qt; s[1] = kt * qt; s[2] = unew0 * qt;
    }
  }
  if (tid < DV) {
    vt = vh[tid]; vbt = vb[tid];
    s[4] = vt * vbt; s[5] = vbt * vbt;
  }
#pragma unroll
  for (int i = 0; i < NS; ++i) {
    const float r = warp_sum(s[i]);
    if (lane == 0) scal[warp][i] = r;
  }

  // ---- 3. U pass: partial dot products of each column with k and q ----------
#pragma unroll
  for (int L = 0; L < NLU; ++L) {
    const int col = (L * NW + warp) * CPL_U + lane / LPC_U;
    float x[EPL];
    Elem<TF>::unpack(ureg[L], x);
    float pk = 0.f, pq = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      if (!M2) pk = fmaf(x[e], kx[e], pk);
      pq = fmaf(x[e], qx[e], pq);
    }
    if (col < m) {
      if (M2) {
        part[col][lane % LPC_U][0] = pq;
      } else {
        part[col][lane % LPC_U][0] = pk;
        part[col][lane % LPC_U][1] = pq;
      }
    }
  }
  __syncthreads();

  if (tid < NX * m) {
    const int col = tid / NX, which = tid % NX;
    float acc = 0.f;
#pragma unroll
    for (int sub = 0; sub < LPC_U; ++sub) acc += part[col][sub][which];
    if (!KDA) acc *= sv.scale[c0 + col];
    xs[which][col] = acc;
  }
  float S[NS];
#pragma unroll
  for (int i = 0; i < NS; ++i) {
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) acc += scal[w][i];
    S[i] = acc;
  }
  __syncthreads();

  // ---- 4. W pass: W x_k and W x_q ------------------------------------------
  {
    float acc[NX][EPL];
#pragma unroll
    for (int j = 0; j < NX; ++j)
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[j][e] = 0.f;
#pragma unroll
    for (int L = 0; L < NLW; ++L) {
      const int col = (L * NW + warp) * CPL_W + lane / LPC_W;
      if (col < m) {
        float x[EPL];
        Elem<TF>::unpack(wreg[L], x);
#pragma unroll
        for (int j = 0; j < NX; ++j) {
          const float xv = xs[j][col];
#pragma unroll
          for (int e = 0; e < EPL; ++e) acc[j][e] = fmaf(x[e], xv, acc[j][e]);
        }
      }
    }
    const int grp = warp * CPL_W + lane / LPC_W;
    const int rw = (lane % LPC_W) * EPL;
#pragma unroll
    for (int j = 0; j < NX; ++j)
#pragma unroll
      for (int e = 0; e < EPL; e += 4)
        *reinterpret_cast<float4 *>(&red[grp][j][rw + e]) =
            make_float4(acc[j][e], acc[j][e + 1], acc[j][e + 2], acc[j][e + 3]);
  }
  __syncthreads();

  // ---- 5. update and read-out ----------------------------------------------
  const float omega = S[4] / S[5];
  int bad = 0;
  TF *Uo = reinterpret_cast<TF *>(sv.U) + (c0 + m) * DK;
  TF *Wo = reinterpret_cast<TF *>(sv.W) + (c0 + m) * DV;

  if (VAR == SEED_GDN) {
    // a' = g a + beta (omega - g k.a) k ;  a'.q = g a.q + beta (omega - g k.a) k.q
    const float coef = beta * (omega - g * S[0]);
    const float aq = fmaf(g, S[1], coef * S[2]);
    if (tid < DK) {
      const float an = fmaf(g, at, coef * kt);
      ah[tid] = an;
      Elem<TF>::store(Uo + tid, kt);
      bad |= !finite(an);
    }
    if (tid < DV) {
      float wxk = 0.f, wxq = 0.f;
#pragma unroll
      for (int grp = 0; grp < NGW; ++grp) { wxk += red[grp][0][tid]; wxq += red[grp][1][tid]; }
      const float eps = fmaf(-omega, vbt, vt);
      const float wn = Elem<TF>::round(beta * fmaf(-g, wxk, eps));
      Elem<TF>::store(Wo + tid, wn);
      const float o = fmaf(vbt, aq, fmaf(g, wxq, S[3] * wn));
      p.o[(int64_t)h * DV + tid] = o;
      bad |= !finite(o);
    }
    if (tid < m) sv.scale[c0 + tid] *= g;
    if (tid == m) sv.scale[c0 + m] = 1.f;
  } else if (KDA) {
    // a' = alpha (a - beta k (k.a)) + beta omega k ; D' = alpha D
    const float aq = S[1] - beta * S[0] * S[2] + beta * omega * S[3];
    if (tid < DK) {
      const float an = alt * fmaf(-beta * kt, S[0], at) + beta * omega * kt;
      ah[tid] = an;
      sv.scale[(int64_t)h * DK + tid] = alt * Dt;
      Elem<TF>::store(Uo + tid, unew0);
      Elem<TF>::store(Uo + DK + tid, unew1);
      bad |= !finite(an);
    }
    if (tid < DV) {
      float wxk = 0.f, wxq = 0.f;
#pragma unroll
      for (int grp = 0; grp < NGW; ++grp) { wxk += red[grp][0][tid]; wxq += red[grp][1][tid]; }
      const float eps = fmaf(-omega, vbt, vt);
      const float w1 = Elem<TF>::round(-beta * wxk);
      const float w2 = Elem<TF>::round(beta * eps);
      Elem<TF>::store(Wo + tid, w1);
      Elem<TF>::store(Wo + DV + tid, w2);
      const float o = fmaf(vbt, aq, wxq + w1 * S[6] + w2 * S[7]);
      p.o[(int64_t)h * DV + tid] = o;
      bad |= !finite(o);
    }
  } else {
    // Mamba-2: a' = g a + dt omega B ; y = xbar (a'.C) + g W x_C + (u_new.C) w_new
    const float coef = dt * omega;
    const float aC = fmaf(g, S[0], coef * S[1]);
    if (tid < DK) {
      const float an = fmaf(g, at, coef * kt);
      ah[tid] = an;
      Elem<TF>::store(Uo + tid, unew0);
      bad |= !finite(an);
    }
    if (tid < DV) {
      float wxq = 0.f;
#pragma unroll
      for (int grp = 0; grp < NGW; ++grp) wxq += red[grp][0][tid];
      const float wn = Elem<TF>::round(fmaf(-omega, vbt, vt));
      Elem<TF>::store(Wo + tid, wn);
      const float o = fmaf(vbt, aC, fmaf(g, wxq, S[2] * wn));
      p.o[(int64_t)h * DV + tid] = o;
      bad |= !finite(o);
    }
    if (tid < m) sv.scale[c0 + tid] *= g;
    if (tid == m) sv.scale[c0 + m] = 1.f;
  }
  bad = __syncthreads_or(bad);
  if (tid == 0 && sv.status) sv.status[h] = bad ? SEED_ERR_NONFINITE : SEED_OK;
}

template <int VAR, typename TF, int DV, int MAXC>
static cudaError_t launch_decode_t(const DecodeArgs &a, cudaStream_t s) {
  constexpr int NW = (sizeof(TF) == 4 && MAXC > 32) ? 8 : 4;
  decode_kernel<VAR, TF, DV, MAXC, NW><<<a.sv.n_heads, NW * 32, 0, s>>>(a);
  return cudaGetLastError();
}

template <int VAR, typename TF, int DV>
static cudaError_t launch_decode_c(const DecodeArgs &a, int cols_max, cudaStream_t s) {
  if (cols_max <= 16) return launch_decode_t<VAR, TF, DV, 16>(a, s);
  if (cols_max <= 32) return launch_decode_t<VAR, TF, DV, 32>(a, s);
  return launch_decode_t<VAR, TF, DV, 64>(a, s);
}

template <int VAR, typename TF>
static cudaError_t launch_decode_d(const DecodeArgs &a, int cols_max, cudaStream_t s) {
  if (a.sv.d_v == 64) return launch_decode_c<VAR, TF, 64>(a, cols_max, s);
  return launch_decode_c<VAR, TF, 128>(a, cols_max, s);
}

template <typename TF>
static cudaError_t launch_decode_v(const DecodeArgs &a, int cols_max, cudaStream_t s) {
  switch (a.sv.variant) {
    case SEED_GDN: return launch_decode_d<SEED_GDN, TF>(a, cols_max, s);
    case SEED_KDA: return launch_decode_d<SEED_KDA, TF>(a, cols_max, s);
    default: return launch_decode_d<SEED_MAMBA2, TF>(a, cols_max, s);
  }
}

cudaError_t launch_decode(const StateView &sv, int factor_dtype, const float *q, const float *k,
                          const float *v, const float *gate, const float *beta, const float *A,
                          float *o, int cols_max, cudaStream_t s) {
  DecodeArgs a{sv, q, k, v, gate, beta, A, o};
  if (factor_dtype == SEED_BF16) return launch_decode_v<__nv_bfloat16>(a, cols_max, s);
  return launch_decode_v<float>(a, cols_max, s);
}

}  // namespace seedk
