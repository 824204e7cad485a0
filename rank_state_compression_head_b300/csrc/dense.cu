// Dense-state kernels: the original model's decode step (in-run comparison)
// and the reconstruction S = a vbar^T + U_eff W^T.
//
// "Shallow Encoding Emits Deep Memories", thelatestinai.com list view,
// abstract: every decode step loads and stores whole recurrent states.  The
// dense step reads the d_k x d_v fp32 state of a head once, keeps it in
// registers, applies the recurrence, reads out the updated state and writes
// it back once.  picx.dev summary, SEED Architecture (decode paragraph): the
// factored state is S = a vbar^T + U V^T.
#include "common.cuh"

namespace seedk {

struct DenseArgs {
  int variant, n_heads;
  float *S;
  const float *q, *k, *v, *gate, *beta, *A;
  const int32_t *dir_index;
  float *o;
};

template <int VAR, int DV>
__global__ void __launch_bounds__(256) dense_decode_kernel(const DenseArgs p) {
  constexpr int DK = kDK;
  constexpr int NW = 8;
  constexpr int LPR = DV / 4;          // lanes per state row (float4 each)
  constexpr int RPW = 32 / LPR;        // rows per warp-wide load
  constexpr int NL = DK / (RPW * NW);  // row loads per thread
  constexpr int NG = NW * RPW;         // partial groups per column
  constexpr bool M2 = VAR == SEED_MAMBA2;
  __shared__ __align__(16) float red[2][NG][DV];

  const int h = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c4 = (lane % LPR) * 4;
  const int grp = warp * RPW + lane / LPR;
  float *Sh = p.S + (int64_t)h * DK * DV;
  const float *qh = p.q + (int64_t)h * DK, *kh = p.k + (int64_t)h * DK, *vh = p.v + (int64_t)h * DV;

  float4 st[NL];
#pragma unroll
  for (int L = 0; L < NL; ++L) {
    const int row = (L * NW + warp) * RPW + lane / LPR;
    st[L] = *reinterpret_cast<const float4 *>(Sh + row * DV + c4);
  }

  float g = 0.f, beta = 0.f, dt = 0.f;
  if (VAR == SEED_GDN) { g = p.gate[h]; beta = p.beta[h]; }
  if (VAR == SEED_KDA) { beta = p.beta[h]; }
  if (M2) {
    dt = p.gate[h];
    const int dir = p.dir_index ? p.dir_index[h] : h;
    g = expf(dt * p.A[dir]);
  }
  const float4 v4 = *reinterpret_cast<const float4 *>(vh + c4);

  if (!M2) {
    // u = k^T S over this thread's rows, then across groups
    float4 u = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int L = 0; L < NL; ++L) {
      const int row = (L * NW + warp) * RPW + lane / LPR;
      const float kr = kh[row];
      u.x = fmaf(kr, st[L].x, u.x); u.y = fmaf(kr, st[L].y, u.y);
      u.z = fmaf(kr, st[L].z, u.z); u.w = fmaf(kr, st[L].w, u.w);
    }
    *reinterpret_cast<float4 *>(&red[0][grp][c4]) = u;
    __syncthreads();
    u = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int gi = 0; gi < NG; ++gi) {
      const float4 t = *reinterpret_cast<const float4 *>(&red[0][gi][c4]);
      u.x += t.x; u.y += t.y; u.z += t.z; u.w += t.w;
    }
    // GDN: S' = alpha S + k (beta (v - alpha u))^T ;  KDA: S'_i = alpha_i (S_i - beta k_i u) + beta k_i v
#pragma unroll
    for (int L = 0; L < NL; ++L) {
      const int row = (L * NW + warp) * RPW + lane / LPR;
      const float kr = kh[row];
      if (VAR == SEED_GDN) {
        st[L].x = fmaf(g, st[L].x, kr * beta * fmaf(-g, u.x, v4.x));
        st[L].y = fmaf(g, st[L].y, kr * beta * fmaf(-g, u.y, v4.y));
        st[L].z = fmaf(g, st[L].z, kr * beta * fmaf(-g, u.z, v4.z));
        st[L].w = fmaf(g, st[L].w, kr * beta * fmaf(-g, u.w, v4.w));
      } else {
        const float ar = p.gate[(int64_t)h * DK + row];
        const float bk = beta * kr;
        st[L].x = fmaf(ar, fmaf(-bk, u.x, st[L].x), bk * v4.x);
        st[L].y = fmaf(ar, fmaf(-bk, u.y, st[L].y), bk * v4.y);
        st[L].z = fmaf(ar, fmaf(-bk, u.z, st[L].z), bk * v4.z);
        st[L].w = fmaf(ar, fmaf(-bk, u.w, st[L].w), bk * v4.w);
      }
    }
  } else {
    // S' = g S + dt B x^T
#pragma unroll
    for (int L = 0; L < NL; ++L) {
      const int row = (L * NW + warp) * RPW + lane / LPR;
      const float b = dt * kh[row];
      st[L].x = fmaf(g, st[L].x, b * v4.x); st[L].y = fmaf(g, st[L].y, b * v4.y);
      st[L].z = fmaf(g, st[L].z, b * v4.z); st[L].w = fmaf(g, st[L].w, b * v4.w);
    }
  }

  // read-out of the updated state, and write back
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int L = 0; L < NL; ++L) {
    const int row = (L * NW + warp) * RPW + lane / LPR;
    const float qr = qh[row];
    o.x = fmaf(qr, st[L].x, o.x); o.y = fmaf(qr, st[L].y, o.y);
    o.z = fmaf(qr, st[L].z, o.z); o.w = fmaf(qr, st[L].w, o.w);
    *reinterpret_cast<float4 *>(Sh + row * DV + c4) = st[L];
  }
  *reinterpret_cast<float4 *>(&red[1][grp][c4]) = o;
  __syncthreads();
  if (tid < DV) {
    float acc = 0.f;
#pragma unroll
    for (int gi = 0; gi < NG; ++gi) acc += red[1][gi][tid];
    p.o[(int64_t)h * DV + tid] = acc;
  }
}

template <int VAR>
static cudaError_t launch_dense_v(const DenseArgs &a, int d_v, cudaStream_t s) {
  if (d_v == 64) dense_decode_kernel<VAR, 64><<<a.n_heads, 256, 0, s>>>(a);
  else dense_decode_kernel<VAR, 128><<<a.n_heads, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_dense_decode(int variant, int n_heads, int d_v, float *S, const float *q,
                                const float *k, const float *v, const float *gate,
                                const float *beta, const float *A, const int32_t *dir_index,
                                float *o, cudaStream_t s) {
  DenseArgs a{variant, n_heads, S, q, k, v, gate, beta, A, dir_index, o};
  switch (variant) {
    case SEED_GDN: return launch_dense_v<SEED_GDN>(a, d_v, s);
    case SEED_KDA: return launch_dense_v<SEED_KDA>(a, d_v, s);
    default: return launch_dense_v<SEED_MAMBA2>(a, d_v, s);
  }
}

// ---------------------------------------------------------------------------
// S = a vbar^T + U_eff W^T
// ---------------------------------------------------------------------------

template <typename TF, int DV, bool KDA>
__global__ void __launch_bounds__(256) materialize_kernel(const StateView sv, float *S_out, int m_max) {
  constexpr int DK = kDK;
  extern __shared__ __align__(16) float sm[];
  const int h = blockIdx.x, tid = threadIdx.x;
  const int r_h = sv.rank_of(h);
  const int m = r_h + sv.growth * sv.steps;
  if (r_h < 0 || m > m_max) return;  // rank table disagrees with r_max
  const int64_t c0 = sv.col0(h);
  float *Ue = sm;               // [m][DK]
  float *Wl = sm + m * DK;      // [m][DV]
  const TF *Uh = reinterpret_cast<const TF *>(sv.U) + c0 * DK;
  const TF *Wh = reinterpret_cast<const TF *>(sv.W) + c0 * DV;
  for (int idx = tid; idx < m * DK; idx += 256) {
    const int j = idx / DK, i = idx % DK;
    const float f = KDA ? sv.scale[(int64_t)h * DK + i] : sv.scale[c0 + j];
    Ue[idx] = Elem<TF>::load(Uh + idx) * f;
  }
  for (int idx = tid; idx < m * DV; idx += 256) Wl[idx] = Elem<TF>::load(Wh + idx);
  __syncthreads();
  const float *ah = sv.a + (int64_t)h * DK;
  const float *vb = sv.vbar + (int64_t)sv.dir_of(h) * DV;
  float *Sh = S_out + (int64_t)h * DK * DV;
  for (int idx = tid; idx < DK * DV; idx += 256) {
    const int i = idx / DV, j = idx % DV;
    float acc = ah[i] * vb[j];
    for (int l = 0; l < m; ++l) acc = fmaf(Ue[l * DK + i], Wl[l * DV + j], acc);
    Sh[idx] = acc;
  }
}

template <typename TF, bool KDA>
static cudaError_t launch_mat_t(const StateView &sv, float *S_out, int m_max, cudaStream_t s) {
  const size_t bytes = (size_t)m_max * (kDK + sv.d_v) * sizeof(float);
  cudaError_t e;
  if (sv.d_v == 64) {
    auto kern = materialize_kernel<TF, 64, KDA>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    kern<<<sv.n_heads, 256, bytes, s>>>(sv, S_out, m_max);
  } else {
    auto kern = materialize_kernel<TF, 128, KDA>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    kern<<<sv.n_heads, 256, bytes, s>>>(sv, S_out, m_max);
  }
  return cudaGetLastError();
}

cudaError_t launch_materialize(const StateView &sv, int factor_dtype, float *S_out, int m_max,
                               cudaStream_t s) {
  const bool kda = sv.variant == SEED_KDA;
  if (factor_dtype == SEED_BF16)
    return kda ? launch_mat_t<__nv_bfloat16, true>(sv, S_out, m_max, s)
               : launch_mat_t<__nv_bfloat16, false>(sv, S_out, m_max, s);
  if (factor_dtype == SEED_F16)
    return kda ? launch_mat_t<__half, true>(sv, S_out, m_max, s) : launch_mat_t<__half, false>(sv, S_out, m_max, s);
  return kda ? launch_mat_t<float, true>(sv, S_out, m_max, s)
             : launch_mat_t<float, false>(sv, S_out, m_max, s);
}

}  // namespace seedk
