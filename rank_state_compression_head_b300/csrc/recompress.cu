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
//   core K = R_a R_b^T (m x m); Q_a, Q_b formed in place from the reflectors
//   K P = Q R (pivoted QR), one-sided Jacobi on R^T: R^T J = V Sigma
//   keep the rank(h) largest sigma; y_k = P v_k (right singular vectors of K)
//   U_new = Q_a K y_k (= sigma_k Q_a x_k),  W_new = Q_b y_k
//   (no rotation is kept: the kept directions are read off R^T J and applied
//   to the original core)
// compress_dense (one CTA of 256 threads per head): sink split, then the
// d_k x d_v matrix C itself takes the place of the core: C P = Q R (pivoted
// QR), one-sided Jacobi on R^T, y_k = P v_k, U_new = C y_k (= sigma_k x_k, C
// read again from S and a), W_new = y_k.
//
// The arithmetic is fp32 FMA: the QR and Jacobi steps are sequences of small
// dependent reductions that do not map onto tensor-core tiles.
#include "recompress_core.cuh"

namespace seedk {

struct CompressArgs {
  StateView sv;
  float *trunc_err;
  int32_t *sweeps;  // Jacobi sweeps per head (or -1: limit reached), optional
  const float *S;   // dense input (compress_dense) or nullptr (recompress)
  int m_max;        // smem sizing: largest column count of any head
  int cs_alloc;     // column stride of the core buffers in the allocation
};

// Dynamic shared-memory layout of compress_dense (offsets in floats, multiples
// of 4): two buffers that hold in turn C (column pitch d_k + 4), the seats of the
// Jacobi (pitch cs) and C again; then a, vbar and the vectors of the core stage.
struct DenseSmem {
  int pc, buf;
  int offB0, offB1, offA, offVb, offVn, offP, offS, offI, offO, offR;
  int total_floats;
  __host__ __device__ DenseSmem(int dk, int dv, int cs) {
    auto up4 = [](int x) { return (x + 3) & ~3; };
    pc = dk + 4;
    const int c_sz = dv * pc, seat_sz = (dv + 1) * cs;
    buf = up4(c_sz > seat_sz ? c_sz : seat_sz);
    offB0 = 0;
    offB1 = offB0 + buf;
    offA = offB1 + buf;
    offVb = offA + up4(dk);
    offVn = offVb + up4(dv);
    offP = offVn + up4(dv);
    offS = offP + up4(dv);
    offI = offS + up4(dv);
    offO = offI + up4(dv);
    offR = offO + up4(dv);
    total_floats = offR + 8;
  }
};

// compress_dense, one CTA of 256 threads per head:
//   a = S vbar / |vbar|^2, C = S - a vbar^T (C in shared memory as columns)
//   C P = Q R (pivoted Householder QR, qrcp_rect), R^T to the seats, scaled by a
//   power of two; one-sided Jacobi on R^T (jacobi_seats): R^T J = V Sigma
//   keep the rank(h) largest sigma: y_k = P v_k, U = C y_k (= sigma_k x_k), W = y_k
// the same numerics as the recompression's core stage, with the 128 x d_v state
// in place of the core.
template <int VAR, typename TF, int DV>
__global__ void __launch_bounds__(256) compress_dense_kernel(const CompressArgs p) {
  constexpr int DK = kDK;
  constexpr int NT = 256;
  constexpr int m = DV;
  extern __shared__ __align__(16) float smem[];
  const int h = blockIdx.x;
  const int tid = threadIdx.x;
  const StateView &sv = p.sv;
  const int r = sv.rank_of(h);
  if (r < 0) {  // rank table disagrees with r_max: touch nothing
    if (tid == 0 && sv.status) sv.status[h] = SEED_ERR_INVALID_ARG;
    return;
  }
  const int64_t c0 = sv.col0(h);
  const JacobiGeom g = seat_geom(m, NT);
  const DenseSmem L(DK, DV, p.cs_alloc);
  const int pc = L.pc, cs = g.cs;
  float *B0 = smem + L.offB0, *B1 = smem + L.offB1, *as = smem + L.offA, *vb = smem + L.offVb;
  float *vn = smem + L.offVn, *sig2 = smem + L.offS, *inv = smem + L.offI, *red = smem + L.offR;
  int *piv = reinterpret_cast<int *>(smem + L.offP);
  int *order = reinterpret_cast<int *>(smem + L.offO);
  TF *Uh = reinterpret_cast<TF *>(sv.U) + c0 * DK;
  TF *Wh = reinterpret_cast<TF *>(sv.W) + c0 * DV;
  const float *Sh = p.S + (int64_t)h * DK * DV;

  // ---- C = S - a vbar^T as columns of B0 --------------------------------------------------
  for (int idx = tid; idx < DK * DV; idx += NT) {
    const int i = idx / DV, j = idx % DV;
    B0[j * pc + i] = Sh[idx];
  }
  for (int j = tid; j < DV; j += NT) vb[j] = sv.vbar[(int64_t)sv.dir_of(h) * DV + j];
  __syncthreads();
  float vv = 0.f;
  for (int j = 0; j < DV; ++j) vv = fmaf(vb[j], vb[j], vv);
  if (tid < DK) {
    float acc = 0.f;
    for (int j = 0; j < DV; ++j) acc = fmaf(B0[j * pc + tid], vb[j], acc);
    const float ai = acc / vv;
    sv.a[(int64_t)h * DK + tid] = ai;
    as[tid] = ai;
    for (int j = 0; j < DV; ++j) B0[j * pc + tid] = fmaf(-ai, vb[j], B0[j * pc + tid]);
  }
  __syncthreads();

  // ---- pivoted QR of C; R^T to the seats of B1, scaled to a largest entry in [1/2, 1) ------
  qrcp_rect<NT>(B0, DK, DV, pc, piv, vn, red);
  float kmax = 0.f;
  for (int idx = tid; idx < m * m; idx += NT) {
    const int i = idx / m, s = idx % m;  // seat i = row i of R, entry s
    const float x = s >= i ? B0[s * pc + i] : 0.f;
    B1[i * cs + s] = x;
    kmax = fmaxf(kmax, fabsf(x));
  }
  kmax = warp_max(kmax);
  static_assert(NT / 32 <= 8, "one reduction slot per warp");
  if ((tid & 31) == 0) red[tid >> 5] = kmax;  // qrcp_rect is done with red (it ends with a barrier)
  __syncthreads();
  kmax = 0.f;
  for (int w = 0; w < NT / 32; ++w) kmax = fmaxf(kmax, red[w]);
  int kexp = 0;
  if (kmax > 0.f) frexpf(kmax, &kexp);
  const float kscale = ldexpf(1.f, -kexp), kunscale = ldexpf(1.f, kexp);
  for (int idx = tid; idx < m * m; idx += NT) B1[(idx / m) * cs + idx % m] *= kscale;
  __syncthreads();
  // bf16 factors: 1e-4 (their own rounding is 2^-9), stop once no pair is beyond
  // sqrt(tol); fp32: four times the rounding noise of a length-m dot product
  // (sqrt(m) eps), run until no pair is beyond tol
  const float tol = sizeof(TF) == 2 ? 1e-4f : 4.f * sqrtf((float)m) * FLT_EPSILON;
  float *F;
  const int sweeps = jacobi_seats<NT, 32>(B1, B0, m, g, tol, sizeof(TF) == 2 ? sqrtf(tol) : tol, &F);

  // ---- sigma^2, order, truncation error ---------------------------------------------------
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
  if (tid == 0) {
    float e = 0.f;
    for (int k = r; k < m; ++k) e += sig2[order[k]];
    if (p.trunc_err) p.trunc_err[h] = sqrtf(e) * kunscale;
    if (sv.status) sv.status[h] = sweeps < 0 ? SEED_ERR_NOT_CONVERGED : SEED_OK;
  }

  // ---- C again into the free buffer; U = C y_k, W = y_k, y_k[piv[s]] = (R^T J)_{s,k} / sigma --
  float *Cs = F == B0 ? B1 : B0;
  for (int idx = tid; idx < DK * DV; idx += NT) {
    const int i = idx / DV, j = idx % DV;
    Cs[j * pc + i] = fmaf(-as[i], vb[j], Sh[idx]);
  }
  __syncthreads();
  const int rk = r < m ? r : m;
  for (int idx = tid; idx < rk * DK; idx += NT) {
    const int k = idx / DK, i = idx % DK;
    const int col = order[k];
    const float *f = F + col * cs;
    float acc = 0.f;
    for (int s2 = 0; s2 < m; ++s2) acc = fmaf(Cs[piv[s2] * pc + i], f[s2], acc);
    Elem<TF>::store(Uh + (int64_t)k * DK + i, stored_elem<TF>(sv, acc * inv[col], c0 + k, i, kSrRebuildU));
  }
  for (int idx = tid; idx < rk * DV; idx += NT) {
    const int k = idx / DV, s2 = idx % DV;
    const int col = order[k];
    Elem<TF>::store(Wh + (int64_t)k * DV + piv[s2],
                    stored_elem<TF>(sv, F[col * cs + s2] * inv[col], c0 + k, piv[s2], kSrRebuildW));
  }
  if (VAR == SEED_KDA) {
    for (int i = tid; i < DK; i += NT) sv.scale[(int64_t)h * DK + i] = 1.f;
  } else {
    for (int k = tid; k < rk; k += NT) sv.scale[c0 + k] = 1.f;
  }
}

// Dynamic shared-memory layout of the single-kernel recompression (offsets in
// floats, multiples of 4): the two factor panels, the two core buffers of the
// pivoted QR and Jacobi (m + 1 seats for an odd m), the unscaled core, vectors.
struct RecSmem {
  int lda, ldb;
  int offA, offB, offK, offT, offK0, offTa, offTb, offS, offI, offV, offO, offP, offQ, offR;
  int total_floats;
  __host__ __device__ RecSmem(int m, int dk, int dv, int cs) {
    lda = dk + 4;
    ldb = dv + 4;
    auto up4 = [](int x) { return (x + 3) & ~3; };
    const int seats = m + 1;
    offA = 0;
    offB = up4(offA + m * lda);
    offK = up4(offB + m * ldb);
    offT = offK + seats * cs;
    offK0 = offT + seats * cs;
    offTa = offK0 + m * cs;
    offTb = offTa + up4(m);
    offS = offTb + up4(m);
    offI = offS + up4(m);
    offV = offI + up4(m);
    offO = offV + up4(m);
    offP = offO + up4(m);
    offQ = offP + up4(m);
    offR = offQ + up4(m);
    total_floats = offR + 8;
  }
};

template <int VAR, typename TF, int DV>
__global__ void __launch_bounds__(128) recompress_kernel(const CompressArgs p) {
  constexpr int DK = kDK;
  constexpr int NT = 128;
  extern __shared__ __align__(16) float smem[];
  const int h = blockIdx.x;
  const int tid = threadIdx.x;
  const StateView &sv = p.sv;
  const int r = sv.rank_of(h);
  const int m = r + sv.growth * sv.steps;
  if (r < 0 || m > p.m_max) {  // rank table disagrees with r_max: touch nothing
    if (tid == 0 && sv.status) sv.status[h] = SEED_ERR_INVALID_ARG;
    return;
  }
  const int64_t c0 = sv.col0(h);
  const RecSmem L(p.m_max, DK, DV, p.cs_alloc);
  const JacobiGeom g = seat_geom(m, NT);
  const int cs = g.cs;
  const int m4 = (m + 3) & ~3;
  float *A = smem + L.offA, *B = smem + L.offB, *Kb = smem + L.offK, *Tb = smem + L.offT;
  float *K0 = smem + L.offK0, *tauA = smem + L.offTa, *tauB = smem + L.offTb;
  float *sig2 = smem + L.offS, *inv = smem + L.offI, *vn = smem + L.offV, *red = smem + L.offR;
  int *order = reinterpret_cast<int *>(smem + L.offO);
  int *piv = reinterpret_cast<int *>(smem + L.offP);
  int *pinv = reinterpret_cast<int *>(smem + L.offQ);
  const int lda = L.lda, ldb = L.ldb;
  TF *Uh = reinterpret_cast<TF *>(sv.U) + c0 * DK;
  TF *Wh = reinterpret_cast<TF *>(sv.W) + c0 * DV;

  // ---- load -------------------------------------------------------------------
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
  __syncthreads();

  // ---- QR of both factors, core K = R_a R_b^T, Q factors in place ----------------------
  const int team = tid / 64, ttid = tid % 64;
  if (team == 0) householder_qr(A, lda, DK, m, tauA, ttid, 64, 1);
  else householder_qr(B, ldb, DV, m, tauB, ttid, 64, 2);
  __syncthreads();
  for (int idx = tid; idx < m * m4; idx += NT) {
    const int j = idx / m4, i = idx % m4;  // K[j][i]: column j, row i
    float acc = 0.f;
    // l from j for every lane of column j (B element a broadcast), l < i skipped
    if (i < m)
      for (int l = j; l < m; ++l)
        if (l >= i) acc = fmaf(A[l * lda + i], B[l * ldb + j], acc);
    Kb[j * cs + i] = acc;
    K0[j * cs + i] = acc;
  }
  __syncthreads();
  if (team == 0) form_q(A, lda, DK, m, tauA, ttid, 64, 1);
  else form_q(B, ldb, DV, m, tauB, ttid, 64, 2);

  // ---- core scaled by a power of two to a largest entry in [1/2, 1), then factored ---------
  float kmax = 0.f;
  for (int idx = tid; idx < m * m4; idx += NT) kmax = fmaxf(kmax, fabsf(Kb[(idx / m4) * cs + idx % m4]));
  kmax = warp_max(kmax);
  if ((tid & 31) == 0) red[tid >> 5] = kmax;
  __syncthreads();
  kmax = 0.f;
  for (int w = 0; w < NT / 32; ++w) kmax = fmaxf(kmax, red[w]);
  int kexp = 0;
  if (kmax > 0.f) frexpf(kmax, &kexp);
  const float kscale = ldexpf(1.f, -kexp), kunscale = ldexpf(1.f, kexp);
  for (int idx = tid; idx < m * m4; idx += NT) Kb[(idx / m4) * cs + idx % m4] *= kscale;
  __syncthreads();
  // bf16 factors: 1e-4 (their own rounding is 2^-9), stop once no pair is beyond
  // sqrt(tol); fp32: four times the rounding noise of a length-m dot product
  // (sqrt(m) eps), run until no pair is beyond tol
  const float tol = sizeof(TF) == 2 ? 1e-4f : 4.f * sqrtf((float)(m > 16 ? m : 16)) * FLT_EPSILON;
  float *F;
  const int sweeps = core_factor<NT>(Kb, Tb, m, g, tol, sizeof(TF) == 2 ? sqrtf(tol) : tol, piv, vn, sig2, inv,
                                     order, red, &F);
  if (tid == 0) {
    float e = 0.f;
    for (int k = r; k < m; ++k) e += sig2[order[k]];
    if (p.trunc_err) p.trunc_err[h] = sqrtf(e) * kunscale;
    if (p.sweeps) p.sweeps[h] = sweeps;
    if (sv.status) sv.status[h] = sweeps < 0 ? SEED_ERR_NOT_CONVERGED : SEED_OK;
  }

  // ---- z_k = K y_k into the free core buffer; y_k[piv[i]] = (R^T J)_{i,order[k]} / sigma_k ----
  const int rk = r < m ? r : m;
  float *Z = F == Kb ? Tb : Kb;  // [rk][m]
  for (int i = tid; i < m; i += NT) pinv[piv[i]] = i;
  for (int idx = tid; idx < rk * m; idx += NT) {
    const int k = idx / m, l = idx % m;
    const int col = order[k];
    const float *f = F + col * cs;
    float acc = 0.f;
    for (int i = 0; i < m; ++i) acc = fmaf(K0[piv[i] * cs + l], f[i], acc);
    Z[idx] = acc * inv[col];
  }
  __syncthreads();

  // ---- U = Q_a Z,  W = Q_b Y -------------------------------------------------------------------
  if (tid < DK) {
    for (int k = 0; k < rk; ++k) {
      float acc = 0.f;
      for (int l = 0; l < m; ++l) acc = fmaf(A[l * lda + tid], Z[k * m + l], acc);
      Elem<TF>::store(Uh + (int64_t)k * DK + tid, stored_elem<TF>(sv, acc, c0 + k, tid, kSrRebuildU));
    }
  }
  if (tid < DV) {
    for (int k = 0; k < rk; ++k) {
      const int col = order[k];
      const float *f = F + col * cs;
      const float ik = inv[col];
      float acc = 0.f;
      for (int l = 0; l < m; ++l) acc = fmaf(B[l * ldb + tid], f[pinv[l]] * ik, acc);
      Elem<TF>::store(Wh + (int64_t)k * DV + tid, stored_elem<TF>(sv, acc, c0 + k, tid, kSrRebuildW));
    }
  }
  if (VAR == SEED_KDA) {
    for (int i = tid; i < DK; i += NT) sv.scale[(int64_t)h * DK + i] = 1.f;
  } else {
    for (int k = tid; k < rk; k += NT) sv.scale[c0 + k] = 1.f;
  }
}

template <int VAR, typename TF, int DV>
static cudaError_t launch_recompress_t(const CompressArgs &a, cudaStream_t s) {
  CompressArgs args = a;
  args.cs_alloc = seat_cs_alloc(a.m_max, 128);
  const RecSmem L(a.m_max, kDK, DV, args.cs_alloc);
  const size_t bytes = (size_t)L.total_floats * sizeof(float);
  auto kern = recompress_kernel<VAR, TF, DV>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  kern<<<a.sv.n_heads, 128, bytes, s>>>(args);
  return cudaGetLastError();
}

template <int VAR, typename TF, int DV>
static cudaError_t launch_dense_t(const CompressArgs &a, cudaStream_t s) {
  CompressArgs args = a;
  args.cs_alloc = seat_geom(DV, 256).cs;
  const DenseSmem L(kDK, DV, args.cs_alloc);
  const size_t bytes = (size_t)L.total_floats * sizeof(float);
  auto kern = compress_dense_kernel<VAR, TF, DV>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  kern<<<a.sv.n_heads, 256, bytes, s>>>(args);
  return cudaGetLastError();
}

template <typename TF, bool DENSE>
static cudaError_t launch_compress_v(const CompressArgs &a, cudaStream_t s) {
  // Only the scale layout differs between variants here.
  const bool kda = a.sv.variant == SEED_KDA, dv64 = a.sv.d_v == 64;
  if (DENSE) {
    if (kda) return dv64 ? launch_dense_t<SEED_KDA, TF, 64>(a, s) : launch_dense_t<SEED_KDA, TF, 128>(a, s);
    return dv64 ? launch_dense_t<SEED_GDN, TF, 64>(a, s) : launch_dense_t<SEED_GDN, TF, 128>(a, s);
  }
  if (kda) return dv64 ? launch_recompress_t<SEED_KDA, TF, 64>(a, s) : launch_recompress_t<SEED_KDA, TF, 128>(a, s);
  return dv64 ? launch_recompress_t<SEED_GDN, TF, 64>(a, s) : launch_recompress_t<SEED_GDN, TF, 128>(a, s);
}

cudaError_t launch_recompress(const StateView &sv, int factor_dtype, float *trunc_err,
                              int32_t *sweeps, int m_max, cudaStream_t s) {
  CompressArgs a{sv, trunc_err, sweeps, nullptr, m_max, 0};
  if (factor_dtype == SEED_BF16) return launch_compress_v<__nv_bfloat16, false>(a, s);
  if (factor_dtype == SEED_F16) return launch_compress_v<__half, false>(a, s);
  return launch_compress_v<float, false>(a, s);
}

cudaError_t launch_compress_dense(const StateView &sv, int factor_dtype, const float *S,
                                  float *trunc_err, cudaStream_t s) {
  CompressArgs a{sv, trunc_err, nullptr, S, sv.d_v, 0};
  if (factor_dtype == SEED_BF16) return launch_compress_v<__nv_bfloat16, true>(a, s);
  if (factor_dtype == SEED_F16) return launch_compress_v<__half, true>(a, s);
  return launch_compress_v<float, true>(a, s);
}

}  // namespace seedk
