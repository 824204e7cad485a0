// Recompression in three phases over a caller-provided device workspace.
//
// The algorithm of the single-kernel recompression in recompress.cu ("Shallow
// Encoding Emits Deep Memories", thelatestinai.com list view, Table 1: the
// decode compresses back to rank R every W steps), laid out so that each phase
// holds only what it needs: the factor panels in registers for the QR, one warp
// per head for the core SVD, a GEMM-like rebuild.  The two paths agree to
// rounding (the summation orders differ), not bit for bit.
//
//   qr_phase      one CTA per head, two teams (U_eff, W) of four threads per
//                 column (qr_registers.cuh): Householder QR of both panels; the
//                 U_eff team forms the core K = R_a R_b^T while the W team
//                 writes out W's reflectors (V_b, tau_b) and R_b; no Q is formed
//   svd_phase     one warp per head (svd_warp.cuh): pivoted QR of the core and
//                 one-sided Jacobi on R^T, ordering, truncation error; writes
//                 the kept right singular vectors Y (y_k)
//   rebuild_phase one CTA per (head, factor): U = U_eff (R_b^T Y), which is
//                 Q_a K Y because U_eff = Q_a R_a; W = Q_b Y by W's reflectors
//                 applied to [Y; 0]; resets the lazy scales
//
// Workspace per head (fp32): V_b [m][d_v] (reflector j in row j), tau_b [m4],
// R_b^T [m][m] (row i = row i of R_b), K [m][m] (column-major), Y [r][m4]
// (m4 = m rounded up to 4, zero padded), each region starting on 16 bytes, the
// whole rounded up to 256 bytes, with m the largest column count of any head at
// this call and r the largest rank.
#include "recompress_core.cuh"
#include "qr_registers.cuh"
#include "svd_warp.cuh"

namespace seedk {

struct SplitLayout {
  int64_t vb, tau, rb, k, y, per_head;  // offsets and stride in floats
  int m4;                               // row stride of Y
  __host__ __device__ SplitLayout(int m, int r, int dk, int dv) {
    (void)dk;
    m4 = (m + 3) & ~3;
    const int64_t mm4 = ((int64_t)m * m + 3) & ~(int64_t)3;
    vb = 0;
    tau = vb + (int64_t)m * dv;
    rb = tau + m4;
    k = rb + mm4;
    y = k + mm4;
    per_head = (y + (int64_t)r * m4 + 63) & ~(int64_t)63;
    if (per_head == 0) per_head = 64;  // no columns: keep a nonzero stride
  }
};

struct SplitArgs {
  StateView sv;
  float *ws;
  int head0;     // first head of this chunk; workspace slot b serves head head0 + b
  int n_group;   // heads in this chunk
  int m_max;     // this launch serves heads with m_lo < m <= m_max (its thread and
  int m_lo;      //   shared-memory sizes follow m_max); m_lo = -1: every head
  int layout_m;  // column count the workspace layout is sized for (the call's m_max)
  int r_max;
  float *trunc_err;
  int32_t *sweeps;
  int cs_alloc;
};

constexpr int kSplitThreads = 128;

__device__ inline bool split_head_ok(const StateView &sv, int h, int m_max, int &r, int &m) {
  r = sv.rank_of(h);
  m = r + sv.growth * sv.steps;
  return r >= 0 && m <= m_max;
}
__device__ inline bool in_class(const SplitArgs &p, int m) { return m > p.m_lo && m <= p.m_max; }

// ---- phase 1: QR of both factors, core, W's reflectors -------------------------------
// Two teams of kTPC x m_max threads (the second starts on a warp boundary),
// kTPC threads per column, the panels in registers (qr_registers.cuh).
__host__ __device__ inline int qr_team_stride(int m_max) { return (kTPC * m_max + 31) / 32 * 32; }

// 80 registers: two CTAs of 384 threads (m_max = 48) per SM, a few bytes of spill
template <int VAR, typename TF, int DV>
__global__ void __maxnreg__(80) qr_phase(const SplitArgs p) {
  constexpr int DK = kDK;
  extern __shared__ __align__(16) float smem[];
  const int h = p.head0 + blockIdx.x;
  const int tid = threadIdx.x;
  const StateView &sv = p.sv;
  int r, m;
  if (!split_head_ok(sv, h, p.layout_m, r, m) || !in_class(p, m)) return;  // bad ranks: reported by the SVD phase
  const int mm = p.m_max;
  const int up = (mm + 3) & ~3;
  const int wbase = qr_team_stride(mm);
  const bool teamU = tid < wbase;   // warps of the U_eff panel, then those of W
  const int t = teamU ? tid : tid - wbase;
  const int l = t / kTPC, part = t % kTPC;
  const int rows = teamU ? DK : DV;
  const bool mine = l < m;
  const unsigned pmask = ((1u << kTPC) - 1) << ((tid & 31) & ~(kTPC - 1));
  // shared: V of each panel [m_max][rows], tau and beta of each panel, R of each panel
  float *V = smem + (teamU ? 0 : mm * DK);
  float *tau = smem + mm * (DK + DV) + (teamU ? 0 : up);
  float *betas = smem + mm * (DK + DV) + 2 * up + (teamU ? 0 : up);
  float *RsU = smem + mm * (DK + DV) + 4 * up;  // [m_max][m_max]: column l, row i
  float *RsW = RsU + mm * mm;
  const int64_t c0 = sv.col0(h);

  // ---- my half of column l: U_eff (scaled) or W -----------------------------------------
  RRCol c;
  c.nch = rows / (4 * kTPC);
#pragma unroll
  for (int i = 0; i < kRRChunks; ++i) c.x[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (mine) {
    const TF *col = reinterpret_cast<const TF *>(teamU ? sv.U : sv.W) + (c0 + l) * rows;
    const float cscale = (teamU && VAR != SEED_KDA) ? sv.scale[c0 + l] : 1.f;
#pragma unroll
    for (int i = 0; i < kRRChunks; ++i) {
      if (i >= c.nch) break;
      const int row = rr_row(part, i, 0);
      float4 a;
      if (sizeof(TF) == 2) {
        const uint2 u = *reinterpret_cast<const uint2 *>(col + row);
        a = make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                        __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
      } else {
        a = *reinterpret_cast<const float4 *>(col + row);
      }
      if (teamU && VAR == SEED_KDA) {
        const float4 d = *reinterpret_cast<const float4 *>(sv.scale + (int64_t)h * DK + row);
        a = make_float4(a.x * d.x, a.y * d.y, a.z * d.z, a.w * d.w);
      } else if (teamU) {
        a = make_float4(a.x * cscale, a.y * cscale, a.z * cscale, a.w * cscale);
      }
      c.x[i] = a;
    }
  }

  // ---- Householder QR of both panels ------------------------------------------------------
  // The teams share nothing until R is in shared memory: each waits only for its
  // own reflector (named barrier 1 or 2 over its wbase threads)
  for (int j = 0; j < m; ++j) {
    if ((t >> 5) == ((kTPC * j) >> 5))  // the warp that holds column j of my panel
      rr_reflector_warp(c, l == j, part, j, rows, V + j * rows, tau + j, betas + j);
    if (teamU) asm volatile("bar.sync 1, %0;" ::"r"(wbase) : "memory");
    else asm volatile("bar.sync 2, %0;" ::"r"(wbase) : "memory");
    if (mine && l > j) rr_apply(c, part, V + j * rows, tau[j], pmask);
  }
  // ---- R factors to shared memory ------------------------------------------------------------
  if (mine) {
    float *Rs = teamU ? RsU : RsW;
#pragma unroll
    for (int i = 0; i < kRRChunks; ++i) {
      if (i >= c.nch) break;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int row = rr_row(part, i, e);
        if (row < m) Rs[l * mm + row] = row < l ? f4get(c.x[i], e) : row == l ? betas[l] : 0.f;
      }
    }
  }
  __syncthreads();
  const SplitLayout L(p.layout_m, p.r_max, DK, DV);
  float *ws = p.ws + (int64_t)blockIdx.x * L.per_head;
  const int team = wbase;  // threads per team
  if (teamU) {
    // ---- core K = R_a R_b^T to the workspace ----------------------------------------------
    // R is zero below the diagonal, so every lane of a column j of K runs k = j..m-1:
    // the R_b element is a broadcast, the R_a elements are consecutive
    float *Kw = ws + L.k;
    for (int idx = t; idx < m * m; idx += team) {
      const int j = idx / m, i = idx % m;  // K[j][i]: column j, row i
      float acc = 0.f;
      for (int k = j; k < m; ++k) acc = fmaf(RsU[k * mm + i], RsW[k * mm + j], acc);
      Kw[idx] = acc;
    }
  } else {
    // ---- W's reflectors and R_b to the workspace ------------------------------------------------
    const float4 *v4 = reinterpret_cast<const float4 *>(V);
    float4 *vb4 = reinterpret_cast<float4 *>(ws + L.vb);
    for (int idx = t; idx < m * (DV / 4); idx += team) vb4[idx] = v4[idx];
    for (int j = t; j < m; j += team) ws[L.tau + j] = tau[j];
    float *rbt = ws + L.rb;
    for (int idx = t; idx < m * m; idx += team) {
      const int i = idx / m, l = idx % m;  // R_b^T row i = row i of R_b
      rbt[idx] = RsW[l * mm + i];
    }
  }
}

// ---- phase 2: SVD of the core, one lane group per head (svd_warp.cuh) ---------------------
// MR: rows and columns of the core held per lane (m_max rounded up to 16); a
// group is a warp, or a half warp when MR <= 32 (two heads per warp).
template <int MR>
constexpr int svd_group() { return MR <= 32 ? 16 : 32; }
template <int MR>
constexpr int svd_heads_per_cta() { return kSvdWarps * (32 / svd_group<MR>()); }

template <typename TF, int DV, int MR>
__global__ void __launch_bounds__(32 * kSvdWarps, MR <= 48 ? 8 : 6) svd_phase(const SplitArgs p) {
  constexpr int DK = kDK;
  constexpr int HW = svd_group<MR>();
  using SW = SvdWarpSmem<MR>;
  extern __shared__ __align__(16) float smem[];
  const int grp = threadIdx.x / HW, lane = threadIdx.x & (HW - 1);
  const unsigned gmask = HW == 32 ? 0xffffffffu : 0xffffu << (threadIdx.x & 16);
  const int b = blockIdx.x * svd_heads_per_cta<MR>() + grp;
  if (b >= p.n_group) return;
  const int h = p.head0 + b;
  const StateView &sv = p.sv;
  int r, m;
  if (!split_head_ok(sv, h, p.layout_m, r, m)) {  // rank table disagrees with r_max: touch nothing
    if (lane == 0 && sv.status) sv.status[h] = SEED_ERR_INVALID_ARG;
    return;
  }
  if (!in_class(p, m)) return;  // served by the launch of its column class
  float *sw = smem + grp * SW::FLOATS;
  float *T = sw + SW::T_OFF;
  const SplitLayout L(p.layout_m, p.r_max, DK, DV);
  float *ws = p.ws + (int64_t)b * L.per_head;
  const float *Kw = ws + L.k;

  // core into the square (coalesced reads; rows m..MR-1 zero), scaled by a power
  // of two to a largest entry in [1/2, 1)
  float kmax = 0.f;
  for (int idx = lane; idx < m * MR; idx += HW) {
    const int c = idx / MR, rr = idx % MR;
    const float x = rr < m ? Kw[c * m + rr] : 0.f;  // column c, row rr
    T[c * SW::TP + rr] = x;
    kmax = fmaxf(kmax, fabsf(x));
  }
#pragma unroll
  for (int o = HW / 2; o > 0; o >>= 1) kmax = fmaxf(kmax, __shfl_xor_sync(gmask, kmax, o));
  int kexp = 0;
  if (kmax > 0.f) frexpf(kmax, &kexp);
  const float kscale = ldexpf(1.f, -kexp), kunscale = ldexpf(1.f, kexp);
  __syncwarp(gmask);
  for (int idx = lane; idx < m * MR; idx += HW) T[(idx / MR) * SW::TP + idx % MR] *= kscale;
  __syncwarp(gmask);
  // bf16 factors: 1e-4 (their own rounding is 2^-9), stop once no pair is beyond
  // sqrt(tol); fp32: four times the rounding noise of a length-m dot product
  // (sqrt(m) eps), run until no pair is beyond tol
  const float tol = sizeof(TF) == 2 ? 1e-4f : 4.f * sqrtf((float)(m > 16 ? m : 16)) * FLT_EPSILON;
  const int sweeps = svd_warp_core<MR, HW>(m, tol, sizeof(TF) == 2 ? sqrtf(tol) : tol, sw);
  const float *sig2 = sw + SW::S_OFF, *inv = sw + SW::I_OFF;
  const int *order = reinterpret_cast<const int *>(sw + SW::O_OFF);
  const int *piv = reinterpret_cast<const int *>(sw + SW::P_OFF);
  if (lane == 0) {
    float e = 0.f;
    for (int k = r; k < m; ++k) e += sig2[order[k]];
    if (p.trunc_err) p.trunc_err[h] = sqrtf(e) * kunscale;
    if (p.sweeps) p.sweeps[h] = sweeps;
    if (sv.status) sv.status[h] = sweeps < 0 ? SEED_ERR_NOT_CONVERGED : SEED_OK;
  }
  // kept right singular vectors y_k[piv[s]] = (R^T J)_{s, order[k]} / sigma_k; rows
  // m..m4-1 zero
  const int rk = r < m ? r : m;
  const int m4 = (m + 3) & ~3;
  float *Y = ws + L.y;
  for (int k = 0; k < rk; ++k) {
    const int col = order[k];
    const float ik = inv[col];
    const float *f = T + col * SW::TP;
    for (int s = lane; s < m4; s += HW) Y[k * L.m4 + (s < m ? piv[s] : s)] = s < m ? f[s] * ik : 0.f;
  }
}

// ---- phase 3: rebuild the factors ---------------------------------------------------------
// U (blockIdx.y = 0): one row of U_eff per thread in registers (MR = m_max
// rounded up to 16 entries), M = R_b^T Y formed in shared memory first and read
// as broadcast 16-byte loads, four outputs at a time; the row is read in full
// before it is overwritten, and every thread has read the scales before they
// are reset.  W (blockIdx.y = 1): kTPC threads per kept column k hold
// [y_k; 0] in registers (qr_registers.cuh) and apply H_{m-1}, ..., H_0, two
// reflectors a pass.
template <int VAR, typename TF, int DV, int MR>
__global__ void __launch_bounds__(kSplitThreads) rebuild_phase(const SplitArgs p) {
  constexpr int DK = kDK;
  constexpr int NO = 4;  // outputs per pass
  extern __shared__ __align__(16) float smem[];
  const int h = p.head0 + blockIdx.x;
  const int tid = threadIdx.x;
  const StateView &sv = p.sv;
  int r, m;
  if (!split_head_ok(sv, h, p.layout_m, r, m) || !in_class(p, m)) return;
  const SplitLayout L(p.layout_m, p.r_max, DK, DV);
  const float *ws = p.ws + (int64_t)blockIdx.x * L.per_head;
  const int rk = r < m ? r : m;
  const int rk4 = (rk + NO - 1) / NO * NO;
  const int64_t c0 = sv.col0(h);
  if (blockIdx.y == 0) {
    // ---- U = U_eff M, M = R_b^T Y ---------------------------------------------------------
    float *rbt = smem;            // [MR][MR]: row i of R_b
    float *yt = rbt + MR * MR;    // [MR][rk4]: y_k[i] at i * rk4 + k
    float *zs = yt + rk4 * MR;    // [rk4][MR]: column k of M, zero beyond m and rk
    for (int idx = tid; idx < m * m; idx += kSplitThreads) rbt[(idx / m) * MR + idx % m] = ws[L.rb + idx];
    for (int idx = tid; idx < MR * rk4; idx += kSplitThreads) {
      const int i = idx / rk4, k = idx % rk4;
      yt[idx] = (k < rk && i < m) ? ws[L.y + k * L.m4 + i] : 0.f;
    }
    __syncthreads();
    // M[l][k] = sum_{i <= l} R_b[i][l] y_k[i], four k a task: one R_b element and
    // one 16-byte broadcast of y an i
    for (int task = tid; task < (rk4 / 4) * MR; task += kSplitThreads) {
      const int l = task % MR, k = 4 * (task / MR);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      if (l < m)
        for (int i = 0; i <= l; ++i) {
          const float rv = rbt[i * MR + l];
          const float4 y = *reinterpret_cast<const float4 *>(yt + i * rk4 + k);
          acc.x = fmaf(rv, y.x, acc.x); acc.y = fmaf(rv, y.y, acc.y);
          acc.z = fmaf(rv, y.z, acc.z); acc.w = fmaf(rv, y.w, acc.w);
        }
      zs[k * MR + l] = acc.x;
      zs[(k + 1) * MR + l] = acc.y;
      zs[(k + 2) * MR + l] = acc.z;
      zs[(k + 3) * MR + l] = acc.w;
    }
    __syncthreads();
    if (tid < DK) {
      TF *pool = reinterpret_cast<TF *>(sv.U) + c0 * DK;
      const float rs = VAR == SEED_KDA ? sv.scale[(int64_t)h * DK + tid] : 1.f;
      float q[MR];
#pragma unroll
      for (int l = 0; l < MR; ++l) {
        q[l] = 0.f;
        if (l < m) q[l] = Elem<TF>::load(pool + (int64_t)l * DK + tid) * (VAR == SEED_KDA ? rs : sv.scale[c0 + l]);
      }
      for (int k = 0; k < rk; k += NO) {
        float acc[NO];
#pragma unroll
        for (int o = 0; o < NO; ++o) acc[o] = 0.f;
#pragma unroll
        for (int l4 = 0; l4 < MR / 4; ++l4) {
#pragma unroll
          for (int o = 0; o < NO; ++o) {
            const float4 z = reinterpret_cast<const float4 *>(zs + (k + o) * MR)[l4];
            acc[o] = fmaf(q[4 * l4], z.x, fmaf(q[4 * l4 + 1], z.y, fmaf(q[4 * l4 + 2], z.z, fmaf(q[4 * l4 + 3], z.w, acc[o]))));
          }
        }
#pragma unroll
        for (int o = 0; o < NO; ++o)
          if (k + o < rk) Elem<TF>::store(pool + (int64_t)(k + o) * DK + tid, acc[o]);
      }
    }
    __syncthreads();  // every thread has read the scales
    if (VAR == SEED_KDA) {
      for (int i = tid; i < DK; i += kSplitThreads) sv.scale[(int64_t)h * DK + i] = 1.f;
    } else {
      for (int k = tid; k < rk; k += kSplitThreads) sv.scale[c0 + k] = 1.f;
    }
  } else {
    // ---- W = Q_b [Y; 0] = H_0 ... H_{m-1} [Y; 0] --------------------------------------------
    float *vs = smem;                    // [m][DV]: v_j, zero above row j
    float *ts = vs + m * DV;             // [m]: tau_j
    float *gs = ts + ((m + 3) & ~3);     // [m]: g_j = v_j . v_{j+1} for j = m-2, m-4, ...
    const float4 *src = reinterpret_cast<const float4 *>(ws + L.vb);
    for (int idx = tid; idx < m * (DV / 4); idx += kSplitThreads) reinterpret_cast<float4 *>(vs)[idx] = src[idx];
    for (int j = tid; j < m; j += kSplitThreads) ts[j] = ws[L.tau + j];
    __syncthreads();
    {
      constexpr int kWarps = kSplitThreads / 32;
      const int warp = tid >> 5, ln = tid & 31;
      for (int j = m - 2 - 2 * warp; j >= 0; j -= 2 * kWarps) {
        float acc = 0.f;
        for (int i = ln; i < DV; i += 32) acc = fmaf(vs[j * DV + i], vs[(j + 1) * DV + i], acc);
        acc = warp_sum(acc);
        if (ln == 0) gs[j] = acc;
      }
    }
    __syncthreads();
    constexpr int kCols = kSplitThreads / kTPC;  // columns per pass
    const int part = tid % kTPC;
    const unsigned pmask = ((1u << kTPC) - 1) << ((tid & 31) & ~(kTPC - 1));
    TF *pool = reinterpret_cast<TF *>(sv.W) + c0 * DV;
    const int m4 = (m + 3) & ~3;  // rows of y_k written by the SVD phase (zero beyond m)
    for (int k0 = 0; k0 < rk; k0 += kCols) {
      const int k = k0 + tid / kTPC;
      if (k >= rk) break;  // whole groups of kTPC lanes leave together
      RRCol c;
      c.nch = DV / (4 * kTPC);
      const float *y = ws + L.y + (int64_t)k * L.m4;
#pragma unroll
      for (int i = 0; i < kRRChunks; ++i) {
        c.x[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i >= c.nch) continue;
        const int row = rr_row(part, i, 0);
        if (row < m4) c.x[i] = *reinterpret_cast<const float4 *>(y + row);
      }
      // H_{m-1} first: pairs (j - 1, j) for j = m-1, m-3, ..., then H_0 alone if m is odd
      int j = m - 1;
      for (; j >= 1; j -= 2) rr_apply2(c, part, vs + (j - 1) * DV, vs + j * DV, ts[j - 1], ts[j], gs[j - 1], pmask);
      if (j == 0) rr_apply(c, part, vs, ts[0], pmask);
#pragma unroll
      for (int i = 0; i < kRRChunks; ++i) {
        if (i >= c.nch) break;
        const int row = rr_row(part, i, 0);
#pragma unroll
        for (int e = 0; e < 4; ++e) Elem<TF>::store(pool + (int64_t)k * DV + row + e, f4get(c.x[i], e));
      }
    }
  }
}

int64_t split_floats_per_head(int factor_dtype, int m_max, int r_max, int d_v) {
  if (factor_dtype != SEED_F32) return gram_floats_per_head(m_max, r_max);
  return SplitLayout(m_max, r_max, kDK, d_v).per_head;
}

template <int VAR, typename TF, int DV, int MR>
static cudaError_t launch_split_t(SplitArgs a, int n_heads, int64_t chunk, cudaStream_t s) {
  const int up = (a.m_max + 3) & ~3;
  const int qr_bytes = (a.m_max * (kDK + DV) + 4 * up + 2 * a.m_max * a.m_max) * 4;
  const int qr_threads = a.m_max > 0 ? qr_team_stride(a.m_max) * 2 : 32;
  const int svd_bytes = svd_heads_per_cta<MR>() * SvdWarpSmem<MR>::FLOATS * 4;
  const int rk4 = (a.r_max + 3) / 4 * 4;
  const int rb_u = MR * MR + 2 * rk4 * MR, rb_w = a.m_max * DV + 2 * ((a.m_max + 3) & ~3);
  const int rb_bytes = ((rb_u > rb_w ? rb_u : rb_w) + 4) * 4;
  auto k1 = qr_phase<VAR, TF, DV>;
  auto k2 = svd_phase<TF, DV, MR>;
  auto k3 = rebuild_phase<VAR, TF, DV, MR>;
  cudaError_t e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, qr_bytes);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, svd_bytes);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k3, cudaFuncAttributeMaxDynamicSharedMemorySize, rb_bytes);
  if (e != cudaSuccess) return e;
  for (int64_t h0 = 0; h0 < n_heads; h0 += chunk) {
    const int n = (int)(n_heads - h0 < chunk ? n_heads - h0 : chunk);
    a.head0 = (int)h0;
    a.n_group = n;
    k1<<<n, qr_threads, qr_bytes, s>>>(a);
    k2<<<(n + svd_heads_per_cta<MR>() - 1) / svd_heads_per_cta<MR>(), 32 * kSvdWarps, svd_bytes, s>>>(a);
    k3<<<dim3(n, 2), kSplitThreads, rb_bytes, s>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

template <int VAR, typename TF, int DV>
static cudaError_t launch_split_m(const SplitArgs &a, int n, int64_t chunk, cudaStream_t s) {
  if (a.m_max <= 16) return launch_split_t<VAR, TF, DV, 16>(a, n, chunk, s);
  if (a.m_max <= 32) return launch_split_t<VAR, TF, DV, 32>(a, n, chunk, s);
  if (a.m_max <= 48) return launch_split_t<VAR, TF, DV, 48>(a, n, chunk, s);
  return launch_split_t<VAR, TF, DV, 64>(a, n, chunk, s);
}

template <typename TF, int DV>
static cudaError_t launch_split_v(const SplitArgs &a, int n, int64_t chunk, cudaStream_t s) {
  // Only the scale layout differs between variants here.
  if (a.sv.variant == SEED_KDA) return launch_split_m<SEED_KDA, TF, DV>(a, n, chunk, s);
  return launch_split_m<SEED_GDN, TF, DV>(a, n, chunk, s);
}

cudaError_t launch_recompress_split(const StateView &sv, int factor_dtype, float *trunc_err,
                                    int32_t *sweeps, int m_max, int r_max, float *ws,
                                    int64_t chunk, cudaStream_t s) {
  // 16-bit factors take the Gram route (recompress_gram.cu)
  if (factor_dtype != SEED_F32)
    return launch_recompress_gram(sv, factor_dtype, trunc_err, sweeps, m_max, r_max, ws, chunk, s);
  SplitArgs a{sv, ws, 0, 0, m_max, -1, m_max, r_max, trunc_err, sweeps, 0};
  const int n = sv.n_heads;
  auto one = [&](const SplitArgs &x) {
    return sv.d_v == 64 ? launch_split_v<float, 64>(x, n, chunk, s) : launch_split_v<float, 128>(x, n, chunk, s);
  };
  if (!sv.rank || m_max <= 16) return one(a);
  // Ragged ranks: one launch per column class (m in (16c - 16, 16c]), each sized
  // for its class, so that small heads do not run in the threads, registers and
  // loop lengths of the largest; heads of other classes leave at once.
  for (int hi = 16; hi - 16 < m_max; hi += 16) {
    SplitArgs c = a;
    c.m_max = hi < m_max ? hi : m_max;
    c.m_lo = hi == 16 ? -1 : hi - 16;  // the first class also takes heads with no columns
    const cudaError_t e = one(c);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// ---- fixed scratch for seed_recompress_noalloc ---------------------------------------------
// One array per device that loads the library.  Host code sees only a stand-in
// for it, so its device address is asked for on every call (a host-side lookup
// that allocates nothing): an address kept from an earlier call would go stale
// if the caller reset the device in between.
static __device__ __align__(256) float g_recompress_scratch[kNoAllocScratchFloats];

cudaError_t noalloc_scratch(float **ptr) {
  void *p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_recompress_scratch);
  if (e != cudaSuccess) return e;
  *ptr = static_cast<float *>(p);
  return cudaSuccess;
}

}  // namespace seedk
