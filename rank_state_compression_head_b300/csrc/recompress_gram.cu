// Recompression of 16-bit factors through a Cholesky of the value-side Gram
// matrix, in three phases over a caller-provided device workspace.
//
// What is computed is the recompression of "Shallow Encoding Emits Deep
// Memories" (thelatestinai.com list view, Table 1: the decode compresses back to
// rank R every W steps): the best rank-r approximation of U_eff W^T.  The route
// differs from the QR-of-both-factors route of recompress_split.cu:
//
//   G_w = W^T W = R_b^T R_b    (tensor cores; Cholesky, so Q_b = W R_b^{-1} has
//                               orthonormal columns and U_eff W^T = B Q_b^T)
//   B   = U_eff R_b^T          (tensor cores, R_b in three bf16 terms)
//   M   = B^T B = Y Sigma^2 Y^T (tensor cores, B in three bf16 terms; pivoted Cholesky +
//                               one-sided Jacobi, evd_warp.cuh)
//   U'  = U_eff R_b^T Y_r = B Y_r,   W' = W R_b^{-1} Y_r = Q_b Y_r  (tensor cores)
//
// With Q_b orthonormal the singular values of U_eff W^T are those of B, Y holds
// B's right singular vectors, and B Y_r Y_r^T Q_b^T is the best rank-r
// approximation, written U' W'^T with W' orthonormal and U' = X_r Sigma_r, the
// same layout as the QR route.  Neither factor is QR-factorized.
//
// Accuracy.  G_w is formed from exact products of the stored 16-bit values with
// fp32 accumulation; B carries an error of order eps |U_eff| |W| (as the QR
// route's core does), M = B^T B one of order eps sigma_1 (sigma_1 + |U_eff| |W|),
// so the kept directions (the r largest) are resolved to about that over
// sigma_r^2 - sigma_{r+1}^2.  Through G_w, a column of W is resolved down to its
// part outside the span of the earlier columns at about sqrt(kCholFloor) = 1e-3
// of its norm: finer than the 2^-9 rounding that a stored 16-bit column already
// carries, so nothing the storage keeps is lost.  Below that, the pivot's row of
// R_b is dropped and the column is carried by its projections.  32-bit factors
// keep the QR route.
//
//   gram_phase     one CTA per head: both factors into shared memory (cp.async),
//                  G_w on mma.sync, Cholesky by one warp in registers,
//                  B = U diag(c) R_b^T on mma.sync (KDA: rows times D), then
//                  M = B^T B on mma.sync from B's three bf16 terms stored over the
//                  tiles, half its rows at a time; M and R_b to the workspace
//   evd_phase      one lane group per head: eigenvectors of M (evd_warp.cuh),
//                  truncation error, the kept Y to the workspace
//   gram_rebuild   one CTA per (head, factor): Z = diag(c) R_b^T Y_r (U) or
//                  R_b^{-1} Y_r (W, back substitution), F' = F Z on mma.sync
//                  with Z split into two 16-bit terms (16 or 22 significant
//                  bits, far finer than the factor's own rounding),
//                  KDA's row scale applied to U', lazy scales reset
//
// Workspace per head (fp32): M [m][m4], R_b [m][m4] (upper, row-major), Y [r][m4]
// (m4 = m rounded up to 4), eight words of class lists, each region on 16 bytes,
// the whole on 256 bytes.  With ragged ranks each 16-column class gets its own
// three launches, sized for it: with the state's class order (seed.h) over
// exactly the class's positions in it, chunk by chunk; without it, over a list
// of the chunk's heads of the class that gram_classify builds first.  Either way
// every lane group of an evd_phase CTA has a head of the class.
#include "evd_warp.cuh"

#include <type_traits>

namespace seedk {

// Cholesky pivot floor, relative to the column's squared norm (1e-3 in norm, finer
// than the 2^-9 rounding of a stored 16-bit column).
constexpr float kCholFloor = 1e-6f;
constexpr int kGramThreads = 128;

// Per-head slot (floats): M, R_b, Y, then eight words of the class lists: word c
// of slot i names the i-th head (slot) of column class c in this chunk, and words
// 4..7 of slot 0 hold the four class counts.
struct GramLayout {
  int64_t mq, rb, y, lst, per_head;  // offsets and stride in floats
  int m4;
  __host__ __device__ GramLayout(int m, int r) {
    m4 = (m + 3) & ~3;
    mq = 0;                        // M: m rows of m4 floats (16-byte rows)
    rb = mq + (int64_t)m * m4;     // R_b: the same
    y = rb + (int64_t)m * m4;
    lst = y + (int64_t)r * m4;
    per_head = (lst + 8 + 63) & ~(int64_t)63;
  }
};

int64_t gram_floats_per_head(int m_max, int r_max) { return GramLayout(m_max, r_max).per_head; }

struct GramArgs {
  StateView sv;
  float *ws;
  int head0, n_group;
  int m_max, m_lo;  // this launch serves heads with m_lo < m <= m_max
  int layout_m, r_max;
  float *trunc_err;
  int32_t *sweeps;
  int cls;          // column class of this launch (its heads from the class list), or -1: every slot
  int pos_lo, pos_hi;  // with the state's class order: this launch's positions in it
};

__device__ inline bool gram_head(const GramArgs &p, int h, int &r, int &m) {
  r = p.sv.rank_of(h);
  m = r + p.sv.growth * p.sv.steps;
  return r >= 0 && r <= p.r_max && m <= p.layout_m;
}
__device__ inline bool gram_in_class(const GramArgs &p, int m) { return m > p.m_lo && m <= p.m_max; }

// The workspace slot and the head that item i of this launch serves: position
// pos_lo + i of the state's class order (slot = position - head0, the chunk's first
// position), an entry of this chunk's class list, or slot i (head head0 + i).
// False past the end.
__device__ inline bool gram_item(const GramArgs &p, int i, int &b, int &h) {
  if (p.sv.order) {
    const int pos = p.pos_lo + i;
    if (pos >= p.pos_hi) return false;
    b = pos - p.head0;
    h = p.sv.order[pos];
    return true;
  }
  if (p.cls < 0) {
    b = i;
    h = p.head0 + i;
    return i < p.n_group;
  }
  const GramLayout L(p.layout_m, p.r_max);
  if (i >= reinterpret_cast<const int *>(p.ws + L.lst)[4 + p.cls]) return false;
  b = reinterpret_cast<const int *>(p.ws + (int64_t)i * L.per_head + L.lst)[p.cls];
  h = p.head0 + b;
  return true;
}

// Class lists of one chunk, in slot order: column class c holds the heads with
// 16c < m <= 16c + 16 (class 0 also those with no columns).  One CTA: per pass of
// 1024 slots a ballot per class, warp offsets scanned in shared memory.  A head
// whose rank disagrees with the state's r_max goes in no list and is reported.
__global__ void __launch_bounds__(1024) gram_classify(const GramArgs p, int n_cls) {
  __shared__ int woff[32][4];
  __shared__ int base[4];
  const GramLayout L(p.layout_m, p.r_max);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid < 4) base[tid] = 0;
  for (int i0 = 0; i0 < p.n_group; i0 += 1024) {
    const int b = i0 + tid;
    int c = -1;
    if (b < p.n_group) {
      int r, m;
      const int h = p.head0 + b;
      if (gram_head(p, h, r, m)) c = m <= 16 ? 0 : (m - 1) / 16;
      else if (p.sv.status) p.sv.status[h] = SEED_ERR_INVALID_ARG;
      if (c >= n_cls) c = -1;
    }
    unsigned bal[4];
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) bal[cc] = __ballot_sync(0xffffffffu, c == cc);
    if (lane < 4) woff[warp][lane] = __popc(bal[lane]);
    __syncthreads();
    if (tid < 4) {
      int acc = base[tid];
      for (int w = 0; w < 32; ++w) {
        const int t = woff[w][tid];
        woff[w][tid] = acc;
        acc += t;
      }
      base[tid] = acc;
    }
    __syncthreads();
    if (c >= 0) {
      const int pos = woff[warp][c] + __popc(bal[c] & ((1u << lane) - 1u));
      reinterpret_cast<int *>(p.ws + (int64_t)pos * L.per_head + L.lst)[c] = b;
    }
    __syncthreads();
  }
  if (tid < 4) reinterpret_cast<int *>(p.ws + L.lst)[4 + tid] = base[tid];
}

// ---- tensor-core helpers (mma.sync m16n8k16, bf16/fp16 in, fp32 accumulate) --------------
__device__ static inline void g_cp_async16(void *dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ static inline void g_cp_commit_wait_all() {
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
}
__device__ static inline void g_cp_async4(void *dst, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ static inline void g_cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// all but the most recently committed group have landed
__device__ static inline void g_cp_wait_but_last() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ static inline void g_ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ static inline void g_ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
template <typename TF>
__device__ static inline void g_mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  Mma16<TF>::mma(d, a[0], a[1], a[2], a[3], b0, b1);
}
// (x, y) as NTERM packed 16-bit terms t0 + t1 (+ t2): 16 (bf16) or 22 (fp16)
// significant bits with two terms, 24 with three, while the terms stay in the type's
// normal range (fp16 callers scale Z by a power of two)
template <typename TF, int NTERM>
__device__ static inline void g_split(float x, float y, uint32_t (&t)[3]) {
  t[0] = Mma16<TF>::pack(x, y);
  float2 h = Mma16<TF>::unpack(t[0]);
  x -= h.x; y -= h.y;
  t[1] = Mma16<TF>::pack(x, y);
  if constexpr (NTERM == 3) {
    h = Mma16<TF>::unpack(t[1]);
    t[2] = Mma16<TF>::pack(x - h.x, y - h.y);
  }
}

// fp16 operands of F Z: each row n of Z^T (a column of Z) scaled by a power of two so
// that its largest magnitude lies in [2^10, 2^11), which keeps the three terms of the
// split inside fp16's normal range; the output column is scaled back exactly.  bf16
// shares fp32's exponent range and needs no scaling (factor 1).
template <typename TF>
__device__ inline void scale_z_rows(float *Zt, int zp, int rows, int cols, float *unscale) {
  for (int n = threadIdx.x; n < rows; n += blockDim.x) {
    float mx = 0.f;
    for (int j = 0; j < cols; ++j) mx = fmaxf(mx, fabsf(Zt[n * zp + j]));
    int e = 0;
    if (std::is_same<TF, __half>::value && mx > 0.f) frexpf(mx, &e);  // mx in [2^(e-1), 2^e)
    const int sh = std::is_same<TF, __half>::value && mx > 0.f ? 11 - e : 0;
    const float f = ldexpf(1.f, sh);
    if (sh)
      for (int j = 0; j < cols; ++j) Zt[n * zp + j] *= f;
    unscale[n] = ldexpf(1.f, -sh);
  }
}

// Shared layout of gram_phase (bytes): both factor tiles (column j of the factor
// in row j, rows padded by 16 bytes so that ldmatrix hits distinct banks; the W
// tile's space is reused for Z once G_w is formed), the three bf16 terms of half of
// B = U_eff R_b^T over both tiles once they have been read (S_BYTES), G_w / R_b
// (row i at i * GP floats), the scales, the original diagonal of G_w.
template <int DV, int MR>
struct GramSmem {
  static constexpr int USTR = kDK * 2 + 16, WSTR = DV * 2 + 16;
  static constexpr int GP = MR + 1;
  static constexpr int ZP = MR + 8;  // Z row pitch (floats): row n = column n of Z
  static constexpr int WZ_BYTES = MR * WSTR > MR * ZP * 4 ? MR * WSTR : MR * ZP * 4;
  static constexpr int U_OFF = 0;
  static constexpr int W_OFF = U_OFF + MR * USTR;  // W tile, then Z
  static constexpr int TILE_BYTES = W_OFF + WZ_BYTES;
  static constexpr int KP = 64 + 8;                // bf16 a row of a term of half of B
  static constexpr int S_BYTES = 3 * MR * KP * 2;  // the three terms, over the tiles
  static constexpr int G_OFF = ((TILE_BYTES > S_BYTES ? TILE_BYTES : S_BYTES) + 15) & ~15;
  static constexpr int SC_OFF = G_OFF + ((MR * GP * 4 + 15) & ~15);
  static constexpr int DG_OFF = SC_OFF + (MR > kDK ? MR : kDK) * 4;
  static constexpr int ZS_OFF = DG_OFF + MR * 4;  // per-column unscale of Z (fp16)
  static constexpr int RR_OFF = ZS_OFF + MR * 4;  // the Cholesky's current row of R_b, two buffers
  static constexpr int BYTES = RR_OFF + 2 * MR * 4;
};

// Cholesky G_w = R_b^T R_b by one warp, the matrix in registers: lane l owns
// columns l and l + 32 of the upper triangle (column c needs rows 0..c only, so
// the first column's array stops at 32).  Step j: the pivot's lane hands round
// the current G[j][j]; every lane forms its entries of row j of R_b (R[j][c] =
// G[j][c] / r_jj, r_jj on the diagonal), writes them over G_w's row j and into a
// row buffer in shared memory; after a warp barrier every lane reads row j back
// with 16-byte broadcast loads and takes R[j][i] R[j][c] off its rows i > j.  A
// pivot below kCholFloor of its column's squared norm means the column lies in
// the span of the earlier ones to within the resolution of the Gram matrix: its
// row of R_b is dropped (zero) and the column is represented by its projections.
// G_w in Gw (row i at i * GP); row j of R_b replaces row j of G_w (entries c >= j;
// below the diagonal untouched), dg gets the original diagonal; rr holds 2 * MR
// floats (the row buffer, double-buffered by step parity).
template <int MR>
__device__ inline void chol_warp(float *Gw, float *dg, float *rr, int m) {
  constexpr int GP = MR + 1;
  constexpr bool TWO = MR > 32;
  constexpr int NA = MR < 32 ? MR : 32;
  const int lane = threadIdx.x & 31;
  const int c0 = lane, c1 = lane + 32;
  // the columns as pairs of consecutive rows, updated on the packed fp32
  // instructions; every row past the step is updated, those from m on included (their
  // multipliers are entries of columns that are never written back), so the unrolled
  // steps carry no per-row conditions
  float2 gA[NA / 2], gB[TWO ? MR / 2 : 1];
#pragma unroll
  for (int i = 0; i < NA / 2; ++i)
    gA[i] = c0 < MR ? make_float2(Gw[2 * i * GP + c0], Gw[(2 * i + 1) * GP + c0]) : make_float2(0.f, 0.f);
  if constexpr (TWO) {
#pragma unroll
    for (int i = 0; i < MR / 2; ++i)
      gB[i] = c1 < MR ? make_float2(Gw[2 * i * GP + c1], Gw[(2 * i + 1) * GP + c1]) : make_float2(0.f, 0.f);
  }
  auto el = [](const float2 &v, int odd) { return odd ? v.y : v.x; };
  if (c0 < m) dg[c0] = Gw[c0 * GP + c0];
  if (TWO && c1 < m) dg[c1] = Gw[c1 * GP + c1];
  __syncwarp();
#pragma unroll
  for (int j = 0; j < MR; ++j) {
    if (j < m) {
      float own;  // my column's entry in row j (pivot lane: the diagonal)
      if constexpr (TWO) own = j < 32 ? el(gA[j < NA ? j / 2 : 0], j & 1) : el(gB[j / 2], j & 1);
      else own = el(gA[j < NA ? j / 2 : 0], j & 1);
      const float d = __shfl_sync(0xffffffffu, own, j & 31);
      // 1 / r_jj and r_jj from one reciprocal square root (a couple of ulp)
      const bool keep = d > kCholFloor * dg[j];
      const float inv = keep ? rsqrtf(d) : 0.f;
      const float rjj = d * inv;
      const float rA = j < NA && c0 > j ? el(gA[j < NA ? j / 2 : 0], j & 1) * inv : (c0 == j ? rjj : 0.f);
      float rB = 0.f;
      if constexpr (TWO) rB = c1 > j ? el(gB[j / 2], j & 1) * inv : (c1 == j ? rjj : 0.f);
      float *row = rr + (j & 1) * MR;
      if (c0 < MR) row[c0] = rA;
      if (TWO && c1 < MR) row[c1] = rB;
      if (c0 >= j && c0 < m) Gw[j * GP + c0] = rA;
      if (TWO && c1 >= j && c1 < m) Gw[j * GP + c1] = rB;
      __syncwarp();
      // S[i][c] -= R[j][i] R[j][c] for the pairs holding a row past j ((-r) v rounds as r (-v))
      const float4 *row4 = reinterpret_cast<const float4 *>(row);
      const float2 mA = make_float2(-rA, -rA), mB = make_float2(-rB, -rB);
#pragma unroll
      for (int q = (j + 1) / 4; q < MR / 4; ++q) {
        const float4 v = row4[q];
        const float2 v01 = make_float2(v.x, v.y), v23 = make_float2(v.z, v.w);
        if (4 * q + 1 > j) {
          if (4 * q < NA) gA[4 * q < NA ? 2 * q : 0] = __ffma2_rn(v01, mA, gA[4 * q < NA ? 2 * q : 0]);
          if constexpr (TWO) gB[2 * q] = __ffma2_rn(v01, mB, gB[2 * q]);
        }
        if (4 * q + 3 > j) {
          if (4 * q + 2 < NA) gA[4 * q + 2 < NA ? 2 * q + 1 : 0] = __ffma2_rn(v23, mA, gA[4 * q + 2 < NA ? 2 * q + 1 : 0]);
          if constexpr (TWO) gB[2 * q + 1] = __ffma2_rn(v23, mB, gB[2 * q + 1]);
        }
      }
    }
  }
}

// G[i0..i0+15][j0..j0+7] += F^T F over `depth` rows of the tiles, F column j in
// smem row j (stride STR bytes): exact products of the stored 16-bit values,
// fp32 accumulation.
template <typename TF, int STR>
__device__ inline void gram_tile(uint32_t base, int i0, int j0, int depth, float (&d)[4]) {
  const int lane = threadIdx.x & 31;
  const uint32_t a_row = base + (uint32_t)((i0 + (lane & 7) + ((lane >> 3) & 1) * 8) * STR + (lane >> 4) * 16);
  const uint32_t b_row = base + (uint32_t)((j0 + (lane & 7)) * STR + (lane >> 3) * 16);
  for (int k0 = 0; k0 < depth; k0 += 32) {
    uint32_t b[4], a0[4], a1[4];
    g_ldsm_x4(b_row + k0 * 2, b);
    g_ldsm_x4(a_row + k0 * 2, a0);
    g_ldsm_x4(a_row + (k0 + 16) * 2, a1);
    g_mma<TF>(d, a0, b[0], b[1]);
    g_mma<TF>(d, a1, b[2], b[3]);
  }
}

// D[r][i][n] += sum_j F[i][j] Z[j][n] for the rows i of tile r (i0 + 16 r .. + 15), the
// columns n0..n0+7 and j < depth16: F column j in smem row j of the tile at `tile`
// (stride STR bytes), Z row n at Zt + n * ZP (fp32, split once into NTERM 16-bit terms,
// g_split; products exact, fp32 accumulation).
template <typename TF, int STR, int ZP, int NR, int KMAX, int NTERM>
__device__ inline void tiles_times_z(uint32_t tile, const float *Zt, int i0, int n0, int depth16,
                                     float (&d)[NR][4]) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int rsel = (lane & 7) + ((lane >> 4) << 3);
  const int cofs = ((lane >> 3) & 1) * 8;
  constexpr int NK = KMAX / 16;
  uint32_t bz[NK][2][3];
#pragma unroll
  for (int kk = 0; kk < NK; ++kk) {
    if (16 * kk < depth16) {
      const float2 z0 = *reinterpret_cast<const float2 *>(Zt + (n0 + g) * ZP + 16 * kk + 2 * t);
      const float2 z1 = *reinterpret_cast<const float2 *>(Zt + (n0 + g) * ZP + 16 * kk + 8 + 2 * t);
      g_split<TF, NTERM>(z0.x, z0.y, bz[kk][0]);
      g_split<TF, NTERM>(z1.x, z1.y, bz[kk][1]);
    }
  }
#pragma unroll
  for (int r = 0; r < NR; ++r) {
#pragma unroll
    for (int kk = 0; kk < NK; ++kk) {
      if (16 * kk < depth16) {
        uint32_t a[4];
        g_ldsm_x4_t(tile + (uint32_t)((16 * kk + rsel) * STR + (i0 + 16 * r + cofs) * 2), a);
#pragma unroll
        for (int q = 0; q < NTERM; ++q) g_mma<TF>(d[r], a, bz[kk][0][q], bz[kk][1][q]);
      }
    }
  }
}

// ---- phase 1: G_w, its Cholesky, B = U_eff R_b^T, M = B^T B ---------------------------------
// Resident CTAs to plan registers for (shared memory allows about this many).
template <int MR>
constexpr int gram_min_blocks() { return MR <= 16 ? 8 : MR <= 32 ? 6 : MR <= 48 ? 5 : 4; }

template <typename TF, int VAR, int DV, int MR>
__global__ void __launch_bounds__(kGramThreads, gram_min_blocks<MR>()) gram_phase(const GramArgs p) {
  constexpr int DK = kDK;
  using L = GramSmem<DV, MR>;
  constexpr int GP = L::GP, ZP = L::ZP;
  constexpr bool KDA = VAR == SEED_KDA;
  extern __shared__ __align__(128) unsigned char smem[];
  int slot, h;
  if (!gram_item(p, blockIdx.x, slot, h)) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const StateView &sv = p.sv;
  int r, m;
  if (!gram_head(p, h, r, m) || !gram_in_class(p, m)) return;  // bad ranks: reported by evd_phase
  const int m16 = (m + 15) & ~15;
  const int64_t c0 = sv.col0(h);
  float *Gw = reinterpret_cast<float *>(smem + L::G_OFF);
  float *Zt = reinterpret_cast<float *>(smem + L::W_OFF);
  float *sc = reinterpret_cast<float *>(smem + L::SC_OFF);
  float *dg = reinterpret_cast<float *>(smem + L::DG_OFF);
  float *zsc = reinterpret_cast<float *>(smem + L::ZS_OFF);

  // ---- factors into shared memory, padding columns zero ---------------------------------
  {
    const TF *Ug = reinterpret_cast<const TF *>(sv.U) + c0 * DK;
    const TF *Wg = reinterpret_cast<const TF *>(sv.W) + c0 * DV;
    constexpr int UCH = DK / 8, WCH = DV / 8;  // 16-byte chunks per column
    for (int idx = tid; idx < m16 * UCH; idx += kGramThreads) {
      const int j = idx / UCH, c = idx % UCH;
      unsigned char *dst = smem + L::U_OFF + j * L::USTR + c * 16;
      if (j < m) g_cp_async16(dst, Ug + (int64_t)j * DK + c * 8);
      else *reinterpret_cast<uint4 *>(dst) = make_uint4(0, 0, 0, 0);
    }
    for (int idx = tid; idx < m16 * WCH; idx += kGramThreads) {
      const int j = idx / WCH, c = idx % WCH;
      unsigned char *dst = smem + L::W_OFF + j * L::WSTR + c * 16;
      if (j < m) g_cp_async16(dst, Wg + (int64_t)j * DV + c * 8);
      else *reinterpret_cast<uint4 *>(dst) = make_uint4(0, 0, 0, 0);
    }
    if (KDA) {
      for (int i = tid; i < DK; i += kGramThreads) sc[i] = sv.scale[(int64_t)h * DK + i];
    } else {
      for (int j = tid; j < m16; j += kGramThreads) sc[j] = j < m ? sv.scale[c0 + j] : 0.f;
    }
    g_cp_commit_wait_all();
  }
  __syncthreads();

  // ---- G_w = W^T W on the tensor cores ----------------------------------------------------------
  {
    const int ncol = m16 / 8, per = (m16 / 16) * ncol;
    const uint32_t wb = smem_u32(smem + L::W_OFF);
    for (int task = warp; task < per; task += kGramThreads / 32) {
      const int i0 = (task / ncol) * 16, j0 = (task % ncol) * 8;
      // only tiles that reach the upper triangle: the Cholesky reads nothing below the
      // diagonal into its results (those registers are updated but never read back)
      if (j0 + 8 <= i0) continue;
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      gram_tile<TF, L::WSTR>(wb, i0, j0, DV, d);
#pragma unroll
      for (int e = 0; e < 4; ++e) Gw[(i0 + g + (e >> 1) * 8) * GP + j0 + 2 * t + (e & 1)] = d[e];
    }
  }
  __syncthreads();

  // ---- Cholesky G_w = R_b^T R_b (upper, in place) by warp 0 --------------------------------------
  if (warp == 0) chol_warp<MR>(Gw, dg, reinterpret_cast<float *>(smem + L::RR_OFF), m);
  __syncthreads();

  // ---- Z = diag(c) R_b^T (Z[l][j] = c_l R_b[j][l]), stored by rows of Z^T --------------------------
  // (the W tile is no longer needed); KDA's row scale D is applied to B instead
  for (int idx = tid; idx < m16 * ZP; idx += kGramThreads) {
    const int j = idx / ZP, l = idx % ZP;
    float z = 0.f;
    if (j < m && l < m && l >= j) z = KDA ? Gw[j * GP + l] : Gw[j * GP + l] * sc[l];
    Zt[idx] = z;
  }
  __syncthreads();
  scale_z_rows<TF>(Zt, ZP, m16, m16, zsc);
  __syncthreads();

  // ---- B = U Z (U_eff = U diag(c)), or diag(D) (U R_b^T) for KDA, on the tensor cores -----------
  // A task is one column tile of B over half of its rows (four row tiles), Z's columns
  // split once per task; the results are held in registers until every warp has read
  // both tiles, then stored over them.
  {
    constexpr int NW = kGramThreads / 32, NTK = 2 * (MR / 8) / NW;  // tasks per warp at most
    const int ntile = m16 / 8, per = 2 * ntile;
    const uint32_t ub = smem_u32(smem + L::U_OFF);
    float bacc[NTK][4][4];
#pragma unroll
    for (int q = 0; q < NTK; ++q) {
      const int task = warp + q * NW;
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int e = 0; e < 4; ++e) bacc[q][r][e] = 0.f;
      if (task < per)
        tiles_times_z<TF, L::USTR, ZP, 4, MR, 3>(ub, Zt, (task / ntile) * 64, (task % ntile) * 8, m16, bacc[q]);
    }
    __syncthreads();  // both tiles are read: they take B, in three bf16 terms, half its rows at a time

    // ---- M = B^T B on the tensor cores ------------------------------------------------------
    // B = B0 + B1 + B2 (bf16 terms of the fp32 values: 24 significant bits, whatever the
    // factor type) and M = sum of Bp^T Bq over p + q <= 2, the six products that carry
    // it to fp32 accuracy (those left out are below 2^-24 of it), with fp32 accumulation.
    // Term p of rows 64h .. 64h + 63 lies at Sp[n * KP + i] (column n of B as a row, so
    // that both operands load by ldmatrix).  A warp keeps its tiles of the upper triangle
    // (16 x 8, j-tile J and l-tile L with L >= 2J) in registers over both halves.
    constexpr int KP = L::KP;                           // bf16 a row of a term: 144 bytes
    constexpr int NUT = (MR / 16) * (MR / 8) - (MR / 16) * (MR / 16 - 1);  // upper tiles
    constexpr int TPW = (NUT + NW - 1) / NW;            // tiles a warp, at most
    static_assert(L::S_BYTES <= L::G_OFF, "the three terms of half of B lie before G_w");
    __nv_bfloat16 *S0 = reinterpret_cast<__nv_bfloat16 *>(smem + L::U_OFF);
    const uint32_t s_base = smem_u32(S0);
    constexpr uint32_t TERM = MR * KP * 2;              // bytes a term
    int tJ[TPW], tL[TPW];
    float dm[TPW][4];
#pragma unroll
    for (int s_ = 0; s_ < TPW; ++s_) {
      int k = warp + NW * s_, J = 0;
      while (J < MR / 16 && k >= MR / 8 - 2 * J) { k -= MR / 8 - 2 * J; ++J; }
      tJ[s_] = J < MR / 16 && 16 * J < m16 ? J : -1;
      tL[s_] = 2 * J + k;
      if (tJ[s_] >= 0 && 8 * tL[s_] >= m16) tJ[s_] = -1;
#pragma unroll
      for (int e = 0; e < 4; ++e) dm[s_][e] = 0.f;
    }
    for (int h = 0; h < 2; ++h) {
#pragma unroll
      for (int q = 0; q < NTK; ++q) {
        const int task = warp + q * NW;
        if (task < per && task / ntile == h) {
          const int n0 = (task % ntile) * 8;
#pragma unroll
          for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int i = 16 * r + g + (e >> 1) * 8, n = n0 + 2 * t + (e & 1);
              float v = bacc[q][r][e] * zsc[n];
              if (KDA) v *= sc[64 * h + i];
              const __nv_bfloat16 b0 = __float2bfloat16_rn(v);
              const float r1 = v - __bfloat162float(b0);
              const __nv_bfloat16 b1 = __float2bfloat16_rn(r1);
              const __nv_bfloat16 b2 = __float2bfloat16_rn(r1 - __bfloat162float(b1));
              S0[n * KP + i] = b0;
              S0[MR * KP + n * KP + i] = b1;
              S0[2 * MR * KP + n * KP + i] = b2;
            }
        }
      }
      __syncthreads();  // this half's terms are in place
#pragma unroll
      for (int s_ = 0; s_ < TPW; ++s_) {
        if (tJ[s_] < 0) continue;
        // A: rows 16J .. of each term (ldmatrix x4); B: rows 8L .. (x2)
        const uint32_t a_row = s_base + (uint32_t)(((16 * tJ[s_] + (lane & 7) + ((lane >> 3) & 1) * 8) * KP + (lane >> 4) * 8) * 2);
        const uint32_t b_row = s_base + (uint32_t)(((8 * tL[s_] + (lane & 7)) * KP + ((lane >> 3) & 1) * 8) * 2);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          uint32_t A[3][4], Bq[3][2];
#pragma unroll
          for (int p_ = 0; p_ < 3; ++p_) {
            g_ldsm_x4(a_row + p_ * TERM + kk * 32, A[p_]);
            asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
                         : "=r"(Bq[p_][0]), "=r"(Bq[p_][1]) : "r"(b_row + p_ * TERM + kk * 32));
          }
          g_mma<__nv_bfloat16>(dm[s_], A[0], Bq[0][0], Bq[0][1]);
          g_mma<__nv_bfloat16>(dm[s_], A[0], Bq[1][0], Bq[1][1]);
          g_mma<__nv_bfloat16>(dm[s_], A[1], Bq[0][0], Bq[0][1]);
          g_mma<__nv_bfloat16>(dm[s_], A[0], Bq[2][0], Bq[2][1]);
          g_mma<__nv_bfloat16>(dm[s_], A[2], Bq[0][0], Bq[0][1]);
          g_mma<__nv_bfloat16>(dm[s_], A[1], Bq[1][0], Bq[1][1]);
        }
      }
      __syncthreads();  // the terms have been read
    }

    // ---- M to the workspace: each entry with j <= l once, and its mirror ---------------------
    const GramLayout W(p.layout_m, p.r_max);
    float *ws = p.ws + (int64_t)slot * W.per_head;
#pragma unroll
    for (int s_ = 0; s_ < TPW; ++s_) {
      if (tJ[s_] < 0) continue;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = 16 * tJ[s_] + g + (e >> 1) * 8, l = 8 * tL[s_] + 2 * t + (e & 1);
        if (j <= l && l < m) {
          ws[W.mq + (int64_t)j * W.m4 + l] = dm[s_][e];
          if (j != l) ws[W.mq + (int64_t)l * W.m4 + j] = dm[s_][e];
        }
      }
    }
  }

  // ---- R_b to the workspace ---------------------------------------------------------------------
  const GramLayout W(p.layout_m, p.r_max);
  float *ws = p.ws + (int64_t)slot * W.per_head;
  for (int i = warp; i < m; i += kGramThreads / 32)  // R_b by rows of W.m4, zero beyond m
    for (int l = lane; l < W.m4; l += 32) ws[W.rb + (int64_t)i * W.m4 + l] = (l >= i && l < m) ? Gw[i * GP + l] : 0.f;
}

// ---- phase 2: eigenvectors of M, one lane group per head -------------------------------------
template <int MR>
constexpr int evd_group() { return MR <= 32 ? 16 : 32; }
template <int MR>
constexpr int evd_heads_per_cta() { return kSvdWarps * (32 / evd_group<MR>()); }

// Resident CTAs to plan registers for: the register Jacobi holds three MR-float
// arrays per lane, so the larger cores get fewer, fatter lanes.
template <int MR>
constexpr int evd_min_blocks() { return MR <= 16 ? 8 : MR <= 32 ? 5 : MR <= 48 ? 5 : 4; }

template <int MR>
__global__ void __launch_bounds__(32 * kSvdWarps, evd_min_blocks<MR>()) evd_phase(const GramArgs p) {
  constexpr int HW = evd_group<MR>();
  using SW = SvdWarpSmem<MR>;
  extern __shared__ __align__(16) float smem_f[];
  const int grp = threadIdx.x / HW, lane = threadIdx.x & (HW - 1);
  const unsigned gmask = HW == 32 ? 0xffffffffu : 0xffffu << (threadIdx.x & 16);
  int b, h;
  if (!gram_item(p, blockIdx.x * evd_heads_per_cta<MR>() + grp, b, h)) return;
  const StateView &sv = p.sv;
  int r, m;
  if (!gram_head(p, h, r, m)) {  // rank table disagrees with r_max: touch nothing
    if (lane == 0 && sv.status) sv.status[h] = SEED_ERR_INVALID_ARG;
    return;
  }
  if (!gram_in_class(p, m)) {  // a head listed in a class too small for it: touch nothing
    if (p.sv.order && lane == 0 && sv.status) sv.status[h] = SEED_ERR_INVALID_ARG;
    return;
  }
  float *sw = smem_f + grp * SW::FLOATS;
  float *T = sw + SW::T_OFF;
  const GramLayout W(p.layout_m, p.r_max);
  float *ws = p.ws + (int64_t)b * W.per_head;
  const float *Mw = ws + W.mq;

  // M is scaled by a power of four to a largest diagonal below one (its square root,
  // sigma, by a power of two); the core loads it straight into registers
  float dmax = 0.f;
  for (int c = lane; c < m; c += HW) dmax = fmaxf(dmax, Mw[(int64_t)c * W.m4 + c]);
#pragma unroll
  for (int o = HW / 2; o > 0; o >>= 1) dmax = fmaxf(dmax, __shfl_xor_sync(gmask, dmax, o));
  int e = 0;
  if (dmax > 0.f) frexpf(dmax, &e);
  const int e2 = e >= 0 ? (e + 1) / 2 : -((-e) / 2);  // ceil(e / 2)
  const float mscale = ldexpf(1.f, -2 * e2), sunscale = ldexpf(1.f, e2);
  const float tol = 1e-4f;  // 16-bit factors: their own rounding is 2^-9
  const int sweeps = evd_warp_core<MR, HW>(m, tol, sqrtf(tol), sw, Mw, W.m4, mscale);
  const float *sig2 = sw + SW::S_OFF, *inv = sw + SW::I_OFF;
  const int *order = reinterpret_cast<const int *>(sw + SW::O_OFF);
  if (lane == 0) {
    float err = 0.f;
    for (int k = r; k < m; ++k) err += sig2[order[k]];
    if (p.trunc_err) p.trunc_err[h] = sqrtf(err) * sunscale;
    if (p.sweeps) p.sweeps[h] = sweeps;
    if (sv.status) sv.status[h] = sweeps < 0 ? SEED_ERR_NOT_CONVERGED : SEED_OK;
  }
  // kept eigenvectors y_k[x] = (Rt^T J)[x][order[k]] / sigma_k, rows m..m4-1 zero
  const int rk = r < m ? r : m;
  float *Y = ws + W.y;
  for (int k = 0; k < rk; ++k) {
    const int col = order[k];
    const float ik = inv[col];
    const float *f = T + col * SW::TP;
    for (int x = lane; x < W.m4; x += HW) Y[k * W.m4 + x] = x < m ? f[x] * ik : 0.f;
  }
}

// ---- phase 3: F' = F Z ---------------------------------------------------------------------------
// blockIdx.y = 0: U' = U_eff R_b^T Y_r (Z = diag(c) R_b^T Y_r on the stored U; KDA: rows
// of U Z times D); blockIdx.y = 1: W' = W R_b^{-1} Y_r.
template <int DV, int MR>
struct RebuildSmem {
  static constexpr int STR = kDK * 2 + 16;      // tile row stride (bytes), the larger factor
  static constexpr int RP = MR + 4;             // R_b row pitch (floats; 16-byte rows)
  static constexpr int YP = MR + 4;             // Y row pitch: row n holds y_n[j] for every j
  static constexpr int ZP = MR + 2;             // Z row pitch (floats): row n = column n of Z;
                                                // 2 mod 4 keeps both access patterns at 2-way
  static constexpr int T_OFF = 0;               // factor tile
  static constexpr int R_OFF = T_OFF + MR * STR;
  static constexpr int Y_OFF = R_OFF + MR * RP * 4;
  static constexpr int O_OFF = R_OFF;           // the output tile, over R_b and Y once Z is formed
  static constexpr int RY_BYTES = MR * STR > (MR * (RP + YP) + MR) * 4 ? MR * STR : (MR * (RP + YP) + MR) * 4;
  static constexpr int Z_OFF = R_OFF + RY_BYTES;
  static constexpr int S_OFF = Z_OFF + MR * ZP * 4;  // scales c [MR] or D [DK]
  static constexpr int ZS_OFF = S_OFF + (MR > kDK ? MR : kDK) * 4;  // per-column unscale of Z
  static constexpr int BYTES = ZS_OFF + MR * 4;
};

template <typename TF, int VAR, int DV, int MR>
__global__ void __launch_bounds__(kGramThreads) gram_rebuild(const GramArgs p) {
  constexpr int DK = kDK;
  using L = RebuildSmem<DV, MR>;
  constexpr int RP = L::RP, YP = L::YP, ZP = L::ZP;
  constexpr bool KDA = VAR == SEED_KDA;
  extern __shared__ __align__(128) unsigned char smem[];
  int slot, h;
  if (!gram_item(p, blockIdx.x, slot, h)) return;
  const bool isU = blockIdx.y == 0;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const StateView &sv = p.sv;
  int r, m;
  if (!gram_head(p, h, r, m) || !gram_in_class(p, m)) return;
  const int rk = r < m ? r : m;
  if (rk == 0) {  // nothing kept: only the scales go back to one
    if (isU) {
      if (KDA) for (int i = tid; i < DK; i += kGramThreads) sv.scale[(int64_t)h * DK + i] = 1.f;
    }
    return;
  }
  const int rows = isU ? DK : DV;
  const int m16 = (m + 15) & ~15, rk8 = (rk + 7) & ~7;
  const int64_t c0 = sv.col0(h);
  const GramLayout W(p.layout_m, p.r_max);
  const float *ws = p.ws + (int64_t)slot * W.per_head;
  float *Rb = reinterpret_cast<float *>(smem + L::R_OFF);
  float *Ys = reinterpret_cast<float *>(smem + L::Y_OFF);   // y_n[j] at n * YP + j
  float *Z = reinterpret_cast<float *>(smem + L::Z_OFF);    // [rk8][ZP]: z_n[j] at n * ZP + j
  float *sc = reinterpret_cast<float *>(smem + L::S_OFF);
  TF *pool = reinterpret_cast<TF *>(isU ? sv.U : sv.W) + c0 * rows;

  // ---- R_b, Y, the scales (first copy group), the factor tile (second) -----------------------
  // R_b upper (zero below the diagonal and beyond m) and Y (zero beyond m and rk) by
  // 16-byte copies of their rows, both stored by rows of W.m4 floats; Z zero
  {
    constexpr int RC = RP / 4;  // 16-byte chunks of a row of R_b in shared memory
    const int m4c = W.m4 / 4 < RC ? W.m4 / 4 : RC;
    for (int idx = tid; idx < m16 * RC; idx += kGramThreads) {
      const int i = idx / RC, c = idx % RC;
      float *dst = Rb + i * RP + 4 * c;
      if (i < m && c < m4c) g_cp_async16(dst, ws + W.rb + (int64_t)i * W.m4 + 4 * c);
      else *reinterpret_cast<float4 *>(dst) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const int rk8r = (rk + 7) & ~7;
    for (int idx = tid; idx < rk8r * RC; idx += kGramThreads) {
      const int n = idx / RC, c = idx % RC;
      float *dst = Ys + n * YP + 4 * c;
      if (n < rk && c < m4c) g_cp_async16(dst, ws + W.y + (int64_t)n * W.m4 + 4 * c);
      else *reinterpret_cast<float4 *>(dst) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  if (isU) {
    if (KDA) for (int i = tid; i < DK; i += kGramThreads) g_cp_async4(sc + i, sv.scale + (int64_t)h * DK + i);
    else for (int j = tid; j < m; j += kGramThreads) g_cp_async4(sc + j, sv.scale + c0 + j);
  }
  g_cp_commit();
  {
    const int CH = rows / 8;
    for (int idx = tid; idx < m16 * CH; idx += kGramThreads) {
      const int j = idx / CH, c = idx % CH;
      unsigned char *dst = smem + L::T_OFF + j * L::STR + c * 16;
      if (j < m) g_cp_async16(dst, pool + (int64_t)j * rows + c * 8);
      else *reinterpret_cast<uint4 *>(dst) = make_uint4(0, 0, 0, 0);
    }
  }
  g_cp_commit();
  for (int idx = tid; idx < rk8 * ZP; idx += kGramThreads) Z[idx] = 0.f;
  g_cp_wait_but_last();  // R_b, Y and the scales are in; the tile may still be on its way
  __syncthreads();

  // ---- Z ------------------------------------------------------------------------------------
  if (isU) {
    // z_n[l] = c_l sum_{j <= l} y_n[j] R_b[j][l], 4 x 4 blocks of (n, l) a thread, four
    // j at a time (rows of Y and R_b are zero from m on)
    const int nbn = (rk + 3) / 4, nbl = (m + 3) / 4;
    for (int blk = tid; blk < nbn * nbl; blk += kGramThreads) {
      const int nb = blk / nbl, lb = blk % nbl;
      float acc[4][4] = {};
      for (int j4 = 0; j4 <= lb; ++j4) {
        float ys[4][4], rs[4][4];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          const float4 y = *reinterpret_cast<const float4 *>(Ys + (4 * nb + a) * YP + 4 * j4);
          ys[a][0] = y.x; ys[a][1] = y.y; ys[a][2] = y.z; ys[a][3] = y.w;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float4 rv = *reinterpret_cast<const float4 *>(Rb + (4 * j4 + u) * RP + 4 * lb);
          rs[u][0] = rv.x; rs[u][1] = rv.y; rs[u][2] = rv.z; rs[u][3] = rv.w;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[a][c] = fmaf(ys[a][u], rs[u][c], acc[a][c]);
      }
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int n = 4 * nb + a, l = 4 * lb + c;
          if (n < rk && l < m) Z[n * ZP + l] = KDA ? acc[a][c] : acc[a][c] * sc[l];
        }
    }
  } else {
    // R_b Z = Y by back substitution in row panels of 16 from the bottom.  The inverses
    // of the panels' diagonal 16 x 16 blocks are formed first, a thread per column of a
    // block (back substitution of a unit vector; a zero pivot, a dropped row, gives a
    // zero row), in Y's space once Y has been copied into Z.  Each panel then takes its
    // triangle as a product with its block's inverse (two threads a column of Z, each
    // warp on the same half of the rows), and the rows above lose the panel's
    // contribution.  In exact arithmetic this is the back substitution itself.
    float *rinv = Ys + MR * YP;  // 1 / R_b[i][i] (0 for a dropped row), after Y
    float *Dv = Ys;              // the block inverses, 256 floats each, once Y is in Z
    for (int idx = tid; idx < rk * m; idx += kGramThreads) {
      const int n = idx / m, i = idx % m;
      Z[n * ZP + i] = Ys[n * YP + i];
    }
    for (int i = tid; i < m; i += kGramThreads) {
      const float piv = Rb[i * RP + i];
      rinv[i] = piv != 0.f ? 1.f / piv : 0.f;
    }
    __syncthreads();
    const int np = (m + 15) / 16;
    for (int tsk = tid; tsk < 16 * np; tsk += kGramThreads) {
      const int kb = tsk >> 4, c = tsk & 15;
      const int bb1 = m - 16 * kb, bb0 = bb1 > 16 ? bb1 - 16 : 0, w = bb1 - bb0;
      float x[16];
#pragma unroll
      for (int q = 15; q >= 0; --q) {
        float s_ = q == c ? 1.f : 0.f;
#pragma unroll
        for (int u = 15; u > q; --u)
          if (u < w) s_ = fmaf(-Rb[(bb0 + q) * RP + bb0 + u], x[u], s_);
        x[q] = q < w ? s_ * rinv[bb0 + q] : 0.f;
      }
#pragma unroll
      for (int q = 0; q < 16; ++q) Dv[kb * 256 + q * 16 + c] = x[q];
    }
    __syncthreads();
    static_assert((MR / 16) * 256 <= MR * YP, "the block inverses fit Y's space");
    for (int b1 = m; b1 > 0; b1 -= 16) {
      const int b0 = b1 > 16 ? b1 - 16 : 0, kb = (m - b1) / 16;
      // z_n[b0 + q] = sum_u Dinv[q][u] z_n[b0 + u], Dinv upper triangular (zero past the
      // block); thread t: column n = t % 64, rows 8h .. 8h + 7 with h = t / 64
      const int n = tid & 63, h = tid >> 6;
      const bool act = n < rk;
      float zp[16];
      if (act) {
#pragma unroll
        for (int u = 0; u < 16; ++u) zp[u] = Z[n * ZP + b0 + u];
      }
      __syncthreads();  // every thread has the panel's old values
      if (act) {
        const float *D = Dv + kb * 256;
        if (h == 0) {
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            float s_ = 0.f;
#pragma unroll
            for (int u = q; u < 16; ++u) s_ = fmaf(D[q * 16 + u], zp[u], s_);
            if (b0 + q < b1) Z[n * ZP + b0 + q] = s_;
          }
        } else {
#pragma unroll
          for (int q = 8; q < 16; ++q) {
            float s_ = 0.f;
#pragma unroll
            for (int u = q; u < 16; ++u) s_ = fmaf(D[q * 16 + u], zp[u], s_);
            if (b0 + q < b1) Z[n * ZP + b0 + q] = s_;
          }
        }
      }
      __syncthreads();
      // z_n[i] -= sum_{b0 <= l < b1} R_b[i][l] z_n[l] for the rows i < b0, in the same
      // order as one element at a time, by 4 x 4 blocks of (n, i) a thread: columns
      // nb + nbn a (neighbouring threads read neighbouring rows of Z) and rows
      // 4 ib .. 4 ib + 3 (shared by neighbouring threads: broadcast reads of R_b);
      // rows of Z from rk on are zero and stay unwritten
      const int nbn = (rk + 3) / 4, nib = (b0 + 3) / 4;
      for (int blk = tid; blk < nbn * nib; blk += kGramThreads) {
        const int ib = blk / nbn, nb = blk % nbn;
        float acc[4][4];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int i = 4 * ib + c;
            acc[a][c] = i < b0 ? Z[(nb + nbn * a) * ZP + i] : 0.f;
          }
        for (int l = b0; l < b1; ++l) {
          float zl[4], rl[4];
#pragma unroll
          for (int a = 0; a < 4; ++a) zl[a] = Z[(nb + nbn * a) * ZP + l];
#pragma unroll
          for (int c = 0; c < 4; ++c) rl[c] = Rb[(4 * ib + c) * RP + l];
#pragma unroll
          for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[a][c] = fmaf(-rl[c], zl[a], acc[a][c]);
        }
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int n = nb + nbn * a, i = 4 * ib + c;
            if (n < rk && i < b0) Z[n * ZP + i] = acc[a][c];
          }
      }
      __syncthreads();
    }
  }
  float *zsc = reinterpret_cast<float *>(smem + L::ZS_OFF);
  __syncthreads();
  scale_z_rows<TF>(Z, ZP, rk8, m16, zsc);
  g_cp_commit_wait_all();
  __syncthreads();

  // ---- F' = F Z on the tensor cores (Z in two 16-bit terms) -------------------------------------
  {
    const int g = lane >> 2, t = lane & 3;
    // a task is one column tile over four row tiles (all of a 64-row factor, half of a
    // 128-row one), Z's columns split once per task
    const int ntile = rk8 / 8, per = (rows / 64) * ntile;
    const uint32_t tb = smem_u32(smem + L::T_OFF);
    TF *out = reinterpret_cast<TF *>(smem + L::O_OFF);
    for (int task = warp; task < per; task += kGramThreads / 32) {
      const int ib = (task / ntile) * 64, n0 = (task % ntile) * 8;
      float d[4][4] = {};
      // two terms of Z: their 2^-17 (bf16) or 2^-23 (fp16) is far below the rounding
      // of the stored factor that the product becomes
      tiles_times_z<TF, L::STR, ZP, 4, MR, 2>(tb, Z, ib, n0, m16, d);
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int i0 = ib + 16 * r;
        // d[r][e]: row i (element of the column), output column n; stochastic rounding:
        // one Philox block for the lane's four elements (counter: its even column, row)
        uint4 rb = make_uint4(0u, 0u, 0u, 0u);
        if (sv.rounding == kRoundStochastic)
          rb = sr_bits(sv.sr_seed, c0 + n0 + 2 * t, (uint32_t)(i0 + g), isU ? kSrRebuildU : kSrRebuildW);
        const uint32_t words[4] = {rb.x, rb.y, rb.z, rb.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int i = i0 + g + (e >> 1) * 8, n = n0 + 2 * t + (e & 1);
          float v = d[r][e] * zsc[n];
          if (isU && KDA) v *= sc[i];
          out[n * (L::STR / 2) + i] = Mma16<TF>::cvt(store_value<TF>(v, sv.rounding, words[e]));
        }
      }
    }
  }
  __syncthreads();
  {
    const int CH = rows / 8;
    for (int idx = tid; idx < rk * CH; idx += kGramThreads) {
      const int n = idx / CH, c = idx % CH;
      *reinterpret_cast<uint4 *>(pool + (int64_t)n * rows + c * 8) =
          *reinterpret_cast<const uint4 *>(smem + L::O_OFF + n * L::STR + c * 16);
    }
  }
  if (isU) {  // every read of the scales happened before the last barrier
    if (KDA) for (int i = tid; i < DK; i += kGramThreads) sv.scale[(int64_t)h * DK + i] = 1.f;
    else for (int k = tid; k < rk; k += kGramThreads) sv.scale[c0 + k] = 1.f;
  }
}

template <typename TF, int VAR, int DV, int MR>
static cudaError_t launch_gram_t(const GramArgs &a, cudaStream_t s) {
  using L1 = GramSmem<DV, MR>;
  using L3 = RebuildSmem<DV, MR>;
  const int evd_bytes = evd_heads_per_cta<MR>() * SvdWarpSmem<MR>::FLOATS * 4;
  auto k1 = gram_phase<TF, VAR, DV, MR>;
  auto k2 = evd_phase<MR>;
  auto k3 = gram_rebuild<TF, VAR, DV, MR>;
  cudaError_t e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, L1::BYTES);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, evd_bytes);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k3, cudaFuncAttributeMaxDynamicSharedMemorySize, L3::BYTES);
  if (e != cudaSuccess) return e;
  const int n = a.n_group;  // the class's heads are a prefix of its list; the rest leave at once
  k1<<<n, kGramThreads, L1::BYTES, s>>>(a);
  k2<<<(n + evd_heads_per_cta<MR>() - 1) / evd_heads_per_cta<MR>(), 32 * kSvdWarps, evd_bytes, s>>>(a);
  k3<<<dim3(n, 2), kGramThreads, L3::BYTES, s>>>(a);
  return cudaGetLastError();
}

template <typename TF, int VAR, int DV>
static cudaError_t launch_gram_m(const GramArgs &a, cudaStream_t s) {
  if (a.m_max <= 16) return launch_gram_t<TF, VAR, DV, 16>(a, s);
  if (a.m_max <= 32) return launch_gram_t<TF, VAR, DV, 32>(a, s);
  if (a.m_max <= 48) return launch_gram_t<TF, VAR, DV, 48>(a, s);
  return launch_gram_t<TF, VAR, DV, 64>(a, s);
}

template <typename TF, int DV>
static cudaError_t launch_gram_v(const GramArgs &a, cudaStream_t s) {
  // Only the scale layout differs between variants here.
  if (a.sv.variant == SEED_KDA) return launch_gram_m<TF, SEED_KDA, DV>(a, s);
  return launch_gram_m<TF, SEED_GDN, DV>(a, s);
}

cudaError_t launch_recompress_gram(const StateView &sv, int factor_dtype, float *trunc_err, int32_t *sweeps,
                                   int m_max, int r_max, float *ws, int64_t chunk, cudaStream_t s) {
  GramArgs a{sv, ws, 0, 0, m_max, -1, m_max, r_max, trunc_err, sweeps, -1, 0, 0};
  const int n = sv.n_heads;
  auto one = [&](const GramArgs &x) {
    if (factor_dtype == SEED_F16)
      return sv.d_v == 64 ? launch_gram_v<__half, 64>(x, s) : launch_gram_v<__half, 128>(x, s);
    return sv.d_v == 64 ? launch_gram_v<__nv_bfloat16, 64>(x, s) : launch_gram_v<__nv_bfloat16, 128>(x, s);
  };
  // With the state's class order: chunks of consecutive positions, and in each one
  // launch triple per class present, sized for the class and covering exactly its
  // heads (a head's columns need only fit its class, so any m up to the class size).
  if (sv.order) {
    for (int64_t p0 = 0; p0 < n; p0 += chunk) {
      const int p1 = (int)(n - p0 < chunk ? n : p0 + chunk);
      for (int c = 0, begin = 0; c < 4; begin = sv.class_end[c], ++c) {
        const int lo = begin > p0 ? begin : (int)p0, hi = sv.class_end[c] < p1 ? sv.class_end[c] : p1;
        if (hi <= lo) continue;
        GramArgs x = a;
        x.head0 = (int)p0;
        x.n_group = hi - lo;
        x.pos_lo = lo;
        x.pos_hi = hi;
        x.m_max = 16 * (c + 1) < m_max ? 16 * (c + 1) : m_max;
        x.m_lo = -1;
        const cudaError_t e = one(x);
        if (e != cudaSuccess) return e;
      }
    }
    return cudaSuccess;
  }
  // Ragged ranks: per chunk, the heads are listed by 16-column class, and each
  // class gets its own launches, sized for it, over its list.
  const bool ragged = sv.rank && m_max > 16;
  const int n_cls = ragged ? (m_max + 15) / 16 : 1;
  for (int64_t h0 = 0; h0 < n; h0 += chunk) {
    a.head0 = (int)h0;
    a.n_group = (int)(n - h0 < chunk ? n - h0 : chunk);
    if (ragged) {
      gram_classify<<<1, 1024, 0, s>>>(a, n_cls);
      const cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
    for (int c = 0; c < n_cls; ++c) {
      GramArgs x = a;
      if (ragged) {
        x.cls = c;
        x.m_max = 16 * (c + 1) < m_max ? 16 * (c + 1) : m_max;
        x.m_lo = c == 0 ? -1 : 16 * c;  // the first class also takes heads with no columns
      }
      const cudaError_t e = one(x);
      if (e != cudaSuccess) return e;
    }
  }
  return cudaSuccess;
}

}  // namespace seedk
