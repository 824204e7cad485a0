// Fused read-out + exact factored update for 16-bit factors (bf16 or fp16), with
// the two contractions of a step on the tensor cores.
//
// "Shallow Encoding Emits Deep Memories", picx.dev summary, Methodology >
// Exact Update (Lemma 2); thelatestinai.com list view, Table 1 (decode
// column: read-out and update of each recurrent state).
//
// A persistent grid of CTAs of 128 threads (as many as fit on the device) walks
// the heads blockIdx.x, blockIdx.x + gridDim.x, ... with one shared-memory stage
// a CTA.  A head's copies form two groups, U and the per-head vectors first and
// W second, and each half of the stage is refilled with the next head's data as
// soon as the current head has read it: the next U during this head's W pass,
// the next W during its update and the next head's U pass.  So every CTA keeps
// copies in flight while it computes.  With the state's class order there is one
// launch per column class, each with a stage sized for its class (seed.h).  The
// threads copy the factor columns (contiguous in HBM) with asynchronous 16-byte
// copies into rows padded to 272 bytes, so that the ldmatrix reads below hit 32
// distinct banks.  Per head the CTA does
//
//   split    rows [k_hi; k_lo; q_hi; q_lo] of the U-pass operand, once (smem)
//   U pass   X[4][m] = [k_hi; k_lo; q_hi; q_lo] U_stored          (mma m16n8k16)
//   scale    x_k = c * (X0 + X1),  x_q = c * (X2 + X3)              (column scales)
//   W pass   [Wx_k Wx_q] = W [x_k_hi x_k_lo x_q_hi x_q_lo]           (mma m16n8k16)
//
// Products of 16-bit values are exact in fp32 and the accumulation is fp32.
// The fp32 operands (k, q, x) enter as a 16-bit pair hi + lo, so they carry 16
// (bf16) or 22 (fp16) significant bits; the result differs from fp32 dot
// products by less than fp32 summation-order noise times ~2^-8.  The read-out
// and the appended columns then follow Lemma 2 exactly as in the CUDA-core
// kernel (decode.cu); an appended element is rounded to the factor type once,
// to nearest or stochastically (seed.h, seed_rounding), and the read-out uses
// the rounded value.
#include "common.cuh"

#include <atomic>

namespace seedk {

constexpr int kMmaThreads = 128;

template <int VAR, int DV, int MAXC>
struct MmaStage {
  static constexpr int DK = kDK;
  static constexpr bool KDA = VAR == SEED_KDA;
  static constexpr int USTR = DK * 2 + 16;  // padded bytes per U column
  static constexpr int WSTR = DV * 2 + 16;  // padded bytes per W column
  static constexpr int U_OFF = 0;
  static constexpr int W_OFF = U_OFF + MAXC * USTR;
  static constexpr int Q_OFF = W_OFF + MAXC * WSTR;
  static constexpr int K_OFF = Q_OFF + DK * 4;
  static constexpr int A_OFF = K_OFF + DK * 4;
  static constexpr int V_OFF = A_OFF + DK * 4;
  static constexpr int VB_OFF = V_OFF + DV * 4;
  static constexpr int SC_OFF = VB_OFF + DV * 4;                 // column scales [MAXC], or D [DK] (KDA)
  static constexpr int AL_OFF = SC_OFF + (KDA ? DK : MAXC) * 4;  // KDA: alpha [DK]
  static constexpr int G_OFF = AL_OFF + (KDA ? DK * 4 : 0);      // gate, beta, A (scalars)
  static constexpr int BYTES = G_OFF + 16;
  static_assert(W_OFF % 16 == 0 && Q_OFF % 16 == 0 && SC_OFF % 16 == 0 && BYTES % 16 == 0,
                "16-byte copies");
};

template <int VAR, int DV, int MAXC>
struct MmaSmem {
  using S = MmaStage<VAR, DV, MAXC>;
  static constexpr int NX = VAR == SEED_MAMBA2 ? 1 : 2;
  static constexpr int XLD = MAXC + 16;                                    // bf16 per x row
  static constexpr int XS_OFF = S::BYTES;                                  // bf16 [2 NX][XLD]
  static constexpr int WX_OFF = XS_OFF + ((2 * NX * XLD * 2 + 15) & ~15);  // f32 [NX][DV]
  static constexpr int SCAL_OFF = WX_OFF + NX * DV * 4;                    // f32 [NW][8]
  static constexpr int ALD = kDK + 8;                                      // 16-bit per operand row
  static constexpr int AS_OFF = SCAL_OFF + (kMmaThreads / 32) * 8 * 4;     // [2 NX][ALD]: U-pass rows
  static constexpr int BYTES = AS_OFF + 2 * NX * ALD * 2;
};

__device__ static inline void cp_async16(void *dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ static inline void cp_async4(void *dst, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ static inline void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ static inline void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ static inline void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ static inline void ldsm_x2(uint32_t addr, uint32_t &r0, uint32_t &r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}
__device__ static inline void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// CTAs an SM should hold: as many as the stage's shared memory allows for the
// larger classes (5 of 40.5 KB, 7 of 32 KB), 8 for the smaller ones
template <int MAXC>
constexpr int mma_min_blocks() { return MAXC > 48 ? 5 : MAXC > 32 ? 7 : 8; }

template <typename TF, int VAR, int DV, int MAXC>
__global__ void __launch_bounds__(kMmaThreads, mma_min_blocks<MAXC>()) decode_mma_kernel(const DecodeArgs p) {
  constexpr int DK = kDK;
  constexpr int NT = kMmaThreads;
  using S = MmaStage<VAR, DV, MAXC>;
  using L = MmaSmem<VAR, DV, MAXC>;
  constexpr int NX = L::NX;
  constexpr int NA = 2 * NX;  // rows of the U-pass operand: hi/lo of k (and q)
  constexpr bool KDA = VAR == SEED_KDA;
  constexpr bool M2 = VAR == SEED_MAMBA2;
  constexpr int NSW = (DK > DV ? DK : DV) / 32;  // warps holding scalar partials
  static_assert(MAXC % 16 == 0 && MAXC <= 64, "column tiles");

  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char *const st = smem;  // the stage: U, W and the per-head vectors
  TF *xs = reinterpret_cast<TF *>(smem + L::XS_OFF);
  float *wxs = reinterpret_cast<float *>(smem + L::WX_OFF);
  float *scal = reinterpret_cast<float *>(smem + L::SCAL_OFF);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;  // mma fragment coordinates
  const StateView &sv = p.sv;
  const int growth = sv.growth;
  const int G = gridDim.x;
  const int first = blockIdx.x;
  const int nmine = first < p.count ? (p.count - first + G - 1) / G : 0;
  // head of launch item i: through the class order when the launch has one
  auto head_at = [&](int i) { return sv.order ? sv.order[p.pos0 + i] : i; };

  // What the copies of an item need: its head, rank, columns and sink direction,
  // read ahead of the copies (below), so that the chain of dependent reads is off
  // their path.
  struct Item {
    int h, r, m, dir;
    int64_t c0;
  };
  auto describe = [&](int h, Item &it) {
    it.h = h;
    it.r = h >= 0 ? sv.rank_of(h) : -1;
    it.m = it.r + growth * sv.steps;
    const bool ok = it.r >= 0 && it.m <= MAXC;
    it.c0 = ok ? sv.col0(h) : 0;
    it.dir = ok ? sv.dir_of(h) : 0;
  };
  auto valid = [&](const Item &it) { return it.r >= 0 && it.m <= MAXC; };

  // The copies of an item form two commit groups (empty for no item, so that the
  // group counting stays uniform): U and the per-head vectors, then W.
  auto issue_u = [&](const Item &it) {
    if (valid(it)) {
      const int h = it.h, m = it.m;
      const int64_t c0 = it.c0;
      const TF *Ug = reinterpret_cast<const TF *>(sv.U) + c0 * DK;
      // 16-byte chunk c of column j: a thread keeps its chunk and walks the
      // columns NT / chunks-per-column apart (pointer increments only)
      constexpr int UCH = DK * 2 / 16;  // 16-byte chunks per column
      constexpr int UJS = NT / UCH;     // column step of a thread
      {
        const int c = tid % UCH;
        unsigned char *d = st + S::U_OFF + (tid / UCH) * S::USTR + c * 16;
        const TF *src = Ug + (int64_t)(tid / UCH) * DK + c * 8;
        for (int j = tid / UCH; j < m; j += UJS, d += UJS * S::USTR, src += UJS * DK) cp_async16(d, src);
      }
      if (tid < DK / 4) {
        cp_async16(st + S::Q_OFF + tid * 16, p.q + (int64_t)h * DK + tid * 4);
        cp_async16(st + S::K_OFF + tid * 16, p.k + (int64_t)h * DK + tid * 4);
        cp_async16(st + S::A_OFF + tid * 16, sv.a + (int64_t)h * DK + tid * 4);
        if (KDA) {
          cp_async16(st + S::SC_OFF + tid * 16, sv.scale + (int64_t)h * DK + tid * 4);
          cp_async16(st + S::AL_OFF + tid * 16, p.gate + (int64_t)h * DK + tid * 4);
        }
      } else if (tid < DK / 4 + DV / 4) {
        const int c = tid - DK / 4;
        cp_async16(st + S::V_OFF + c * 16, p.v + (int64_t)h * DV + c * 4);
        cp_async16(st + S::VB_OFF + c * 16, sv.vbar + (int64_t)it.dir * DV + c * 4);
      } else if (tid == DK / 4 + DV / 4) {
        float *gates = reinterpret_cast<float *>(st + S::G_OFF);
        if (!KDA) cp_async4(gates + 0, p.gate + h);
        if (!M2) cp_async4(gates + 1, p.beta + h);
        if (M2) cp_async4(gates + 2, p.A + it.dir);
      } else if (!KDA && scales_in_stage(c0, it.r + growth * sv.T)) {
        const int c = tid - DK / 4 - DV / 4 - 1;
        for (int cc = c; cc * 4 < m; cc += NT - DK / 4 - DV / 4 - 1)
          cp_async16(st + S::SC_OFF + cc * 16, sv.scale + c0 + cc * 4);
      }
    }
    cp_async_commit();
  };
  auto issue_w = [&](const Item &it) {
    if (valid(it)) {
      constexpr int WCH = DV * 2 / 16, WJS = NT / WCH;
      const int c = tid % WCH;
      unsigned char *d = st + S::W_OFF + (tid / WCH) * S::WSTR + c * 16;
      const TF *src = reinterpret_cast<const TF *>(sv.W) + it.c0 * DV + (int64_t)(tid / WCH) * DV + c * 8;
      for (int j = tid / WCH; j < it.m; j += WJS, d += WJS * S::WSTR, src += WJS * DV) cp_async16(d, src);
    }
    cp_async_commit();
  };

  // One stage, refilled in two halves as soon as each is free: item i+1's U and
  // vectors are copied in during item i's W pass and update (its U pass and scalars
  // have read them into registers by barrier B), and its W during item i's update
  // and item i+1's U pass (item i's W pass is done at barrier C).  So a CTA always
  // has copies in flight, and several CTAs per SM share the SM's bandwidth.
  Item cur, nxt;
  describe(nmine > 0 ? head_at(first) : -1, cur);
  issue_u(cur);
  issue_w(cur);
  // The next item's head index is read an iteration ahead and its rank and columns
  // at the top of the iteration before its copies are issued: after the step's
  // first items these reads have a whole iteration to arrive.
  int h_next = nmine > 1 ? head_at(first + G) : -1;

  for (int i = 0; i < nmine; ++i) {
    describe(h_next, nxt);
    h_next = i + 2 < nmine ? head_at(first + (i + 2) * G) : -1;
    cp_async_wait<1>();  // this thread's copies of item i's U and vectors have landed

    const int h = cur.h;
    const int r_h = cur.r;
    const int m = cur.m;
    const bool bad_rank = !valid(cur);
    const int64_t c0 = cur.c0;
    float *scw = reinterpret_cast<float *>(st + S::SC_OFF);
    if (!bad_rank && !KDA && !scales_in_stage(c0, r_h + growth * sv.T))
      for (int j = tid; j < m; j += NT) scw[j] = sv.scale[c0 + j];  // unaligned column scales
    __syncthreads();  // barrier A: item i's U and vectors are in shared memory
    if (tid == 0 && sv.status) sv.status[h] = bad_rank ? SEED_ERR_INVALID_ARG : SEED_OK;
    if (bad_rank) {  // nothing was copied for it; the stage is free
      issue_u(nxt);
      issue_w(nxt);
      cur = nxt;
      continue;
    }

    const uint32_t u_base = smem_u32(st + S::U_OFF), w_base = smem_u32(st + S::W_OFF);
    const float *qs = reinterpret_cast<const float *>(st + S::Q_OFF);
    const float *ks = reinterpret_cast<const float *>(st + S::K_OFF);
    const float *as = reinterpret_cast<const float *>(st + S::A_OFF);
    const float *vs = reinterpret_cast<const float *>(st + S::V_OFF);
    const float *vbs = reinterpret_cast<const float *>(st + S::VB_OFF);
    const float *scs = scw;
    const float *als = reinterpret_cast<const float *>(st + S::AL_OFF);
    const float *gts = reinterpret_cast<const float *>(st + S::G_OFF);
    float g = 0.f, beta = 0.f, dt = 0.f;
    if (VAR == SEED_GDN) { g = gts[0]; beta = gts[1]; }
    if (KDA) beta = gts[1];
    if (M2) { dt = gts[0]; g = expf(dt * gts[2]); }
    const int m16 = (m + 15) & ~15;

    // padding: x rows and W columns [m, m16) must be zero for the W pass
    if (tid < NA * 16) {
      const int j = m + (tid & 15);
      if (j < m16) xs[(tid >> 4) * L::XLD + j] = Mma16<TF>::cvt(0.f);
    }
    {
      constexpr int CH = DV * 2 / 16;  // 16-byte chunks of a W column read by the W pass
      for (int idx = tid; idx < (m16 - m) * CH; idx += NT) {
        const int j = m + idx / CH, c = idx % CH;
        *reinterpret_cast<uint4 *>(st + S::W_OFF + j * S::WSTR + c * 16) = make_uint4(0, 0, 0, 0);
      }
    }

    // ---- U-pass operand rows, split once: [k_hi; k_lo; q_hi; q_lo] (KDA: D k and
    // alpha D q; Mamba-2: C alone), thread t splits element t of each vector ---------------
    {
      TF *as_ = reinterpret_cast<TF *>(smem + L::AS_OFF);
      if (tid < DK) {
        float vk = M2 ? qs[tid] : ks[tid], vq = qs[tid];
        if (KDA) {
          vk *= scs[tid];
          vq *= als[tid] * scs[tid];
        }
        const TF kh = Mma16<TF>::cvt(vk);
        as_[tid] = kh;
        as_[L::ALD + tid] = Mma16<TF>::cvt(vk - Mma16<TF>::back(kh));
        if (NX == 2) {
          const TF qh = Mma16<TF>::cvt(vq);
          as_[2 * L::ALD + tid] = qh;
          as_[3 * L::ALD + tid] = Mma16<TF>::cvt(vq - Mma16<TF>::back(qh));
        }
      }
    }
    __syncthreads();  // barrier A2: the split operand rows are visible

    // ---- U pass: column tiles of 8, round robin over the warps -----------------------
    if (warp * 8 < m) {
      // A fragments (rows 0..7; rows from NA on repeat row 0 and their products are
      // not used): one ldmatrix of four 8x8 matrices covers two k-steps
      uint32_t a0[8], a2[8];
      {
        const int rr = lane & 7;
        const uint32_t arow = smem_u32(smem + L::AS_OFF) + (uint32_t)((rr < NA ? rr : 0) * L::ALD * 2 + (lane >> 3) * 16);
#pragma unroll
        for (int pp = 0; pp < 4; ++pp) {
          uint32_t r[4];
          ldsm_x4(arow + pp * 64, r);
          a0[2 * pp] = r[0];
          a2[2 * pp] = r[1];
          a0[2 * pp + 1] = r[2];
          a2[2 * pp + 1] = r[3];
        }
      }
      for (int n0 = warp * 8; n0 < m; n0 += NT / 4) {
      float d[4] = {0.f, 0.f, 0.f, 0.f}, e[4] = {0.f, 0.f, 0.f, 0.f};  // two chains of k-steps
      const uint32_t row_addr = u_base + (uint32_t)((n0 + (lane & 7)) * S::USTR + (lane >> 3) * 16);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        uint32_t b[4];
        ldsm_x4(row_addr + kk * 64, b);
        Mma16<TF>::mma(d, a0[2 * kk], 0u, a2[2 * kk], 0u, b[0], b[1]);
        Mma16<TF>::mma(e, a0[2 * kk + 1], 0u, a2[2 * kk + 1], 0u, b[2], b[3]);
      }
      d[0] += e[0];
      d[1] += e[1];
      // rows 2r and 2r+1 (hi, lo) of the same vector: lane 4g+t and lane 4(g+1)+t
      const float o0 = __shfl_down_sync(0xffffffffu, d[0], 4);
      const float o1 = __shfl_down_sync(0xffffffffu, d[1], 4);
      if (gq < NA && (gq & 1) == 0) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int j = n0 + 2 * tq + e;
          if (j < m) {
            const float c = KDA ? 1.f : scs[j];
            const float x = c * (e ? d[1] + o1 : d[0] + o0);
            const TF xh = Mma16<TF>::cvt(x);
            xs[gq * L::XLD + j] = xh;
            xs[(gq + 1) * L::XLD + j] = Mma16<TF>::cvt(x - Mma16<TF>::back(xh));
          }
        }
      }
      }
    }

    // ---- block scalars: thread t owns row t (< DK) and value column t (< DV) ----------
    // stochastic rounding of the appended elements: one Philox block a thread, words
    // x, y for U and W of column m, z, w for column m + 1 (KDA)
    uint4 rb = make_uint4(0u, 0u, 0u, 0u);
    if (sv.rounding == kRoundStochastic) rb = sr_bits(sv.sr_seed, c0 + m, (uint32_t)tid, kSrAppend);
    float S_loc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) S_loc[j] = 0.f;
    float kt = 0.f, qt = 0.f, at = 0.f, vt = 0.f, vbt = 0.f, alt = 0.f, Dt = 0.f, ct = 0.f;
    float unew0 = 0.f, unew1 = 0.f;
    if (tid < DK) {
      kt = ks[tid]; qt = qs[tid]; at = as[tid];
      if (VAR == SEED_GDN) {
        unew0 = store_value<TF>(kt, sv.rounding, rb.x);
        S_loc[0] = kt * at; S_loc[1] = qt * at; S_loc[2] = kt * qt; S_loc[3] = unew0 * qt;
      } else if (KDA) {
        alt = als[tid];
        Dt = scs[tid];
        const float Dn = alt * Dt;
        unew0 = store_value<TF>(kt / Dt, sv.rounding, rb.x);
        unew1 = store_value<TF>(kt / Dn, sv.rounding, rb.z);
        S_loc[0] = kt * at; S_loc[1] = alt * at * qt; S_loc[2] = alt * kt * qt; S_loc[3] = kt * qt;
        S_loc[6] = unew0 * Dn * qt; S_loc[7] = unew1 * Dn * qt;
      } else {
        unew0 = store_value<TF>(dt * kt, sv.rounding, rb.x);
        S_loc[0] = at * qt; S_loc[1] = kt * qt; S_loc[2] = unew0 * qt;
      }
    }
    if (tid < DV) {
      vt = vs[tid]; vbt = vbs[tid];
      S_loc[4] = vt * vbt; S_loc[5] = vbt * vbt;
    }
    if (!KDA && tid < m) ct = scs[tid];
    if (warp < NSW) {
      const float r = warp_reduce8(S_loc, lane);
      if ((lane & 3) == 0) scal[warp * 8 + reduce8_index(lane)] = r;
    }
    cp_async_wait<0>();  // and its copies of item i's W
    __syncthreads();  // barrier B: x, W, the padding and the scalar partials are visible
    issue_u(nxt);     // U and the vectors have been read: the next item's go in
    float Sg[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int w = 0; w < NSW; ++w) {
      const float4 lo = reinterpret_cast<const float4 *>(scal + w * 8)[0];
      const float4 hi = reinterpret_cast<const float4 *>(scal + w * 8)[1];
      Sg[0] += lo.x; Sg[1] += lo.y; Sg[2] += lo.z; Sg[3] += lo.w;
      Sg[4] += hi.x; Sg[5] += hi.y; Sg[6] += hi.z; Sg[7] += hi.w;
    }

    // ---- W pass: row tiles of 16 of W x, round robin over the warps -------------------
    // B fragments (the x rows, the same for every row tile), loaded once: columns n
    // from NA on repeat row 0 and their products are not used; k-steps past m16 are
    // loaded (inside the x rows) but not used
    constexpr int KS = MAXC / 16;
    uint32_t bx0[KS], bx1[KS];
    {
      const int rr = lane & 7;
      const uint32_t xrow = smem_u32(xs) + (uint32_t)(((rr < NA ? rr : 0) * L::XLD + (lane >> 3) * 8) * 2);
#pragma unroll
      for (int kk = 0; kk < KS; kk += 2) {
        if (kk + 1 < KS) {
          uint32_t r[4];
          ldsm_x4(xrow + kk * 32, r);
          bx0[kk] = r[0]; bx1[kk] = r[1]; bx0[kk + 1] = r[2]; bx1[kk + 1] = r[3];
        } else {
          ldsm_x2(xrow + kk * 32, bx0[kk], bx1[kk]);
        }
      }
    }
    for (int i0 = warp * 16; i0 < DV; i0 += NT / 2) {
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      const int rsel = (lane & 7) + ((lane >> 4) << 3);
      const int csel = i0 + ((lane >> 3) & 1) * 8;
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        if (kk * 16 < m16) {
          uint32_t a[4];
          ldsm_x4_t(w_base + (uint32_t)((kk * 16 + rsel) * S::WSTR + csel * 2), a);
          Mma16<TF>::mma(d, a[0], a[1], a[2], a[3], bx0[kk], bx1[kk]);
        }
      }
      if (tq < NX) {
        wxs[tq * DV + i0 + gq] = d[0] + d[1];
        wxs[tq * DV + i0 + gq + 8] = d[2] + d[3];
      }
    }
    __syncthreads();  // barrier C: W x complete; the stage is no longer read
    issue_w(nxt);

    // ---- update and read-out (registers, scal, wxs only) -------------------------------
    const float omega = __fdividef(Sg[4], Sg[5]);  // Sg[5] = |vbar|^2, about 1
    int bad = 0;
    TF *Uo = reinterpret_cast<TF *>(sv.U) + (c0 + m) * DK;
    TF *Wo = reinterpret_cast<TF *>(sv.W) + (c0 + m) * DV;
    float wx[NX];
#pragma unroll
    for (int j = 0; j < NX; ++j) wx[j] = tid < DV ? wxs[j * DV + tid] : 0.f;
    if (VAR == SEED_GDN) {
      const float coef = beta * (omega - g * Sg[0]);
      const float aq = fmaf(g, Sg[1], coef * Sg[2]);
      if (tid < DK) {
        const float an = fmaf(g, at, coef * kt);
        sv.a[(int64_t)h * DK + tid] = an;
        Elem<TF>::store(Uo + tid, unew0);
        bad |= !finite(an);
      }
      if (tid < DV) {
        const float eps = fmaf(-omega, vbt, vt);
        const float wn = store_value<TF>(beta * fmaf(-g, wx[0], eps), sv.rounding, rb.y);
        Elem<TF>::store(Wo + tid, wn);
        const float o = fmaf(vbt, aq, fmaf(g, wx[NX - 1], Sg[3] * wn));
        p.o[(int64_t)h * DV + tid] = o;
        bad |= !finite(o);
      }
      if (tid < m) sv.scale[c0 + tid] = g * ct;
      if (tid == m) sv.scale[c0 + m] = 1.f;
    } else if (KDA) {
      const float aq = Sg[1] - beta * Sg[0] * Sg[2] + beta * omega * Sg[3];
      if (tid < DK) {
        const float an = alt * fmaf(-beta * kt, Sg[0], at) + beta * omega * kt;
        sv.a[(int64_t)h * DK + tid] = an;
        sv.scale[(int64_t)h * DK + tid] = alt * Dt;
        Elem<TF>::store(Uo + tid, unew0);
        Elem<TF>::store(Uo + DK + tid, unew1);
        bad |= !finite(an);
      }
      if (tid < DV) {
        const float eps = fmaf(-omega, vbt, vt);
        const float w1 = store_value<TF>(-beta * wx[0], sv.rounding, rb.y);
        const float w2 = store_value<TF>(beta * eps, sv.rounding, rb.w);
        Elem<TF>::store(Wo + tid, w1);
        Elem<TF>::store(Wo + DV + tid, w2);
        const float o = fmaf(vbt, aq, wx[NX - 1] + w1 * Sg[6] + w2 * Sg[7]);
        p.o[(int64_t)h * DV + tid] = o;
        bad |= !finite(o);
      }
    } else {
      const float coef = dt * omega;
      const float aC = fmaf(g, Sg[0], coef * Sg[1]);
      if (tid < DK) {
        const float an = fmaf(g, at, coef * kt);
        sv.a[(int64_t)h * DK + tid] = an;
        Elem<TF>::store(Uo + tid, unew0);
        bad |= !finite(an);
      }
      if (tid < DV) {
        const float wn = store_value<TF>(fmaf(-omega, vbt, vt), sv.rounding, rb.y);
        Elem<TF>::store(Wo + tid, wn);
        const float o = fmaf(vbt, aC, fmaf(g, wx[0], Sg[2] * wn));
        p.o[(int64_t)h * DV + tid] = o;
        bad |= !finite(o);
      }
      if (tid < m) sv.scale[c0 + tid] = g * ct;
      if (tid == m) sv.scale[c0 + m] = 1.f;
    }
    // thread 0 wrote OK before barriers B and C, so this write lands after it
    if (bad && sv.status) sv.status[h] = SEED_ERR_NONFINITE;
    cur = nxt;
  }
  cp_async_wait<0>();
}

// A persistent grid: as many CTAs as fit on the device at once (or one per head
// when there are fewer heads), each walking its heads with the two-half refill.
template <typename TF, int VAR, int DV, int MAXC>
static cudaError_t launch_mma_t(const DecodeArgs &a, cudaStream_t s) {
  using L = MmaSmem<VAR, DV, MAXC>;
  auto kern = decode_mma_kernel<TF, VAR, DV, MAXC>;
  // attributes and the resident grid belong to (kernel, device): set and measure
  // them the first time this kernel runs on each device of the process
  constexpr int kDevs = 64;
  static std::atomic<int> resident[kDevs];  // CTAs resident on the device, 0 = not yet known
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int grid = dev < kDevs ? resident[dev].load(std::memory_order_acquire) : 0;
  if (grid == 0) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::BYTES);
    if (e == cudaSuccess)  // all of the unified L1/shared capacity as shared memory: more heads per SM
      e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    int per_sm = 0, sms = 0;
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kMmaThreads, L::BYTES);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    grid = per_sm * sms;
    if (grid < 1) return cudaErrorInvalidConfiguration;
    if (dev < kDevs) resident[dev].store(grid, std::memory_order_release);
  }
  if (a.count <= 0) return cudaSuccess;
  kern<<<a.count < grid ? a.count : grid, kMmaThreads, L::BYTES, s>>>(a);
  return cudaGetLastError();
}

template <typename TF, int VAR, int DV>
static cudaError_t launch_mma_c(const DecodeArgs &a, int cols_max, cudaStream_t s) {
  if (cols_max <= 16) return launch_mma_t<TF, VAR, DV, 16>(a, s);
  if (cols_max <= 32) return launch_mma_t<TF, VAR, DV, 32>(a, s);
  if (cols_max <= 48) return launch_mma_t<TF, VAR, DV, 48>(a, s);
  return launch_mma_t<TF, VAR, DV, 64>(a, s);
}

template <typename TF, int VAR>
static cudaError_t launch_mma_d(const DecodeArgs &a, int cols_max, cudaStream_t s) {
  if (a.sv.d_v == 64) return launch_mma_c<TF, VAR, 64>(a, cols_max, s);
  return launch_mma_c<TF, VAR, 128>(a, cols_max, s);
}

template <typename TF>
static cudaError_t launch_mma_v(const DecodeArgs &a, int cols_max, cudaStream_t s) {
  switch (a.sv.variant) {
    case SEED_GDN: return launch_mma_d<TF, SEED_GDN>(a, cols_max, s);
    case SEED_KDA: return launch_mma_d<TF, SEED_KDA>(a, cols_max, s);
    default: return launch_mma_d<TF, SEED_MAMBA2>(a, cols_max, s);
  }
}

cudaError_t launch_decode_mma(const DecodeArgs &a, int factor_dtype, int cols_max, cudaStream_t s) {
  if (factor_dtype == SEED_F16) return launch_mma_v<__half>(a, cols_max, s);
  return launch_mma_v<__nv_bfloat16>(a, cols_max, s);
}

}  // namespace seedk
