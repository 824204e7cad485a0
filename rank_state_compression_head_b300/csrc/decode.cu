// Fused read-out + exact factored update (one decode step of every head).
//
// "Shallow Encoding Emits Deep Memories", picx.dev summary, Methodology >
// Exact Update (Lemma 2): the sink + low-rank form is closed under the Gated
// DeltaNet, Kimi Delta Attention and Mamba-2 updates; each step appends
// columns to the factors.  thelatestinai.com list view, Table 1 (decode
// column): every step reads out and updates each recurrent state.
//
// This file holds the CUDA-core version, used for fp32 factors; bf16 factors
// use the tensor-core version in decode_mma.cu.  Persistent, warp-specialised kernel.  Each CTA walks the heads
// blockIdx.x, blockIdx.x + gridDim.x, ...  A producer warp streams each
// head's m stored columns of U and W (contiguous blocks) and its small
// vectors (q, k, v, a, the sink direction, the column scales) into a
// two-stage shared-memory ring with bulk copies on the TMA engine, counted
// on an mbarrier per stage; eight consumer warps compute
//     x_k = U_eff^T k  and  x_q = U_eff^T q           (one pass over U)
//     W x_k and W x_q                                   (one pass over W)
// and write the appended column(s), the sink coefficient, the scales and
// the read-out, then hand the stage back.  So the next heads' factor blocks
// are in flight while one is being computed.  Existing columns are never
// rewritten: the gate of existing columns lives in fp32 scales, so each
// stored bf16 column is rounded exactly once.
#include "common.cuh"

#include <atomic>

namespace seedk {

constexpr int kConsumerWarps = 8;
constexpr int kStages = 2;

// Byte layout of one pipeline stage.
template <int VAR, typename TF, int DV, int MAXC>
struct Stage {
  static constexpr int DK = kDK;
  static constexpr int ESZ = (int)sizeof(TF);
  static constexpr bool KDA = VAR == SEED_KDA;
  static constexpr int U_OFF = 0;
  static constexpr int W_OFF = U_OFF + MAXC * DK * ESZ;
  static constexpr int Q_OFF = W_OFF + MAXC * DV * ESZ;
  static constexpr int K_OFF = Q_OFF + DK * 4;
  static constexpr int A_OFF = K_OFF + DK * 4;
  static constexpr int V_OFF = A_OFF + DK * 4;
  static constexpr int VB_OFF = V_OFF + DV * 4;
  static constexpr int SC_OFF = VB_OFF + DV * 4;                 // column scales [MAXC], or D [DK] (KDA)
  static constexpr int AL_OFF = SC_OFF + (KDA ? DK : MAXC) * 4;  // KDA: alpha [DK]
  static constexpr int BYTES = AL_OFF + (KDA ? DK * 4 : 0);
  static_assert(W_OFF % 16 == 0 && Q_OFF % 16 == 0 && SC_OFF % 16 == 0 && BYTES % 16 == 0,
                "16-byte copies");
};

template <int VAR, typename TF, int DV, int MAXC>
struct DecodeSmem {
  using S = Stage<VAR, TF, DV, MAXC>;
  static constexpr int NX = VAR == SEED_MAMBA2 ? 1 : 2;
  static constexpr int RED_OFF = kStages * S::BYTES;                            // [2][NW][NX][DV] f32
  static constexpr int SCAL_OFF = RED_OFF + 2 * kConsumerWarps * NX * DV * 4;  // [2][NW][8] f32
  static constexpr int XW_OFF = SCAL_OFF + 2 * kConsumerWarps * 8 * 4;         // [NW][4][2] f32
  static constexpr int BAR_OFF = XW_OFF + kConsumerWarps * 8 * 4;              // full[NS], empty[NS]
  static constexpr int BYTES = BAR_OFF + 2 * kStages * 8;
};

template <int VAR, typename TF, int DV, int MAXC>
__global__ void __launch_bounds__((kConsumerWarps + 1) * 32, 1)
decode_kernel(const DecodeArgs p) {
  constexpr int DK = kDK;
  constexpr int NW = kConsumerWarps;
  constexpr int NT = NW * 32;  // consumer threads
  constexpr int NS = kStages;
  using S = Stage<VAR, TF, DV, MAXC>;
  using L = DecodeSmem<VAR, TF, DV, MAXC>;
  constexpr int NX = L::NX;
  constexpr bool KDA = VAR == SEED_KDA;
  constexpr bool M2 = VAR == SEED_MAMBA2;
  constexpr int EPL = Elem<TF>::kPer16B;  // elements in one 16-byte chunk
  constexpr int LPC_U = DK / EPL;         // lanes covering one U column
  constexpr int CPL_U = 32 / LPC_U;       // U columns per warp-wide load
  constexpr int LPC_W = DV / EPL;
  constexpr int CPL_W = 32 / LPC_W;
  constexpr int GU = CPL_U > CPL_W ? CPL_U : CPL_W;  // columns per work unit (one warp)
  constexpr int NUNITS = (MAXC + GU - 1) / GU;
  constexpr int UPW = (NUNITS + NW - 1) / NW;        // units per warp
  static_assert(GU <= 4, "unit staging buffer holds 4 columns");
  static_assert(NT >= DK && NT >= DV, "one thread per state row / column");

  extern __shared__ __align__(128) unsigned char smem[];
  float *red = reinterpret_cast<float *>(smem + L::RED_OFF);
  float *scal = reinterpret_cast<float *>(smem + L::SCAL_OFF);
  float *xw = reinterpret_cast<float *>(smem + L::XW_OFF);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::BAR_OFF);
  uint64_t *empty = full + NS;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const StateView &sv = p.sv;
  const int G = gridDim.x;
  const int first = blockIdx.x;
  const int nmine = first < sv.n_heads ? (sv.n_heads - first + G - 1) / G : 0;
  const int growth = sv.growth;

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NW);
    }
    fence_mbar_init();
  }
  __syncthreads();

  // ---------------------------------------------------------------- producer
  if (warp == NW) {
    if (lane == 0) {
      for (int i = 0; i < nmine; ++i) {
        const int s = i % NS;
        const uint32_t use = (uint32_t)(i / NS);
        if (!mbar_wait(&empty[s], (use & 1u) ^ 1u)) break;  // consumers stopped
        const int h = first + i * G;
        const int r_h = sv.rank_of(h);
        const int m = r_h + growth * sv.steps;
        if (r_h < 0 || m > MAXC) {  // bad rank table: complete the stage empty
          mbar_arrive_expect_tx(&full[s], 0);
          continue;
        }
        const int64_t c0 = sv.col0(h);
        const int dir = sv.dir_of(h);
        unsigned char *st = smem + s * S::BYTES;
        const bool sc_stage = !KDA && scales_in_stage(c0, r_h + growth * sv.T);
        const int sc_bytes = KDA ? DK * 4 : (sc_stage ? ((m + 3) & ~3) * 4 : 0);
        const uint32_t bytes = (uint32_t)(m * DK * S::ESZ + m * DV * S::ESZ + 3 * DK * 4 + 2 * DV * 4 +
                                          sc_bytes + (KDA ? DK * 4 : 0));
        mbar_arrive_expect_tx(&full[s], bytes);
        if (m > 0) {
          bulk_g2s(st + S::U_OFF, reinterpret_cast<const TF *>(sv.U) + c0 * DK, m * DK * S::ESZ, &full[s]);
          bulk_g2s(st + S::W_OFF, reinterpret_cast<const TF *>(sv.W) + c0 * DV, m * DV * S::ESZ, &full[s]);
        }
        bulk_g2s(st + S::Q_OFF, p.q + (int64_t)h * DK, DK * 4, &full[s]);
        bulk_g2s(st + S::K_OFF, p.k + (int64_t)h * DK, DK * 4, &full[s]);
        bulk_g2s(st + S::A_OFF, sv.a + (int64_t)h * DK, DK * 4, &full[s]);
        bulk_g2s(st + S::V_OFF, p.v + (int64_t)h * DV, DV * 4, &full[s]);
        bulk_g2s(st + S::VB_OFF, sv.vbar + (int64_t)dir * DV, DV * 4, &full[s]);
        if (KDA) {
          bulk_g2s(st + S::SC_OFF, sv.scale + (int64_t)h * DK, DK * 4, &full[s]);
          bulk_g2s(st + S::AL_OFF, p.gate + (int64_t)h * DK, DK * 4, &full[s]);
        } else if (sc_bytes) {
          bulk_g2s(st + S::SC_OFF, sv.scale + c0, sc_bytes, &full[s]);
        }
      }
    }
    return;
  }

  // --------------------------------------------------------------- consumers
  for (int i = 0; i < nmine; ++i) {
    const int s = i % NS;
    const uint32_t use = (uint32_t)(i / NS);
    const int buf = i & 1;
    const int h = first + i * G;
    const int r_h = sv.rank_of(h);
    const int m = r_h + growth * sv.steps;
    const bool bad_rank = r_h < 0 || m > MAXC;
    const int64_t c0 = bad_rank ? 0 : sv.col0(h);
    const int dir = sv.dir_of(h);
    // gates: issued early, used at the end
    float g = 0.f, beta = 0.f, dt = 0.f;
    if (VAR == SEED_GDN) { g = p.gate[h]; beta = p.beta[h]; }
    if (KDA) beta = p.beta[h];
    if (M2) { dt = p.gate[h]; g = expf(dt * p.A[dir]); }
    const bool sc_stage = !KDA && scales_in_stage(c0, r_h + growth * sv.T);

    const bool arrived = mbar_wait(&full[s], use & 1u);
    const unsigned char *st = smem + s * S::BYTES;
    const TF *Us = reinterpret_cast<const TF *>(st + S::U_OFF);
    const TF *Ws = reinterpret_cast<const TF *>(st + S::W_OFF);
    const float *qs = reinterpret_cast<const float *>(st + S::Q_OFF);
    const float *ks = reinterpret_cast<const float *>(st + S::K_OFF);
    const float *as = reinterpret_cast<const float *>(st + S::A_OFF);
    const float *vs = reinterpret_cast<const float *>(st + S::V_OFF);
    const float *vbs = reinterpret_cast<const float *>(st + S::VB_OFF);
    const float *scs = (KDA || sc_stage) ? reinterpret_cast<const float *>(st + S::SC_OFF) : sv.scale + c0;
    const float *als = reinterpret_cast<const float *>(st + S::AL_OFF);
    if (tid == 0 && sv.status) sv.status[h] = bad_rank ? SEED_ERR_INVALID_ARG : SEED_OK;

    float S_loc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) S_loc[j] = 0.f;
    float kt = 0.f, qt = 0.f, at = 0.f, vt = 0.f, vbt = 0.f, alt = 0.f, Dt = 0.f;
    float unew0 = 0.f, unew1 = 0.f;

    if (arrived && !bad_rank) {
      // ---- row slices of k and q for the U pass -----------------------------
      const int r0 = (lane % LPC_U) * EPL;
      float kx[EPL], qx[EPL];
#pragma unroll
      for (int e = 0; e < EPL; e += 4) {
        const float4 q4 = *reinterpret_cast<const float4 *>(qs + r0 + e);
        const float4 k4 = *reinterpret_cast<const float4 *>(ks + r0 + e);
        qx[e] = q4.x; qx[e + 1] = q4.y; qx[e + 2] = q4.z; qx[e + 3] = q4.w;
        kx[e] = k4.x; kx[e + 1] = k4.y; kx[e + 2] = k4.z; kx[e + 3] = k4.w;
      }
      if (KDA) {  // x_k = U^T (D k), x_q = U^T (D' q) with D' = alpha D
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
          const float d = scs[r0 + e];
          kx[e] *= d;
          qx[e] *= als[r0 + e] * d;
        }
      }

      // ---- U and W passes, one work unit (GU columns) at a time ---------------
      float acc[NX][EPL];
#pragma unroll
      for (int j = 0; j < NX; ++j)
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[j][e] = 0.f;
      float *xu = xw + warp * 8;
#pragma unroll
      for (int uu = 0; uu < UPW; ++uu) {
        const int cbase = (warp + uu * NW) * GU;
        if (cbase >= m) break;
#pragma unroll
        for (int l = 0; l < GU / CPL_U; ++l) {
          const int cl = l * CPL_U + lane / LPC_U;  // column within the unit
          const int col = cbase + cl;
          float pk = 0.f, pq = 0.f;
          if (col < m) {
            float x[EPL];
            Elem<TF>::unpack(*reinterpret_cast<const uint4 *>(Us + col * DK + r0), x);
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
              if (!M2) pk = fmaf(x[e], kx[e], pk);
              pq = fmaf(x[e], qx[e], pq);
            }
          }
#pragma unroll
          for (int o = LPC_U / 2; o >= 1; o >>= 1) {
            if (!M2) pk += __shfl_xor_sync(0xffffffffu, pk, o);
            pq += __shfl_xor_sync(0xffffffffu, pq, o);
          }
          if ((lane % LPC_U) == 0 && col < m) {
            const float c = KDA ? 1.f : scs[col];
            if (M2) {
              xu[cl * 2] = c * pq;
            } else {
              xu[cl * 2] = c * pk;
              xu[cl * 2 + 1] = c * pq;
            }
          }
        }
        __syncwarp();
#pragma unroll
        for (int l = 0; l < GU / CPL_W; ++l) {
          const int cl = l * CPL_W + lane / LPC_W;
          const int col = cbase + cl;
          if (col < m) {
            float x[EPL];
            Elem<TF>::unpack(*reinterpret_cast<const uint4 *>(Ws + col * DV + (lane % LPC_W) * EPL), x);
#pragma unroll
            for (int j = 0; j < NX; ++j) {
              const float xv = xu[cl * 2 + j];
#pragma unroll
              for (int e = 0; e < EPL; ++e) acc[j][e] = fmaf(x[e], xv, acc[j][e]);
            }
          }
        }
        __syncwarp();
      }
      // the CPL_W column groups of the warp hold partials of the same rows
#pragma unroll
      for (int o = LPC_W; o < 32; o <<= 1)
#pragma unroll
        for (int j = 0; j < NX; ++j)
#pragma unroll
          for (int e = 0; e < EPL; ++e) acc[j][e] += __shfl_xor_sync(0xffffffffu, acc[j][e], o);
      if (lane < LPC_W) {
#pragma unroll
        for (int j = 0; j < NX; ++j)
#pragma unroll
          for (int e = 0; e < EPL; e += 4)
            *reinterpret_cast<float4 *>(red + ((buf * NW + warp) * NX + j) * DV + lane * EPL + e) =
                make_float4(acc[j][e], acc[j][e + 1], acc[j][e + 2], acc[j][e + 3]);
      }

      // ---- block scalars: thread t owns row t (< DK) and value column t (< DV) --
      if (tid < DK) {
        kt = ks[tid]; qt = qs[tid]; at = as[tid];
        if (VAR == SEED_GDN) {
          unew0 = Elem<TF>::round(kt);
          S_loc[0] = kt * at; S_loc[1] = qt * at; S_loc[2] = kt * qt; S_loc[3] = unew0 * qt;
        } else if (KDA) {
          alt = als[tid];
          Dt = scs[tid];
          const float Dn = alt * Dt;
          unew0 = Elem<TF>::round(kt / Dt);
          unew1 = Elem<TF>::round(kt / Dn);
          S_loc[0] = kt * at; S_loc[1] = alt * at * qt; S_loc[2] = alt * kt * qt; S_loc[3] = kt * qt;
          S_loc[6] = unew0 * Dn * qt; S_loc[7] = unew1 * Dn * qt;
        } else {
          unew0 = Elem<TF>::round(dt * kt);
          S_loc[0] = at * qt; S_loc[1] = kt * qt; S_loc[2] = unew0 * qt;
        }
      }
      if (tid < DV) {
        vt = vs[tid]; vbt = vbs[tid];
        S_loc[4] = vt * vbt; S_loc[5] = vbt * vbt;
      }
      if (warp * 32 < (DK > DV ? DK : DV)) {
        const float r = warp_reduce8(S_loc, lane);
        if ((lane & 3) == 0) scal[(buf * NW + warp) * 8 + reduce8_index(lane)] = r;
      }
    }
    // one barrier per head: partial sums visible; a failed wait stops every consumer
    const int timed_out = team_or(1, NT, !arrived);
    if (timed_out) {
      if (tid == 0 && sv.status)
        for (int j = i; j < nmine; ++j) sv.status[first + j * G] = SEED_ERR_TIMEOUT;
      if (tid == 0)  // let copies already issued land before the CTA leaves
        for (int j = i; j < nmine && j < i + NS; ++j) mbar_wait(&full[j % NS], (uint32_t)(j / NS) & 1u);
      break;
    }
    if (bad_rank) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      continue;
    }

    // ---- update and read-out ---------------------------------------------------
    constexpr int NSW = (DK > DV ? DK : DV) / 32;  // warps holding scalar partials
    float Sg[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float a = 0.f;
#pragma unroll
      for (int w = 0; w < NSW; ++w) a += scal[(buf * NW + w) * 8 + j];
      Sg[j] = a;
    }
    const float omega = Sg[4] / Sg[5];
    int bad = 0;
    TF *Uo = reinterpret_cast<TF *>(sv.U) + (c0 + m) * DK;
    TF *Wo = reinterpret_cast<TF *>(sv.W) + (c0 + m) * DV;
    float wx[NX];
#pragma unroll
    for (int j = 0; j < NX; ++j) wx[j] = 0.f;
    if (tid < DV) {
#pragma unroll
      for (int j = 0; j < NX; ++j) {
        float a = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) a += red[((buf * NW + w) * NX + j) * DV + tid];
        wx[j] = a;
      }
    }
    if (VAR == SEED_GDN) {
      // a' = g a + beta (omega - g k.a) k ;  a'.q = g a.q + beta (omega - g k.a) k.q
      const float coef = beta * (omega - g * Sg[0]);
      const float aq = fmaf(g, Sg[1], coef * Sg[2]);
      if (tid < DK) {
        const float an = fmaf(g, at, coef * kt);
        sv.a[(int64_t)h * DK + tid] = an;
        Elem<TF>::store(Uo + tid, kt);
        bad |= !finite(an);
      }
      if (tid < DV) {
        const float eps = fmaf(-omega, vbt, vt);
        const float wn = Elem<TF>::round(beta * fmaf(-g, wx[0], eps));
        Elem<TF>::store(Wo + tid, wn);
        const float o = fmaf(vbt, aq, fmaf(g, wx[NX - 1], Sg[3] * wn));
        p.o[(int64_t)h * DV + tid] = o;
        bad |= !finite(o);
      }
      if (tid < m) sv.scale[c0 + tid] = g * scs[tid];
      if (tid == m) sv.scale[c0 + m] = 1.f;
    } else if (KDA) {
      // a' = alpha (a - beta k (k.a)) + beta omega k ; D' = alpha D
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
        const float w1 = Elem<TF>::round(-beta * wx[0]);
        const float w2 = Elem<TF>::round(beta * eps);
        Elem<TF>::store(Wo + tid, w1);
        Elem<TF>::store(Wo + DV + tid, w2);
        const float o = fmaf(vbt, aq, wx[NX - 1] + w1 * Sg[6] + w2 * Sg[7]);
        p.o[(int64_t)h * DV + tid] = o;
        bad |= !finite(o);
      }
    } else {
      // Mamba-2: a' = g a + dt omega B ; y = xbar (a'.C) + g W x_C + (u_new.C) w_new
      const float coef = dt * omega;
      const float aC = fmaf(g, Sg[0], coef * Sg[1]);
      if (tid < DK) {
        const float an = fmaf(g, at, coef * kt);
        sv.a[(int64_t)h * DK + tid] = an;
        Elem<TF>::store(Uo + tid, unew0);
        bad |= !finite(an);
      }
      if (tid < DV) {
        const float wn = Elem<TF>::round(fmaf(-omega, vbt, vt));
        Elem<TF>::store(Wo + tid, wn);
        const float o = fmaf(vbt, aC, fmaf(g, wx[0], Sg[2] * wn));
        p.o[(int64_t)h * DV + tid] = o;
        bad |= !finite(o);
      }
      if (tid < m) sv.scale[c0 + tid] = g * scs[tid];
      if (tid == m) sv.scale[c0 + m] = 1.f;
    }
    if (bad && sv.status) sv.status[h] = SEED_ERR_NONFINITE;
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);  // this warp is done with the stage
  }
}

template <int VAR, typename TF, int DV, int MAXC>
static cudaError_t launch_decode_t(const DecodeArgs &a, cudaStream_t s) {
  using L = DecodeSmem<VAR, TF, DV, MAXC>;
  auto kern = decode_kernel<VAR, TF, DV, MAXC>;
  // attributes belong to (kernel, device): set them the first time this kernel runs on
  // each device of the process; the SM count is the current device's
  static std::atomic<uint64_t> ready{0};
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (uint64_t)1 << dev : 0;
  if (!bit || !(ready.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::BYTES);
    if (e != cudaSuccess) return e;
    ready.fetch_or(bit, std::memory_order_acq_rel);
  }
  const int per_sm = (227 * 1024) / (L::BYTES + 1024) >= 2 ? 2 : 1;
  int grid = (sms > 0 ? sms : 1) * per_sm;
  if (grid > a.sv.n_heads) grid = a.sv.n_heads;
  kern<<<grid, (kConsumerWarps + 1) * 32, L::BYTES, s>>>(a);
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
  DecodeArgs a{sv, q, k, v, gate, beta, A, o, 0, sv.n_heads};
  if (factor_dtype == SEED_F32) {
    a.sv.order = nullptr;
    return launch_decode_v<float>(a, cols_max, s);
  }
  // 16-bit factors: the two contractions run on the tensor cores (decode_mma.cu);
  // with a class order, one launch per column class, sized for it
  if (!sv.order) return launch_decode_mma(a, factor_dtype, cols_max, s);
  const int cols16 = (cols_max + 15) & ~15;
  for (int c = 0, begin = 0; c < 4; begin = sv.class_end[c], ++c) {
    const int end = sv.class_end[c];
    if (end <= begin) continue;
    a.pos0 = begin;
    a.count = end - begin;
    const int cls_cols = 16 * (c + 1) < cols16 ? 16 * (c + 1) : cols16;
    const cudaError_t e = launch_decode_mma(a, factor_dtype, cls_cols, s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace seedk
