// fused_gemm.cuh — the warp-specialised tcgen05 GEMM with the row
// normalization fused in, for sm_103a.
//
// One kernel template covers every form of the path:
//   * plain GEMM (identity epilogue);
//   * Lazy Pre-RMSNorm: C = rmsnorm(A) @ B computed as (A @ B) * rstd(A).  The
//     sum of squares of each A row is taken from the A tiles already staged in
//     shared memory by a dedicated norm warpgroup while the tensor cores run,
//     and rstd scales the fp32 accumulator in the epilogue ([FNF-ru] "Lazy
//     Pre-Norm"; [FNF-es] "Lazy Pre-Norm: el truco matemático");
//   * epilogue post-norm, C = norm(A @ B) * gamma + beta, LayerNorm or RMSNorm.
//     When a row is wider than one CTA tile, the CTAs of a cluster split it
//     along N, push per-row partial statistics (count is implicit, mean and
//     M2 for LayerNorm, sum of squares for RMSNorm) to every peer through
//     distributed shared memory, combine them in rank order and normalise
//     their own slice ([FNF-ru] "Multi-CTA Norm Fusion": the norm splits into
//     a row reduction and an element-wise step, and only the reduction needs
//     the whole row, one scalar per row to exchange);
//   * both at once: norm(rmsnorm(A) @ B).
//
// Warp roles (one CTA per SM, persistent over tiles):
//   warp 0      TMA producer: A [128 x BK] and B [BK x BN_CTA] tiles into an
//               S-stage shared-memory ring (128-byte swizzle).
//   warp 1      TMEM allocator and MMA issuer: tcgen05.mma kind::f16, M = 128,
//               N = BN_SUB, K = 16, accumulators in tensor memory, double
//               buffered when a tile needs at most half of it.
//   warps 2-5   epilogue: tcgen05.ld of the accumulator in register subtiles
//               of 32 or 64 columns, statistics, normalise / scale, bf16,
//               swizzled shared-memory staging and TMA stores.
//   warps 6-9   (Lazy Pre-Norm only) sum of squares of the staged A rows.
// A stage is released when the MMA commit and (for Lazy Pre-Norm) the four
// norm warps have all arrived on its "empty" barrier.
#pragma once

#include "ptx.cuh"

namespace fnorm {

enum : int {
  MODE_PRE = 1,       // lazy pre-RMSNorm of A (sum of squares + epilogue scale)
  MODE_POST = 2,      // post-norm of the accumulator rows
  MODE_LN = 4,        // post-norm is LayerNorm (else RMSNorm)
  MODE_CLUSTER = 8,   // rows split over a cluster of up to 8 CTAs along N
  MODE_CL16 = 16,     // ... of up to 16 CTAs (non-portable cluster size)
};

struct FusedParams {
  int M, N, K;
  int cluster;  // CTAs per cluster along N (1 without MODE_CLUSTER)
  float eps, pre_eps;
  const __nv_bfloat16* gamma;
  const __nv_bfloat16* beta;
  float* mean_out;
  float* rstd_out;
  float* pre_rstd_out;
  uint32_t* status;
  unsigned long long wait_limit_ns;
};

__host__ __device__ constexpr int pow2_at_least(int x, int lo) {
  int p = lo;
  while (p < x) p <<= 1;
  return p;
}

template <int STAGES_, int BN_CTA, int CLMAX>
struct Aux {
  uint64_t full[STAGES_];
  uint64_t empty[STAGES_];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t ss_full[2];
  uint64_t ss_empty[2];
  uint64_t xbar[2];
  uint64_t teardown;
  uint32_t tmem_base;
  int abort_flag;
  float ss[2][128];
  float gam[BN_CTA];
  float bet[BN_CTA];
  float2 xstat[2][CLMAX > 0 ? CLMAX : 1][128];
};

constexpr uint32_t kSmemLimit = 232448;  // 227 KB of opt-in shared memory per CTA
constexpr int kMaxStages = 8;

template <int BN_SUB_, int NSUB_, int BK_, int MODE_>
struct KCfg {
  static constexpr int BN_SUB = BN_SUB_, NSUB = NSUB_, BK = BK_, MODE = MODE_;
  static constexpr bool PRE = (MODE & MODE_PRE) != 0;
  static constexpr bool POST = (MODE & MODE_POST) != 0;
  static constexpr bool LN = (MODE & MODE_LN) != 0;
  static constexpr bool CLUSTER = (MODE & (MODE_CLUSTER | MODE_CL16)) != 0;
  static constexpr int CLMAX = (MODE & MODE_CL16) ? 16 : (CLUSTER ? 8 : 0);
  static constexpr int BM = 128;
  static constexpr int BN_CTA = BN_SUB * NSUB;
  static constexpr int NBUF = (NSUB == 1) ? 2 : 1;  // accumulator buffers in TMEM
  static constexpr int TMEM_COLS = pow2_at_least(NBUF * BN_CTA, 32);
  static constexpr uint32_t A_BYTES = BM * BK * 2;
  static constexpr uint32_t B_BYTES = BK * BN_CTA * 2;
  static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr uint32_t STG_BYTES = 4 * 2 * 4096;  // 4 epilogue warps x 2 buffers x [32 x 64] bf16
  static constexpr uint32_t AUX_BYTES = (sizeof(Aux<kMaxStages, BN_CTA, CLMAX>) + 15) / 16 * 16;
  static constexpr int STAGES_FIT = (int)((kSmemLimit - 1024 - STG_BYTES - AUX_BYTES) / STAGE_BYTES);
  static constexpr int STAGES = STAGES_FIT < kMaxStages ? STAGES_FIT : kMaxStages;
  static constexpr uint32_t SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + STG_BYTES + AUX_BYTES;
  static constexpr int NUM_THREADS = 32 * (2 + 4 + (PRE ? 4 : 0));
  static constexpr uint32_t SW_A = (BK == 64) ? kSwizzle128B : kSwizzle64B;
  static constexpr uint32_t IDESC = make_idesc_bf16_f32(BM, BN_SUB, true);

  static_assert(BK == 64 || BK == 32, "BK must be 64 (128B swizzle) or 32 (64B swizzle)");
  static_assert(BN_SUB % 64 == 0 && BN_SUB >= 64 && BN_SUB <= 256, "UMMA N in 64..256, step 64");
  static_assert(NSUB == 1 || NSUB == 2, "one or two accumulator subtiles per tile");
  static_assert(NBUF * BN_CTA <= 512, "tensor memory holds 512 fp32 columns");
  static_assert(STAGES >= 2, "shared memory too small for a 2-stage ring");
  static_assert(!(PRE && !POST) || !CLUSTER, "Lazy Pre-Norm alone never needs a cluster");
};

// ---------------------------------------------------------------------------
template <class Cfg>
__global__ void __launch_bounds__(Cfg::NUM_THREADS, 1)
    fused_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmC, const FusedParams p) {
  constexpr int BK = Cfg::BK, BN_SUB = Cfg::BN_SUB, NSUB = Cfg::NSUB, BN_CTA = Cfg::BN_CTA;
  constexpr int STAGES = Cfg::STAGES, NBUF = Cfg::NBUF;
  constexpr bool PRE = Cfg::PRE, POST = Cfg::POST, LN = Cfg::LN, CLUSTER = Cfg::CLUSTER;
  constexpr uint32_t A_BYTES = Cfg::A_BYTES, STAGE_BYTES = Cfg::STAGE_BYTES;
  using AuxT = Aux<STAGES, BN_CTA, Cfg::CLMAX>;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;  // swizzle atoms need 1024-byte alignment
  uint8_t* smem = smem_raw + (base - raw_addr);
  const uint32_t stg_base = base + STAGES * STAGE_BYTES;
  AuxT* aux = reinterpret_cast<AuxT*>(smem + STAGES * STAGE_BYTES + Cfg::STG_BYTES);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int M = p.M, N = p.N, K = p.K;
  const int C = CLUSTER ? p.cluster : 1;
  const int rank = CLUSTER ? static_cast<int>(cluster_ctarank()) : 0;
  const int num_m = (M + Cfg::BM - 1) / Cfg::BM;
  const int group_cols = BN_CTA * C;
  const int ngroups = (N + group_cols - 1) / group_cols;
  const int total = num_m * ngroups;
  const int cid = static_cast<int>(blockIdx.x) / C;
  const int ncl = static_cast<int>(gridDim.x) / C;
  const int num_kb = (K + BK - 1) / BK;

  const WaitCtx wc{p.wait_limit_ns, p.status, &aux->abort_flag};

  // ---------------- set-up ----------------
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&aux->full[s]), 1);
      mbar_init(smem_u32(&aux->empty[s]), 1 + (PRE ? 4 : 0));
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&aux->acc_full[b]), 1);
      mbar_init(smem_u32(&aux->acc_empty[b]), 4);
      mbar_init(smem_u32(&aux->ss_full[b]), 128);
      mbar_init(smem_u32(&aux->ss_empty[b]), 128);
      mbar_init(smem_u32(&aux->xbar[b]), 1);
    }
    mbar_init(smem_u32(&aux->teardown), 1);
    aux->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmC);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&aux->tmem_base), Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  if (POST && warp >= 2 && warp < 6) {
    // post-norm CTAs own a fixed column slice: the whole row fits the cluster
    const int n0 = rank * BN_CTA;
    for (int j = static_cast<int>(threadIdx.x) - 64; j < BN_CTA; j += 128) {
      const int n = n0 + j;
      aux->gam[j] = (p.gamma != nullptr && n < N) ? __bfloat162float(p.gamma[n]) : 1.0f;
      aux->bet[j] = (p.beta != nullptr && n < N) ? __bfloat162float(p.beta[n]) : 0.0f;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (CLUSTER) cluster_sync();  // peers' barriers are initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem_base = aux->tmem_base;

  if (warp == 0) {
    // ======================= TMA producer =======================
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, filled = 0, fill_par = 0;
      bool ok = true;
      for (int t = cid; t < total && ok; t += ncl) {
        const int m0 = (t / ngroups) * Cfg::BM;
        const int n0 = ((t % ngroups) * C + rank) * BN_CTA;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(wc, smem_u32(&aux->empty[stage]), phase ^ 1u, kSiteProducer)) {
            ok = false;
            break;
          }
          const uint32_t full = smem_u32(&aux->full[stage]);
          mbar_arrive_expect_tx(full, STAGE_BYTES);
          const uint32_t sa = base + stage * STAGE_BYTES;
          tma_load_2d(sa, &tmA, kb * BK, m0, full);
          const uint32_t sb = sa + A_BYTES;
#pragma unroll
          for (int c = 0; c < BN_CTA / 64; ++c) tma_load_2d(sb + c * (BK * 128), &tmB, n0 + c * 64, kb * BK, full);
          filled |= 1u << stage;
          fill_par = (fill_par & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // teardown drain: every copy issued into shared memory lands before exit
      for (int s = 0; s < STAGES; ++s)
        if ((filled >> s) & 1u)
          mbar_wait<false, true>(wc, smem_u32(&aux->full[s]), (fill_par >> s) & 1u, kSiteTeardown);
    }
  } else if (warp == 1) {
    // ======================= MMA issuer =======================
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      int it = 0;
      bool ok = true;
      for (int t = cid; t < total && ok; t += ncl, ++it) {
        const int buf = (NBUF == 2) ? (it & 1) : 0;
        const uint32_t aph = static_cast<uint32_t>((NBUF == 2) ? (it >> 1) : it) & 1u;
        if (!mbar_wait(wc, smem_u32(&aux->acc_empty[buf]), aph ^ 1u, kSiteMma)) break;
        tc_fence_after();
        const uint32_t d0 = tmem_base + static_cast<uint32_t>(buf * BN_CTA);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(wc, smem_u32(&aux->full[stage]), phase, kSiteMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = base + stage * STAGE_BYTES;
          const uint32_t sb = sa + A_BYTES;
#pragma unroll
          for (int ks = 0; ks < BK / 16; ++ks) {
            // A: K-major, rows of BK*2 bytes, 8-row groups BK*16 bytes apart;
            // a K step of 16 elements is 32 bytes inside the swizzle row.
            const uint64_t da = make_smem_desc(sa + ks * 32, 16, 8 * BK * 2, Cfg::SW_A);
#pragma unroll
            for (int sub = 0; sub < NSUB; ++sub) {
              // B: MN-major, 64-column chunks of BK rows x 128 bytes;
              // LBO = chunk stride along N, SBO = 8-row group stride along K;
              // a K step of 16 rows is 2048 bytes.
              const uint64_t db = make_smem_desc(sb + sub * (BN_SUB / 64) * (BK * 128) + ks * (16 * 128),
                                                 BK * 128, 1024, kSwizzle128B);
              umma_bf16(d0 + sub * BN_SUB, da, db, Cfg::IDESC, (kb | ks) != 0 ? 1u : 0u);
            }
          }
          umma_commit(smem_u32(&aux->empty[stage]));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) umma_commit(smem_u32(&aux->acc_full[buf]));
      }
      // every MMA issued has completed before tensor memory is released
      umma_commit(smem_u32(&aux->teardown));
      mbar_wait<false, true>(wc, smem_u32(&aux->teardown), 0, kSiteTeardown);
    }
  } else if (warp < 6) {
    // ======================= epilogue =======================
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;
    const uint32_t stg = stg_base + static_cast<uint32_t>(warp - 2) * 8192u;
    uint32_t sbuf = 0;
    int it = 0;
    for (int t = cid; t < total; t += ncl, ++it) {
      const int m0 = (t / ngroups) * Cfg::BM;
      const int g = t % ngroups;
      const int n0 = (g * C + rank) * BN_CTA;
      const int buf = (NBUF == 2) ? (it & 1) : 0;
      const uint32_t aph = static_cast<uint32_t>((NBUF == 2) ? (it >> 1) : it) & 1u;
      if (!mbar_wait_warp(wc, smem_u32(&aux->acc_full[buf]), aph, kSiteEpilogue)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(buf * BN_CTA);

      // ---- lazy pre-norm scale: rstd of the A row ----
      float pre = 1.0f;
      if (PRE) {
        const int sb = it & 1;
        if (!mbar_wait_warp(wc, smem_u32(&aux->ss_full[sb]), static_cast<uint32_t>(it >> 1) & 1u, kSiteEpilogue))
          break;
        const float ss = aux->ss[sb][row];
        mbar_arrive(smem_u32(&aux->ss_empty[sb]));
        pre = rsqrtf(ss / static_cast<float>(K) + p.pre_eps);
      }

      // ---- post-norm statistics ----
      float mean = 0.0f, rstd = 1.0f;
      if (POST) {
        const int nvalid = min(max(N - n0, 0), BN_CTA);
        float part0 = 0.0f, part1 = 0.0f;  // LN: (mean, M2) of the slice; RMS: (sum x^2, 0)
        {
          float s[4] = {0.f, 0.f, 0.f, 0.f};
          for (int c = 0; c < BN_CTA / 32; ++c) {
            if (c * 32 >= nvalid) break;
            uint32_t r[32];
            tmem_ld_32x32b_x32(tb + c * 32, r);
            tmem_ld_wait();
            reg_fence(r);
            const int lim = nvalid - c * 32;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float v = __uint_as_float(r[j]) * pre;
              const float add = LN ? v : v * v;
              s[j & 3] += (j < lim) ? add : 0.0f;
            }
          }
          const float tot = (s[0] + s[1]) + (s[2] + s[3]);
          if (LN) {
            const float m_loc = nvalid > 0 ? tot / static_cast<float>(nvalid) : 0.0f;
            float d2[4] = {0.f, 0.f, 0.f, 0.f};
            for (int c = 0; c < BN_CTA / 32; ++c) {
              if (c * 32 >= nvalid) break;
              uint32_t r[32];
              tmem_ld_32x32b_x32(tb + c * 32, r);
              tmem_ld_wait();
              reg_fence(r);
              const int lim = nvalid - c * 32;
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                const float d = __uint_as_float(r[j]) * pre - m_loc;
                d2[j & 3] += (j < lim) ? d * d : 0.0f;
              }
            }
            part0 = m_loc;
            part1 = (d2[0] + d2[1]) + (d2[2] + d2[3]);
          } else {
            part0 = tot;
          }
        }
        if (CLUSTER) {
          // push (part0, part1) for this row to every CTA of the cluster
          const int xp = it & 1;
          const uint32_t xb = smem_u32(&aux->xbar[xp]);
          if (threadIdx.x == 64) mbar_arrive_expect_tx(xb, static_cast<uint32_t>(C) * 128u * 8u);
          const uint32_t mine = smem_u32(&aux->xstat[xp][rank][row]);
          for (int r2 = 0; r2 < C; ++r2)
            st_async_f32x2(mapa_shared(mine, r2), part0, part1, mapa_shared(xb, r2));
          if (!mbar_wait_warp<true>(wc, xb, static_cast<uint32_t>(it >> 1) & 1u, kSiteExchange)) break;
          // combine the slices in rank order (identical on every CTA)
          float n_acc = 0.0f, m_acc = 0.0f, q_acc = 0.0f;
          for (int r2 = 0; r2 < C; ++r2) {
            const float2 v = aux->xstat[xp][r2][row];
            const int nq = min(max(N - (g * C + r2) * BN_CTA, 0), BN_CTA);
            if (LN) {
              if (nq > 0) {
                const float nqf = static_cast<float>(nq);
                const float nn = n_acc + nqf;
                const float d = v.x - m_acc;
                m_acc += d * (nqf / nn);
                q_acc += v.y + d * d * (n_acc * nqf / nn);
                n_acc = nn;
              }
            } else {
              q_acc += v.x;
            }
          }
          part0 = LN ? m_acc : q_acc;
          part1 = q_acc;
        }
        if (LN) {
          mean = part0;
          rstd = rsqrtf(part1 / static_cast<float>(N) + p.eps);
        } else {
          rstd = rsqrtf(part0 / static_cast<float>(N) + p.eps);
        }
      }

      // ---- normalise / scale, bf16, stage, TMA store: 64 columns at a time ----
      for (int c = 0; c < BN_CTA / 64; ++c) {
        const int col0 = n0 + c * 64;
        if (col0 >= N) break;
        uint32_t r0[32], r1[32];
        tmem_ld_32x32b_x32(tb + c * 64, r0);
        tmem_ld_32x32b_x32(tb + c * 64 + 32, r1);
        tmem_ld_wait();
        reg_fence(r0);
        reg_fence(r1);
        uint32_t w[32];
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          float y0 = __uint_as_float(r0[j]) * pre, y1 = __uint_as_float(r0[j + 1]) * pre;
          if (POST) {
            const int cj = c * 64 + j;
            y0 = (LN ? (y0 - mean) : y0) * rstd * aux->gam[cj] + aux->bet[cj];
            y1 = (LN ? (y1 - mean) : y1) * rstd * aux->gam[cj + 1] + aux->bet[cj + 1];
          }
          w[j >> 1] = pack_bf16x2(y0, y1);
        }
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          float y0 = __uint_as_float(r1[j]) * pre, y1 = __uint_as_float(r1[j + 1]) * pre;
          if (POST) {
            const int cj = c * 64 + 32 + j;
            y0 = (LN ? (y0 - mean) : y0) * rstd * aux->gam[cj] + aux->bet[cj];
            y1 = (LN ? (y1 - mean) : y1) * rstd * aux->gam[cj + 1] + aux->bet[cj + 1];
          }
          w[16 + (j >> 1)] = pack_bf16x2(y0, y1);
        }
        const uint32_t sbase = stg + sbuf * 4096u;
        if (lane == 0) bulk_wait_read<1>();  // the store that used this buffer has read it
        __syncwarp();
        // row `lane` of a [32 x 64] bf16 box, 128-byte swizzle: 16-byte chunk
        // ch of the row sits at chunk (ch ^ (row & 7))
        const uint32_t rbase = sbase + static_cast<uint32_t>(lane) * 128u;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          const uint32_t a = rbase + (static_cast<uint32_t>(ch ^ (lane & 7)) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(w[4 * ch]), "r"(w[4 * ch + 1]),
                       "r"(w[4 * ch + 2]), "r"(w[4 * ch + 3])
                       : "memory");
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (m0 + q * 32 < M) tma_store_2d(&tmC, sbase, col0, m0 + q * 32);
          bulk_commit();
        }
        sbuf ^= 1u;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&aux->acc_empty[buf]));

      // ---- row statistics ----
      const int m = m0 + row;
      if (m < M) {
        if (POST) {
          if (rank == 0) {
            if (LN && p.mean_out != nullptr) p.mean_out[m] = mean;
            if (p.rstd_out != nullptr) p.rstd_out[m] = rstd;
            if (PRE && p.pre_rstd_out != nullptr) p.pre_rstd_out[m] = pre;
          }
        } else if (PRE) {
          if (g == 0 && p.rstd_out != nullptr) p.rstd_out[m] = pre;
        }
      }
    }
    if (lane == 0) bulk_wait<0>();
  } else {
    // ======================= norm warps (Lazy Pre-Norm) =======================
    if (PRE) {
      const int row = (warp - 6) * 32 + lane;
      constexpr int ROW_BYTES = BK * 2;
      constexpr int CHUNKS = ROW_BYTES / 16;
      // swizzle phase of this row: chunk index XOR (row address bits 7..)
      const int swz = ((row * ROW_BYTES) >> 7) & (CHUNKS - 1);
      uint32_t stage = 0, phase = 0;
      int it = 0;
      for (int t = cid; t < total; t += ncl, ++it) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        bool ok = true;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait_warp(wc, smem_u32(&aux->full[stage]), phase, kSiteNorm)) {
            ok = false;
            break;
          }
          const uint8_t* arow = smem + stage * STAGE_BYTES + row * ROW_BYTES;
#pragma unroll
          for (int ch = 0; ch < CHUNKS; ++ch) {
            // visit the row's physical chunks in a bank-conflict-free order;
            // the sum does not depend on the order
            const uint4 v = *reinterpret_cast<const uint4*>(arow + ((ch ^ swz) << 4));
            float x;
            x = bf16_lo(v.x); acc[0] = fmaf(x, x, acc[0]);
            x = bf16_hi(v.x); acc[1] = fmaf(x, x, acc[1]);
            x = bf16_lo(v.y); acc[2] = fmaf(x, x, acc[2]);
            x = bf16_hi(v.y); acc[3] = fmaf(x, x, acc[3]);
            x = bf16_lo(v.z); acc[0] = fmaf(x, x, acc[0]);
            x = bf16_hi(v.z); acc[1] = fmaf(x, x, acc[1]);
            x = bf16_lo(v.w); acc[2] = fmaf(x, x, acc[2]);
            x = bf16_hi(v.w); acc[3] = fmaf(x, x, acc[3]);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&aux->empty[stage]));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        const int sb = it & 1;
        if (!mbar_wait_warp(wc, smem_u32(&aux->ss_empty[sb]), (static_cast<uint32_t>(it >> 1) & 1u) ^ 1u, kSiteNorm))
          break;
        aux->ss[sb][row] = (acc[0] + acc[1]) + (acc[2] + acc[3]);
        mbar_arrive(smem_u32(&aux->ss_full[sb]));
      }
    }
  }

  // ---------------- teardown ----------------
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
  }
  if (CLUSTER) cluster_sync();  // no CTA leaves while a peer may still address it
}

}  // namespace fnorm
