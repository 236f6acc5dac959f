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
//   * epilogue post-norm, C = norm(A @ B) * gamma + beta, LayerNorm or RMSNorm
//     ([FNF-ru] "Multi-CTA Norm Fusion": a norm is a row reduction plus an
//     element-wise step, only the reduction needs the whole row, and its
//     result is one scalar per row).  Four layouts of a row block:
//       - resident, one CTA: the CTA's accumulator spans the whole row;
//       - resident, cluster: the CTAs of a cluster split the row along N, each
//         keeps its slice in tensor memory, pushes its per-row partial
//         statistics to every peer through distributed shared memory, combines
//         them in rank order and normalises its slice;
//       - spill, cluster: each CTA owns S slices of 256 columns, computed one
//         after another in double-buffered tensor memory; each slice is written
//         to C un-normalised while its statistics accumulate, and once the row
//         block's statistics are exchanged the slices are re-read from L2 and
//         normalised in place while the next row block's MMAs run.  Rows of
//         any width, on small clusters, with no workspace;
//       - resident, grid-wide: the plain GEMM's 256-column tiles, each kept in
//         tensor memory until the row block's statistics are known; the tiles
//         of a row block, on any CTAs of the grid, publish their per-row
//         partial statistics to a global workspace and count in on the row
//         block's counter, then each combines all of them in tile order and
//         normalises its tile from tensor memory (a cooperative launch, all
//         CTAs resident at once, of one CTA per SM or of the co-resident
//         2-CTA clusters that share B; the other accumulator buffer keeps the
//         tensor cores busy meanwhile);
//   * both at once: norm(rmsnorm(A) @ B);
//   * residual: norm(A @ B + R), R written into the accumulator before the
//     tile's MMAs accumulate onto it;
//   * pre-norm with the affine folded into B: (norm(A) * gamma + beta) @ B
//     as rstd * (A @ B' - mean * colsum(B')) + beta @ B, the LayerNorm's
//     shifted sums of the A rows taken by the norm warps;
//   * the backward's GEMMs: B^T and A^T operands read straight from their
//     row-major arrays, and the Lazy Pre-RMSNorm's dgrad epilogue
//     y = u + c_m * x;
//   * the post-norm's backward regrouped onto the GEMM that produces its
//     output gradient ([TFN] "fusion regrouping": the consuming layer's
//     data-gradient GEMM): the accumulator holds dC, the epilogue rebuilds
//     the normalised rows from the forward output, takes the row reductions
//     of the norm's backward (exchanged like the forward's statistics), writes
//     dH and the per-32-row column partials of dgamma and dbeta;
//   * the plain and lazy pre-norm GEMMs on a CTA pair (tcgen05 cta_group::2):
//     a 2-CTA cluster computes each [256 x 256] tile, each CTA staging its 128
//     rows of A and 128 of the tile's B columns; the second CTA's copies
//     complete on the first CTA's full barriers, the first CTA issues the
//     MMAs of both, and their commits release the stages (and accumulators)
//     of both.
//
// Warp roles (one CTA per SM, persistent over work units):
//   warp 0      TMA producer: A [128 x 64] and B [64 x BN] tiles into an
//               S-stage shared-memory ring (128-byte swizzle), or A only when
//               all of B is resident in shared memory.
//   warp 1      TMEM allocator and MMA issuer: tcgen05.mma kind::f16, M = 128,
//               N = BN, K = 16, fp32 accumulators in tensor memory, double
//               buffered (CTA pair: M = 256, issued by the first CTA).
//   warps 2-9   epilogue, two warps per TMEM lane quarter: warps 2-5 own the
//               first BN/2 columns of a tile, warps 6-9 the second half.
//               tcgen05.ld of 32-column register subtiles, statistics (the two
//               halves combine theirs through shared memory), normalise /
//               scale, bf16, swizzled shared-memory staging, TMA stores.
//   warps 10-13 Lazy Pre-Norm: sum of squares of the staged A rows (warps
//               10-17 for the pre-LayerNorm, each row's chunks in two parts);
//               spill layout (without Lazy Pre-Norm): the in-place
//               normalisation of finished row blocks, from L2.
// A stage is released when the MMA commit and (for Lazy Pre-Norm) the four
// norm warps have all arrived on its "empty" barrier.
//
// LayerNorm statistics are one pass of shifted sums per column range: with k0
// the row's first value in the range, s1 = sum(x - k0), s2 = sum((x - k0)^2),
// mean = k0 + s1/n, M2 = s2 - s1^2/n (k0 is a sample of the row, so the
// subtraction does not cancel catastrophically); ranges combine by the
// parallel-variance rule M2 = sum M2_i + sum n_i (mean_i - mean)^2.
#pragma once

#include "ptx.cuh"

namespace fnorm {

enum : int {
  MODE_PRE = 1,       // lazy pre-RMSNorm of A (sum of squares + epilogue scale)
  MODE_POST = 2,      // post-norm of the accumulator rows
  MODE_LN = 4,        // post-norm is LayerNorm (else RMSNorm)
  MODE_CLUSTER = 8,   // rows split over a cluster of CTAs along N
  MODE_SPILL = 16,    // spill layout: S slices per CTA, normalised from L2
  MODE_BRES = 32,     // all of B (K x BN, <= 128 KB) resident in shared memory
  MODE_PRE_LN = 64,   // the lazy pre-norm is LayerNorm (mean removed by a column-sum correction)
  MODE_AFF = 128,     // lazy pre-norm affine folded into B: column sums and a bias per column
  MODE_RES = 256,     // residual R added to the accumulator before the post-norm
  // backward of the Lazy Pre-RMSNorm GEMM
  MODE_BT = 512,      // B operand K-major: read from a row-major [N, K] array (B^T of a [K, N] matrix)
  MODE_AT = 1024,     // A operand MN-major: read from a row-major [K, M] array (A^T of an [M, K] matrix)
  MODE_DGRAD = 4096,  // RMSNorm backward epilogue: y = u + c[m] * X[m, n]
  // post-norm of rows wider than a cluster holds: the row statistics are
  // exchanged grid-wide through global memory (a cooperative launch), each
  // CTA keeping one 256-column tile in tensor memory while the row block's
  // other tiles, on any CTAs of the grid, publish theirs
  MODE_GX = 8192,
  // two-CTA MMA: the two CTAs of a cluster compute one [256 x BN] tile with
  // tcgen05 cta_group::2, each staging its own 128 rows of A and half of B's
  // BN columns, so that each SM takes in a third less per tile
  MODE_CTA2 = 16384,
  // B shared by a 2-CTA cluster along M: the two CTAs compute the tiles of
  // two neighbouring row blocks at the same columns, each with its own
  // one-CTA MMAs, and each loads half of every stage's B tile with a TMA
  // multicast into both CTAs' shared memory, so each SM takes in a third less
  // per k-block; a stage is free again once both CTAs' MMAs have read it
  MODE_MCB = 32768,
  // post-norm backward epilogue on the GEMM whose accumulator is dC = dL/dC
  // (with MODE_POST; MODE_LN for LayerNorm): with h_hat = (X - beta) / gamma
  // rebuilt from the forward output X and dh = dC * gamma,
  //   dH = rstd * (dh - mean_n(dh) - h_hat * mean_n(dh * h_hat))
  // (RMSNorm: no mean_n(dh) term), rstd the forward's; the two row sums are
  // exchanged like the forward's statistics.  Column partials of dC * h_hat
  // (dgamma) and dC (dbeta) over each 32 rows go to a workspace.
  MODE_NBWD = 65536,
};

struct FusedParams {
  int M, N, K;
  int cluster;      // CTAs per cluster along N (1 without MODE_CLUSTER)
  int slices;       // S: BN-column slices per CTA and row block (1 unless MODE_SPILL)
  int wave;         // 256-row units of one wave of 2-CTA clusters (half the SMs): the A^T GEMMs' k order
  int l2_hints;     // the backward GEMMs' L2 policy: 0 none, 1 A evict_first, 2 and B evict_last
  float eps, pre_eps;
  const __nv_bfloat16* gamma;
  const __nv_bfloat16* beta;
  __nv_bfloat16* C;  // the output, re-read by the spill layout
  float* mean_out;
  float* rstd_out;
  float* pre_rstd_out;
  const float* colsum;        // [N] column sums of the (gamma-folded) B (MODE_PRE_LN)
  const float* bias;          // [N] beta @ B, or NULL (MODE_AFF)
  const __nv_bfloat16* R;     // [M, N] residual (MODE_RES)
  const float* rowcoef;       // MODE_DGRAD: [M] coefficients c of the forward rows
  const __nv_bfloat16* X;     // MODE_DGRAD: [M, N] forward input rows; MODE_NBWD: [M, N] forward output
  const float* rstd_in;       // MODE_NBWD: [M] the forward's rstd
  float* cpart;               // MODE_NBWD: [ceil(M/32)][2][N] column partials (dgamma, dbeta), or NULL
  // MODE_GX workspace: per-(row block, tile) row statistics, per-row-block
  // arrival counters (zero at launch; the last CTA to finish zeroes them
  // again) and the CTA finish counter
  float2* gx_part;
  unsigned long long* gx_cnt;
  uint32_t* gx_finish;
  uint32_t* status;
  unsigned long long wait_limit_ns;
};

__host__ __device__ constexpr int pow2_at_least(int x, int lo) {
  int p = lo;
  while (p < x) p <<= 1;
  return p;
}

// Shared-memory control block.  Arrays a mode does not use shrink to one
// element (SSN: pre-norm row sums, SS1N: pre-LayerNorm shifted sums, NSN:
// spill-layout handoff, NBR: resident-B k-blocks), so each kernel carries
// only what it needs.
template <int STAGES_, int GB, int CLMAX, int SSN, int SS1N, int NSN, int NPART, int HD, int NBR, int GW, int GI,
          int GWI>
struct Aux {
  uint64_t full[STAGES_];
  uint64_t empty[STAGES_];
  uint64_t mdone[STAGES_];  // CTA pair, rank 1: the MMAs have read the stage (its norm warps' signal)
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t ss_full[2];
  uint64_t ss_empty[2];
  uint64_t xbar[2];
  uint64_t gxbar[2];  // grid exchange: the polling lane's "row block complete" to the other epilogue warps
  uint64_t nstat_full[HD];   // epilogue -> normaliser handoff, HD deep
  uint64_t nstat_empty[HD];
  uint64_t ebar[4][2];  // bounded barrier of the two epilogue warps of each TMEM lane quarter
  uint64_t teardown;
  uint64_t bres_full[NBR];  // one per k-block of resident B
  uint64_t rload;           // the first residual tile, loaded by TMA (one arrival per epilogue warp)
  uint32_t tmem_base;
  int abort_flag;
  int gx_last;   // grid exchange: this CTA finished last
  int nstat_m0[HD];
  int nstat_c0[HD];
  float ss[2][NPART][SSN];    // pre-norm row sums, one slot per norm-warp part
  float ss1[2][NPART][SS1N];  // pre-LayerNorm: shifted sums of the A rows and the shift
  float ssk[2][SS1N];
  float2 nstat[HD][NSN];
  float2 hstat[2][2][128];  // [parity][column half][row]: partial statistics of each half
  alignas(16) float gam[GB];
  alignas(16) float bet[GB];
  alignas(16) float igam[GI];  // post-norm backward: 1 / gamma of the CTA's columns (bet: -beta / gamma)
  // resident grid exchange: each epilogue warp's gamma/beta for the columns
  // of its half of the current tile (tiles change column group)
  alignas(16) float wgam[GW > 1 ? 8 : 1][GW];
  alignas(16) float wbet[GW > 1 ? 8 : 1][GW];  // (post-norm backward: -beta / gamma)
  alignas(16) float wigam[GWI > 1 ? 8 : 1][GWI];  // post-norm backward: 1 / gamma
  float2 xstat[2][CLMAX > 0 ? CLMAX : 1][CLMAX > 0 ? 128 : 1];  // cluster exchange: the C CTAs' partials
};

constexpr uint32_t kSmemLimit = 232448;  // 227 KB of opt-in shared memory per CTA
constexpr int kMaxStages = 8;
constexpr int kEpiWarps = 8;
constexpr uint32_t kBoxBytes = 32 * 64;  // one [32 rows x 32 columns] bf16 store box

template <int BN_, int MODE_, int CLMAX_ = 0>
struct KCfg {
  static constexpr int BN = BN_, MODE = MODE_, BK = 64, BM = 128;
  static constexpr bool PRE = (MODE & MODE_PRE) != 0;
  static constexpr bool POST = (MODE & MODE_POST) != 0;
  static constexpr bool LN = (MODE & MODE_LN) != 0;
  static constexpr bool CLUSTER = (MODE & MODE_CLUSTER) != 0;
  static constexpr bool SPILL = (MODE & MODE_SPILL) != 0;
  static constexpr bool BRES = (MODE & MODE_BRES) != 0;
  static constexpr bool PRE_LN = (MODE & MODE_PRE_LN) != 0;
  static constexpr bool AFF = (MODE & MODE_AFF) != 0;
  static constexpr bool RES = (MODE & MODE_RES) != 0;
  static constexpr bool BT = (MODE & MODE_BT) != 0;
  static constexpr bool AT = (MODE & MODE_AT) != 0;
  static constexpr bool DGRAD = (MODE & MODE_DGRAD) != 0;
  static constexpr bool GX = (MODE & MODE_GX) != 0;
  static constexpr bool CTA2 = (MODE & MODE_CTA2) != 0;
  static constexpr bool MCB = (MODE & MODE_MCB) != 0;
  static constexpr bool NBWD = (MODE & MODE_NBWD) != 0;
  static constexpr bool PAIR = CTA2 || MCB;    // a 2-CTA cluster along M shares each tile sequence
  static constexpr int CG = CTA2 ? 2 : 1;      // CTA group of every tcgen05 instruction
  static constexpr int RB = PAIR ? 256 : 128;  // rows of one tile sequence unit (one or two row blocks)
  static constexpr int BNS = CTA2 ? BN / 2 : BN;  // columns of B this CTA stages
  // the spill layout's in-place normalisation runs in its own warps (10-13)
  // unless those warps compute the Lazy Pre-Norm sums of squares
  static constexpr bool NORMW = SPILL && !PRE;
  static constexpr bool AUXW = PRE || NORMW;  // warps 10-13 present
  static constexpr int HALF = BN / 2;          // columns per epilogue half
  static constexpr int NCH = HALF / 32;        // 32-column subtiles per half
  // 32-column subtiles loaded from TMEM per wait: the whole half when the
  // register budget allows (320 threads: 168 registers), else two (448
  // threads: 128 registers; cluster exchange code needs the room too), or
  // one where two do not divide the half (192-column tiles: three subtiles)
  static constexpr int LDB = (DGRAD || NBWD) ? 1  // (these also hold their X values)
                             : (AUXW || ((CLUSTER || GX) && NCH > 2)) ? (NCH < 2 ? NCH : (NCH % 2 == 0 ? 2 : 1))
                                                                       : NCH;
  static_assert(NCH % LDB == 0, "the TMEM load batches cover the half tile exactly");
  static constexpr bool KEEP = (LDB == NCH);  // one TMEM read serves statistics and output
  static constexpr int CLMAX = CLUSTER ? CLMAX_ : 0;  // largest cluster the exchange buffers hold
  static constexpr int GB = (POST && !SPILL && !GX) ? BN : 1;  // gamma/beta kept in shared memory
  static constexpr int GW = GX ? HALF : 1;  // grid exchange: per-warp gamma/beta of a half tile
  static constexpr int GI = (NBWD && !GX) ? BN : 1;    // post-norm backward: 1 / gamma of the CTA's slice
  static constexpr int GWI = (NBWD && GX) ? HALF : 1;  // post-norm backward, grid exchange: per warp
  static constexpr int TMEM_COLS = pow2_at_least(2 * BN, 32);  // two accumulator buffers
  static constexpr uint32_t A_BYTES = BM * BK * 2;
  static constexpr uint32_t B_BYTES = BK * BNS * 2;
  // resident B: up to 128 KB, i.e. KB_MAX k-blocks of [64 x BN]
  static constexpr int KB_MAX = BRES ? (int)(131072u / B_BYTES) : 0;
  static constexpr uint32_t BRES_BYTES = (uint32_t)KB_MAX * B_BYTES;
  static constexpr uint32_t STAGE_BYTES = A_BYTES + (BRES ? 0u : B_BYTES);
  static constexpr int SSN = PRE ? 128 : 1, SS1N = PRE_LN ? 128 : 1, NSN = SPILL ? 128 : 1;
  // depth of the epilogue -> normaliser handoff (a power of two; 4 measured
  // no faster than 2 for the grid exchange)
  static constexpr int HDEPTH = 2;
  // norm warps: 4 (one row per thread), or 8 for the pre-LayerNorm, whose
  // shifted sums cost more per element: two parts take half of each row's
  // 16-byte chunks each
  static constexpr int NPART = PRE_LN ? 2 : 1;
  static constexpr int AUX_WARPS = AUXW ? 4 * NPART : 0;
  static constexpr uint32_t AUX_BYTES =
      (sizeof(Aux<kMaxStages, GB, CLMAX, SSN, SS1N, NSN, NPART, HDEPTH, (BRES ? KB_MAX : 1), GW, GI, GWI>) + 15) /
      16 * 16;
  // epilogue staging: 8 warps x STG_BUFS store boxes.  One box per warp when
  // that buys a pipeline stage and either the ring is below 4 stages, or a
  // warp stores only one box per tile (64-column tiles), so that nothing
  // waits on the single buffer within a tile (a narrow tile streams A at a
  // rate set by the bytes its ring keeps in flight), or the tile is a CTA
  // pair's (six stages measured 160 us against 169 us for five on an
  // 8192 x 4096 x 4096 GEMM).  Not for the post-norm backward's grid
  // exchange, whose tiles are bound by an epilogue that stores as much as it
  // reads: at 16384 x 4096 x 2048 its kernel took 212-215 us with two
  // buffers and three stages, 252 us with one and four, 228 us with three or
  // four buffers and three stages.
  static constexpr int stages_with(int bufs) {
    return (int)((kSmemLimit - 1024 - BRES_BYTES - kEpiWarps * bufs * kBoxBytes - AUX_BYTES) / STAGE_BYTES);
  }
  static constexpr int STG_BUFS =
      ((stages_with(2) < 4 || NCH == 1 || CTA2) && stages_with(1) > stages_with(2) && stages_with(2) < kMaxStages &&
       !(NBWD && GX))
          ? 1
          : 2;
  static constexpr uint32_t STG_BYTES = kEpiWarps * STG_BUFS * kBoxBytes;
  static constexpr int STAGES = stages_with(STG_BUFS) < kMaxStages ? stages_with(STG_BUFS) : kMaxStages;
  static constexpr uint32_t SMEM_BYTES = 1024 + BRES_BYTES + STAGES * STAGE_BYTES + STG_BYTES + AUX_BYTES;
  static constexpr int NUM_THREADS = 32 * (2 + kEpiWarps + AUX_WARPS);
  // M of each MMA: 256 only for the CTA pair's cta_group::2 MMAs; every
  // one-CTA MMA (B multicast included) is M = 128
  static constexpr uint32_t IDESC = make_idesc_bf16_f32(CG * BM, BN, !BT, AT);
  static_assert(((IDESC >> 24) & 31u) * 16u == (CTA2 ? 256u : 128u), "MMA M: 128 per CTA, 256 for a CTA pair");

  static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "UMMA N in 64..256, step 64");
  static_assert(STAGES >= 2, "shared memory too small for a 2-stage ring");
  static_assert(!SPILL || (BN == 256 && POST && CLUSTER), "spill layout: 256-column slices, post-norm, a cluster");
  static_assert(!GX || (POST && BN == 256 && !CLUSTER && !SPILL && !RES && !BRES),
                "grid exchange: resident 256-column tiles, no cluster");
  static_assert(!CLUSTER || (POST && CLMAX_ >= 1 && CLMAX_ <= 8), "clusters serve the post-norm, up to 8 CTAs");
  static_assert(!BRES || !CLUSTER, "resident B serves one CTA per row block");
  static_assert(!(PRE_LN || AFF) || (PRE && !POST), "the folded-affine pre-norm serves the pre-norm GEMM alone");
  static_assert(!PRE_LN || AFF, "the pre-LayerNorm needs its column sums");
  static_assert(!RES || (POST && !PRE), "the residual serves the post-norm");
  static_assert(!(BT || AT || DGRAD) || ((!POST || (NBWD && !AT && !DGRAD)) && !BRES && !AFF && !RES),
                "backward operand layouts serve the plain and lazy GEMMs and the post-norm backward");
  static_assert(!NBWD || (POST && !PRE && !RES && !SPILL && !BRES && !MCB && !CTA2 && HALF <= 128),
                "post-norm backward: resident tiles (one CTA, a cluster or the grid exchange), X values of a half "
                "tile in registers");
  static_assert(!DGRAD || (BT && !AT && !PRE), "the dgrad: B^T operand, per-row coefficients from memory");
  static_assert(!DGRAD || HALF <= 128, "the dgrad holds a half tile of X in registers");
  static_assert(!CTA2 || (BN == 256 && !POST && !BRES && !RES && !BT && !AT && !DGRAD),
                "two-CTA MMA: 256-column tiles of the plain and lazy pre-norm GEMMs");
  static_assert(!MCB || (!CTA2 && (BN == 128 || BN == 256) && !CLUSTER && !SPILL && !BRES && !RES && (!POST || GX)),
                "B multicast: the plain, transposed, lazy pre-norm, dgrad and grid-exchange post-norm GEMMs "
                "(not the post-norm backward)");
};

// Spill layout: normalise in place `nrows` rows (r0..) of one 256-column slice
// (columns c0..c0+255) of C, re-read from L2.  Lane l owns columns
// c0+8l..c0+8l+7; mean and rstd of row r0+i are held by lane lane_off+i.
// RIF rows of loads are in flight per lane: the pass is bound by L2 round
// trips, nrows / RIF of them.
template <bool LN, int RIF = 8>
__device__ __forceinline__ void normalize_slice(const FusedParams& p, int r0, int nrows, int lane_off, int c0,
                                                float mean, float rstd, int lane) {
  const int col = c0 + lane * 8;
  const bool colok = col < p.N;
  float gv[8], bv[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    gv[j] = 1.0f;
    bv[j] = 0.0f;
  }
  if (colok && p.gamma != nullptr) {
    const uint4 u = *reinterpret_cast<const uint4*>(p.gamma + col);
    gv[0] = bf16_lo(u.x); gv[1] = bf16_hi(u.x); gv[2] = bf16_lo(u.y); gv[3] = bf16_hi(u.y);
    gv[4] = bf16_lo(u.z); gv[5] = bf16_hi(u.z); gv[6] = bf16_lo(u.w); gv[7] = bf16_hi(u.w);
  }
  if (colok && p.beta != nullptr) {
    const uint4 u = *reinterpret_cast<const uint4*>(p.beta + col);
    bv[0] = bf16_lo(u.x); bv[1] = bf16_hi(u.x); bv[2] = bf16_lo(u.y); bv[3] = bf16_hi(u.y);
    bv[4] = bf16_lo(u.z); bv[5] = bf16_hi(u.z); bv[6] = bf16_lo(u.w); bv[7] = bf16_hi(u.w);
  }
  uint64_t g2[4], b2[4];  // gamma, beta as packed pairs
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    g2[h] = f2(gv[2 * h], gv[2 * h + 1]);
    b2[h] = f2(bv[2 * h], bv[2 * h + 1]);
  }
#pragma unroll 1
  for (int rr = 0; rr < nrows; rr += RIF) {
    uint4 v[RIF];
#pragma unroll
    for (int u = 0; u < RIF; ++u) {
      const int m = r0 + rr + u;
      v[u] = make_uint4(0, 0, 0, 0);
      if (colok && rr + u < nrows && m < p.M) v[u] = ld_global_cg_v4(p.C + static_cast<size_t>(m) * p.N + col);
    }
#pragma unroll
    for (int u = 0; u < RIF; ++u) {
      const float mu = __shfl_sync(0xffffffffu, mean, (lane_off + rr + u) & 31);
      const float rs = __shfl_sync(0xffffffffu, rstd, (lane_off + rr + u) & 31);
      const int m = r0 + rr + u;
      if (colok && rr + u < nrows && m < p.M) {
        const uint32_t in[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
        const uint64_t mu2 = f2(mu, mu), rs2 = f2(rs, rs);
        uint32_t o[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          // y = (x - mean) * rstd * gamma + beta
          const uint64_t x = f2(bf16_lo(in[h]), bf16_hi(in[h]));
          o[h] = pack_bf16x2_f2(f2_fma(f2_mul(LN ? f2_sub(x, mu2) : x, rs2), g2[h], b2[h]));
        }
        st_global_v4(p.C + static_cast<size_t>(m) * p.N + col, make_uint4(o[0], o[1], o[2], o[3]));
      }
    }
  }
}

// Load NB consecutive 32-column subtiles of this warp's TMEM lanes with a
// single wait (one round trip instead of NB).
template <int NB>
__device__ __forceinline__ void tmem_load_batch(uint32_t taddr, uint32_t (&r)[NB][32]) {
#pragma unroll
  for (int b = 0; b < NB; ++b) tmem_ld_32x32b_x32(taddr + b * 32, r[b]);
  tmem_ld_wait();
#pragma unroll
  for (int b = 0; b < NB; ++b) reg_fence(r[b]);
}

// Accumulate one 32-column subtile of raw accumulator values into row sums:
// LayerNorm s1 += u - k, s2 += (u - k)^2 (k: the shift); RMSNorm s2 += u^2.
// Even and odd columns go to separate sums ([0], [1]); a full subtile runs
// them as packed pairs.  Columns j >= lim are ignored.
template <bool LN>
__device__ __forceinline__ void accum_stats(const uint32_t (&r)[32], int lim, float k, float (&s1)[2],
                                            float (&s2)[2]) {
  if (lim >= 32) {
    const uint64_t kk = f2(k, k);
    uint64_t a1 = f2(s1[0], s1[1]), a2 = f2(s2[0], s2[1]);
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
      const uint64_t u = f2u(r[j], r[j + 1]);
      const uint64_t d = LN ? f2_sub(u, kk) : u;
      if (LN) a1 = f2_add(a1, d);
      a2 = f2_fma(d, d, a2);
    }
    if (LN) {
      s1[0] = f2_lo(a1);
      s1[1] = f2_hi(a1);
    }
    s2[0] = f2_lo(a2);
    s2[1] = f2_hi(a2);
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (j < lim) {
        const float d = LN ? __uint_as_float(r[j]) - k : __uint_as_float(r[j]);
        if (LN) s1[j & 1] += d;
        s2[j & 1] = fmaf(d, d, s2[j & 1]);
      }
    }
  }
}

// y = (u * a + b) * gamma_j + beta_j for one 32-column subtile, packed to
// bf16 pairs (two FMAs per element; gamma/beta read as float4 broadcasts)
__device__ __forceinline__ void affine_pack(const uint32_t (&r)[32], float a, float b, const float* gam,
                                            const float* bet, uint32_t (&w)[16]) {
  const uint64_t aa = f2(a, a), bb = f2(b, b);
#pragma unroll
  for (int j = 0; j < 32; j += 4) {
    const float4 g = *reinterpret_cast<const float4*>(gam + j);
    const float4 be = *reinterpret_cast<const float4*>(bet + j);
    const uint64_t y01 = f2_fma(f2_fma(f2u(r[j], r[j + 1]), aa, bb), f2(g.x, g.y), f2(be.x, be.y));
    const uint64_t y23 = f2_fma(f2_fma(f2u(r[j + 2], r[j + 3]), aa, bb), f2(g.z, g.w), f2(be.z, be.w));
    w[j >> 1] = pack_bf16x2_f2(y01);
    w[(j >> 1) + 1] = pack_bf16x2_f2(y23);
  }
}

// y = u * a (a = 1 for the plain GEMM), packed to bf16 pairs
template <bool SCALE>
__device__ __forceinline__ void scale_pack(const uint32_t (&r)[32], float a, uint32_t (&w)[16]) {
  const uint64_t aa = f2(a, a);
#pragma unroll
  for (int j = 0; j < 32; j += 2) {
    const uint64_t u = f2u(r[j], r[j + 1]);
    w[j >> 1] = pack_bf16x2_f2(SCALE ? f2_mul(u, aa) : u);
  }
}

// Lazy pre-norm with folded affine: y = u * a + (colsum_n * c + bias_n) for
// one 32-column subtile (c = -mean * rstd for LayerNorm, 0 for RMSNorm), whose
// column sums and bias are held by the warp's lanes, four columns each (lane
// l: columns 4l .. 4l + 3 of the half tile, zero past N), not read from
// memory per subtile: column j of the subtile comes from lane src0 + j / 4 by
// a shuffle.  Every lane of the warp must call it.
template <bool HAS_CS>
__device__ __forceinline__ void prenorm_pack_lanes(const uint32_t (&r)[32], float a, float c, const float4& cs4,
                                                   const float4& bi4, bool has_bias, int src0, uint32_t (&w)[16]) {
  const uint64_t aa = f2(a, a), cc = f2(c, c);
#pragma unroll
  for (int j = 0; j < 32; j += 4) {
    const int src = src0 + (j >> 2);
    float4 sc = make_float4(0.f, 0.f, 0.f, 0.f), bb = make_float4(0.f, 0.f, 0.f, 0.f);
    if (HAS_CS) {
      sc.x = __shfl_sync(0xffffffffu, cs4.x, src);
      sc.y = __shfl_sync(0xffffffffu, cs4.y, src);
      sc.z = __shfl_sync(0xffffffffu, cs4.z, src);
      sc.w = __shfl_sync(0xffffffffu, cs4.w, src);
    }
    if (has_bias) {
      bb.x = __shfl_sync(0xffffffffu, bi4.x, src);
      bb.y = __shfl_sync(0xffffffffu, bi4.y, src);
      bb.z = __shfl_sync(0xffffffffu, bi4.z, src);
      bb.w = __shfl_sync(0xffffffffu, bi4.w, src);
    }
    const uint64_t y01 = f2_fma(f2u(r[j], r[j + 1]), aa, f2_fma(f2(sc.x, sc.y), cc, f2(bb.x, bb.y)));
    const uint64_t y23 = f2_fma(f2u(r[j + 2], r[j + 3]), aa, f2_fma(f2(sc.z, sc.w), cc, f2(bb.z, bb.w)));
    w[j >> 1] = pack_bf16x2_f2(y01);
    w[(j >> 1) + 1] = pack_bf16x2_f2(y23);
  }
}

// Residual through the accumulator: write R[m, col0 .. col0 + 32*NC) (bf16,
// widened exactly to fp32) into this warp's TMEM lanes of an accumulator
// buffer, which the MMAs of the next tile in that buffer then accumulate onto
// (D = A @ B + R).  Rows past M and columns past N are written as zero (N is
// a multiple of 8, so 8-column groups are whole).  Returns after the stores
// have completed.
template <int NC>
__device__ __forceinline__ void preload_residual(const FusedParams& p, uint32_t taddr, int m, int col0) {
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    uint32_t v[32];
#pragma unroll
    for (int g8 = 0; g8 < 4; ++g8) {
      const int col = col0 + c * 32 + g8 * 8;
      uint4 x = make_uint4(0, 0, 0, 0);
      if (m < p.M && col < p.N) x = __ldg(reinterpret_cast<const uint4*>(p.R + static_cast<size_t>(m) * p.N + col));
      const uint32_t in[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int hh = 0; hh < 4; ++hh) {
        v[g8 * 8 + 2 * hh] = __float_as_uint(bf16_lo(in[hh]));
        v[g8 * 8 + 2 * hh + 1] = __float_as_uint(bf16_hi(in[hh]));
      }
    }
    tmem_st_32x32b_x32(taddr + c * 32, v);
  }
  tmem_st_wait();
}

// Parallel-variance combination: fold (mean_b, m2_b) over nb values into
// (mean, m2) over n values.
__device__ __forceinline__ void combine_mean_m2(float& mean, float& m2, float& n, float mean_b, float m2_b,
                                                float nb) {
  if (nb <= 0.0f) return;
  const float nn = n + nb;
  const float d = mean_b - mean;
  const float w = nb / nn;
  mean += d * w;
  m2 += m2_b + d * d * (n * w);
  n = nn;
}

// Column sums over the 32 rows a warp holds (one row per lane): v[j] is this
// lane's value of column j; lane l returns the sum of column l.  Five
// butterfly rounds, each halving the columns a lane keeps (16 + 8 + 4 + 2 + 1
// shuffles); the additions run in a fixed order, so the sums are the same on
// every run.  v is consumed.
__device__ __forceinline__ float warp_column_sums(float (&v)[32], int lane) {
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const bool upper = (lane & w) != 0;
#pragma unroll
    for (int j = 0; j < w; ++j) {
      const float keep = upper ? v[j + w] : v[j];
      const float send = upper ? v[j] : v[j + w];
      v[j] = keep + __shfl_xor_sync(0xffffffffu, send, w);
    }
  }
  return v[0];
}

// element e (0..7) of eight bf16 values packed in a uint4, widened to fp32
__device__ __forceinline__ float bf16_of(const uint4& v, int e) {
  const uint32_t w = (e >> 1) == 0 ? v.x : (e >> 1) == 1 ? v.y : (e >> 1) == 2 ? v.z : v.w;
  return (e & 1) ? bf16_hi(w) : bf16_lo(w);
}

// ---------------------------------------------------------------------------
template <class Cfg>
__global__ void __launch_bounds__(Cfg::NUM_THREADS, 1)
    fused_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmR,
                      const FusedParams p) {
  constexpr int BK = Cfg::BK, BN = Cfg::BN, STAGES = Cfg::STAGES, HALF = Cfg::HALF, NCH = Cfg::NCH;
  constexpr bool PRE = Cfg::PRE, POST = Cfg::POST, LN = Cfg::LN, CLUSTER = Cfg::CLUSTER, SPILL = Cfg::SPILL;
  constexpr bool BRES = Cfg::BRES, NORMW = Cfg::NORMW;
  constexpr bool PRE_LN = Cfg::PRE_LN, AFF = Cfg::AFF, RES = Cfg::RES;
  constexpr bool BT = Cfg::BT, AT = Cfg::AT, DGRAD = Cfg::DGRAD, GX = Cfg::GX;
  constexpr bool CTA2 = Cfg::CTA2, MCB = Cfg::MCB, PAIR = Cfg::PAIR, NBWD = Cfg::NBWD;
  constexpr int CG = Cfg::CG, RB = Cfg::RB;
  constexpr uint32_t A_BYTES = Cfg::A_BYTES, STAGE_BYTES = Cfg::STAGE_BYTES;
  using AuxT = Aux<STAGES, Cfg::GB, Cfg::CLMAX, Cfg::SSN, Cfg::SS1N, Cfg::NSN, Cfg::NPART, Cfg::HDEPTH,
                   (Cfg::BRES ? Cfg::KB_MAX : 1), Cfg::GW, Cfg::GI, Cfg::GWI>;
  constexpr int HD = Cfg::HDEPTH;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base0 = (raw_addr + 1023u) & ~1023u;  // swizzle atoms need 1024-byte alignment
  const uint32_t bres_base = base0;                     // resident B (MODE_BRES)
  const uint32_t base = base0 + Cfg::BRES_BYTES;        // the stage ring
  uint8_t* smem = smem_raw + (base - raw_addr);
  const uint32_t stg_base = base + STAGES * STAGE_BYTES;
  AuxT* aux = reinterpret_cast<AuxT*>(smem + STAGES * STAGE_BYTES + Cfg::STG_BYTES);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int M = p.M, N = p.N, K = p.K;
  const int C = CLUSTER ? p.cluster : 1;
  const int S = SPILL ? p.slices : 1;
  const int rank = CLUSTER ? static_cast<int>(cluster_ctarank()) : 0;
  // CTA pair: rank 0 issues the MMAs of both CTAs; each CTA owns rows
  // prank * 128 .. + 127 of every 256-row tile
  // (B multicast: the same rows split, but each CTA issues its own MMAs)
  const int prank = PAIR ? static_cast<int>(cluster_ctarank()) : 0;
  const bool issuer = !CTA2 || prank == 0;
  const int num_m = (M + RB - 1) / RB;
  const int cta_cols = S * BN;
  const int group_cols = cta_cols * C;
  const int ngroups = (N + group_cols - 1) / group_cols;
  const int total = num_m * ngroups;  // row blocks (x column groups) to visit
  const int CP = PAIR ? 2 : C;  // CTAs that share each tile sequence
  const int cid = static_cast<int>(blockIdx.x) / CP;
  const int ncl = static_cast<int>(gridDim.x) / CP;
  const int num_kb = (K + BK - 1) / BK;
  // The k-th tile of this CTA (t = row block * ngroups + column group):
  // cid + k * ncl.  The lazy pre-norm GEMMs without a post-norm whose rows
  // span several column groups take runs of RUN neighbouring tiles instead:
  // iterations RUN q .. RUN q + RUN - 1 take tiles RUN (q ncl + cid) and the
  // next RUN - 1, mostly of one row block, so the norm warps sum its rows once
  // per run; a round of runs still spans only RUN * ncl consecutive tiles (a
  // few row blocks of A), and the last, partial round goes back to single
  // tiles.  (Runs of four measured 0.7-0.9 % faster than pairs, with the same
  // outputs bit for bit.)
  constexpr bool PAIRS = PRE && !POST && !CLUSTER && !SPILL;
  constexpr int RUN = 4;
  const int full_rounds = PAIRS && ngroups > 1 ? total / (RUN * ncl) : 0;
  auto tile_of = [&](int k) -> int {
    if (k < RUN * full_rounds) return RUN * ((k / RUN) * ncl + cid) + (k % RUN);
    return RUN * full_rounds * ncl + cid + (k - RUN * full_rounds) * ncl;
  };
  // The per-row statistics multiply by 1/N and 1/K (correctly rounded
  // reciprocals: exact, as a division would be, whenever N and K are powers
  // of two) instead of dividing; a division costs far more on the epilogue's
  // critical path.  Recomputed where used, so no register holds them.
  auto inv_N = [&]() { return __frcp_rn(static_cast<float>(N)); };
  auto inv_K = [&]() { return __frcp_rn(static_cast<float>(K)); };

  const WaitCtx wc{p.wait_limit_ns, p.status, &aux->abort_flag};

  // a clustered kernel run in a cluster of any other size only reports it
  if ((CLUSTER || PAIR) && !cluster_shape_ok(static_cast<uint32_t>(PAIR ? 2 : C), p.status)) return;

  // ---------------- set-up ----------------
  if (warp == 0) {
    // the barriers, initialised by the 32 lanes of warp 0 in parallel
    for (int s = lane; s < STAGES; s += 32) {
      mbar_init(smem_u32(&aux->full[s]), 1);
      mbar_init(smem_u32(&aux->mdone[s]), 1);
      // the MMA's commit (B multicast: both CTAs' MMAs, which read what this
      // CTA's multicast wrote), and for the lazy pre-norm the norm warps' reads
      mbar_init(smem_u32(&aux->empty[s]), (MCB ? 2 : 1) + (PRE ? 4 * Cfg::NPART : 0));
    }
    if (lane < 2) {
      const int b = lane;
      mbar_init(smem_u32(&aux->acc_full[b]), 1);
      // (CTA pair: the epilogue warps of both CTAs, on rank 0's barrier)
      mbar_init(smem_u32(&aux->acc_empty[b]), kEpiWarps * CG);
      // handoffs between warp groups: one arrival per warp, after __syncwarp
      mbar_init(smem_u32(&aux->ss_full[b]), 4 * Cfg::NPART);
      mbar_init(smem_u32(&aux->ss_empty[b]), kEpiWarps);
      mbar_init(smem_u32(&aux->xbar[b]), 1);
      mbar_init(smem_u32(&aux->gxbar[b]), 1);
      for (int qq = 0; qq < 4; ++qq) mbar_init(smem_u32(&aux->ebar[qq][b]), kEpiWarps / 4);
    }
    if (lane >= 2 && lane < 2 + HD) {
      mbar_init(smem_u32(&aux->nstat_full[lane - 2]), kEpiWarps);
      mbar_init(smem_u32(&aux->nstat_empty[lane - 2]), 4);
    }
    for (int kb = lane; kb < (BRES ? Cfg::KB_MAX : 1); kb += 32) mbar_init(smem_u32(&aux->bres_full[kb]), 1);
    if (lane == 31) {
      mbar_init(smem_u32(&aux->teardown), 1);
      mbar_init(smem_u32(&aux->rload), kEpiWarps);
      aux->abort_flag = 0;
    }
    fence_mbar_init();
  }
  if (warp == 2 && lane == 0) {
    // (an epilogue warp, idle until the set-up ends, so that the warm-up
    // starts at kernel entry rather than after the barrier set-up)
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmC);
    if (tile_of(0) < total) {
      // Warm L2 with the first ring of the first tile while the previous grid
      // in the stream finishes.  L2 is the point of coherence, so a line
      // brought in now still sees that grid's later writes; the loads proper
      // are issued after griddepcontrol.wait.  (The residual layouts warm two
      // k-blocks only: their first MMA waits for the residual tile, whose
      // loads a deeper warm-up would delay; measured 10.7 -> 10.3 us.)
      const int t0 = tile_of(0);
      const int m0 = (t0 / ngroups) * RB + prank * Cfg::BM;
      const int n0 = ((t0 % ngroups) * C + rank) * cta_cols + (CTA2 ? prank * Cfg::BNS : 0);
      constexpr int kWarm = RES ? 2 : STAGES;
      const int nk = m0 < M ? (num_kb < kWarm ? num_kb : kWarm) : 0;
      for (int kb = 0; kb < nk; ++kb) {
        if (AT) {
          tma_prefetch_l2_2d(&tmA, m0, kb * BK);
          tma_prefetch_l2_2d(&tmA, m0 + 64, kb * BK);
        } else {
          tma_prefetch_l2_2d(&tmA, kb * BK, m0);
        }
        if (BT) {
          // (B multicast: this CTA's half of the B^T rows, the box it loads)
          tma_prefetch_l2_2d(&tmB, kb * BK, n0 + (MCB ? prank * (BN / 2) : 0));
        } else {
          for (int c = 0; c < Cfg::BNS / 64; ++c) tma_prefetch_l2_2d(&tmB, n0 + c * 64, kb * BK);
        }
      }
    }
  }
  if (warp == 1) {
    tmem_alloc<CG>(smem_u32(&aux->tmem_base), Cfg::TMEM_COLS);
    tmem_relinquish<CG>();
  }
  tc_fence_before();
  __syncthreads();
  if (CLUSTER || PAIR) cluster_sync();  // peers' barriers are initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem_base = aux->tmem_base;
  // Set-up above overlaps the previous grid in the stream; every global
  // access below comes after it has completed.
  grid_dependency_wait();
  if (threadIdx.x == 0) grid_launch_dependents();

  if (warp == 0) {
    // ======================= TMA producer =======================
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, filled = 0, fill_par = 0;
      int bres_issued = 0;  // resident-B k-blocks issued (each on its own barrier)
      // CTA pair, rank 1: rank 0's full barrier of a stage, and the copies
      // into this CTA's shared memory that complete on it
      auto peer_full0 = [&](uint32_t st) { return mapa_shared(smem_u32(&aux->full[st]), 0); };
      auto load_pair = [&](uint32_t dst, const CUtensorMap* m, int c0, int c1, uint32_t bar) {
        if (issuer) tma_load_2d(dst, m, c0, c1, bar);
        else tma_load_2d_pair(dst, m, c0, c1, bar);
      };
      // The backward's GEMMs (the A^T weight gradients and the Lazy Pre-Norm
      // data gradient) stream each A slab through one wave of tiles only,
      // while every wave reads all of B.  With more than one wave their A
      // loads go first out of L2, and B, where it fits, last, so that B
      // stays for the next wave (l2_hints; evict_normal is the default).
      constexpr bool HINT = AT || DGRAD;
      const uint64_t pol_a = !HINT ? 0 : p.l2_hints >= 1 ? l2_policy_evict_first() : l2_policy_evict_normal();
      const uint64_t pol_b = !HINT ? 0 : p.l2_hints >= 2 ? l2_policy_evict_last() : l2_policy_evict_normal();
      bool ok = true;
      for (int k = 0, t = tile_of(0); t < total && ok; t = tile_of(++k)) {
        const int m0 = (t / ngroups) * RB + prank * Cfg::BM;
        for (int s = 0; s < S && ok; ++s) {
          // (CTA pair: this CTA's half of the tile's B columns)
          const int n0 = ((t % ngroups) * C + rank) * cta_cols + s * BN + (CTA2 ? prank * Cfg::BNS : 0);
          // The A^T GEMMs (weight gradients: a reduction over the long M)
          // walk the reduction backwards on every other wave of B-multicast
          // clusters, their default schedule.  Each tile streams a column
          // slab of A and of B from end to end, so a wave that starts where
          // the previous one ended finds those k-blocks still in L2.  The
          // direction is a function of the output tile alone (the wave that
          // its 256-row unit and column group fall in), so that both CTAs of
          // a pair walk the same k-blocks and one-CTA tiles sum each output
          // in the same order (the MMA's accumulate flag follows the loop
          // order, not kb).
          const bool back = AT && ((((m0 / 256) * ngroups + t % ngroups) / p.wave) & 1);
          for (int kj = 0; kj < num_kb; ++kj) {
            const int kb = back ? num_kb - 1 - kj : kj;
            // (CTA pair: the stage is released by rank 0's MMA commit)
            if (!mbar_wait(wc, smem_u32(&aux->empty[stage]), phase ^ 1u, kSiteProducer)) {
              ok = false;
              break;
            }
            if (BRES && k == 0) {
              // all of B once, during the first tile: k-block kb just ahead
              // of the A stage that pairs with it, so the first MMAs need not
              // wait for the whole of B
              const uint32_t bf = smem_u32(&aux->bres_full[kb]);
              mbar_arrive_expect_tx(bf, Cfg::B_BYTES);
#pragma unroll
              for (int c = 0; c < BN / 64; ++c)
                tma_load_2d(bres_base + kb * Cfg::B_BYTES + c * (BK * 128), &tmB, c * 64, kb * BK, bf);
              bres_issued = kb + 1;
            }
            // CTA pair: both CTAs' copies complete on rank 0's full barrier,
            // which rank 0 arms with the bytes of both (rank 1's may land
            // first: the transaction count runs negative until rank 0 arrives)
            const uint32_t full = (CTA2 && !issuer) ? peer_full0(stage) : smem_u32(&aux->full[stage]);
            if (!CTA2 || issuer) mbar_arrive_expect_tx(full, CTA2 ? 2u * STAGE_BYTES : STAGE_BYTES);
            const uint32_t sa = base + stage * STAGE_BYTES;
            if (CTA2) {
              load_pair(sa, &tmA, kb * BK, m0, full);
            } else if (AT) {
              // A^T: two MN-major chunks of [64 k-rows x 64 m] from the [K, M] array
              tma_load_2d_hint(sa, &tmA, m0, kb * BK, full, pol_a);
              tma_load_2d_hint(sa + BK * 128, &tmA, m0 + 64, kb * BK, full, pol_a);
            } else if (HINT) {
              tma_load_2d_hint(sa, &tmA, kb * BK, m0, full, pol_a);
            } else {
              tma_load_2d(sa, &tmA, kb * BK, m0, full);
            }
            if (!BRES) {
              const uint32_t sb = sa + A_BYTES;
              if (BT) {
                // B^T: one K-major box of [BN n-rows x 64 k] from the [N, K] array
                // (B multicast: this CTA's half of its rows, a [BN/2 x 64]
                // box, into both CTAs at the same offset)
                if (MCB && HINT)
                  tma_load_2d_mc_hint(sb + static_cast<uint32_t>(prank * (BN / 2) * 128), &tmB, kb * BK,
                                      n0 + prank * (BN / 2), full, 0x3, pol_b);
                else if (MCB)
                  tma_load_2d_mc(sb + static_cast<uint32_t>(prank * (BN / 2) * 128), &tmB, kb * BK,
                                 n0 + prank * (BN / 2), full, 0x3);
                else if (HINT)
                  tma_load_2d_hint(sb, &tmB, kb * BK, n0, full, pol_b);
                else
                  tma_load_2d(sb, &tmB, kb * BK, n0, full);
              } else {
#pragma unroll
                for (int c = 0; c < Cfg::BNS / 64; ++c) {
                  if (CTA2) {
                    load_pair(sb + c * (BK * 128), &tmB, n0 + c * 64, kb * BK, full);
                  } else if (MCB) {
                    // this CTA's half of the tile's B boxes, into both CTAs
                    // (same offset; each CTA's full barrier counts all of B)
                    if (c / (BN >= 128 ? BN / 128 : 1) == prank) {
                      if (HINT)
                        tma_load_2d_mc_hint(sb + c * (BK * 128), &tmB, n0 + c * 64, kb * BK, full, 0x3, pol_b);
                      else
                        tma_load_2d_mc(sb + c * (BK * 128), &tmB, n0 + c * 64, kb * BK, full, 0x3);
                    }
                  } else if (HINT) {
                    tma_load_2d_hint(sb + c * (BK * 128), &tmB, n0 + c * 64, kb * BK, full, pol_b);
                  } else {
                    tma_load_2d(sb + c * (BK * 128), &tmB, n0 + c * 64, kb * BK, full);
                  }
                }
              }
            }
            filled |= 1u << stage;
            fill_par = (fill_par & ~(1u << stage)) | (phase << stage);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      // teardown drain: every copy issued into shared memory lands before exit
      // (CTA pair, rank 1: its copies complete on rank 0's barriers; it waits
      // instead until the MMAs have read each stage it filled.  After an
      // abort those reads may never come: each wait is then cut to 100 us,
      // ample for copies already in flight to land, so the launch returns in
      // well under a millisecond instead of a wait limit per stage)
      const bool pair_short = CTA2 && !issuer && *wc.abort_flag;
      const WaitCtx wdrain{pair_short ? (wc.limit_ns < 100000ull ? wc.limit_ns : 100000ull) : wc.limit_ns, wc.status,
                           wc.abort_flag};
      for (int s = 0; s < STAGES; ++s)
        if ((filled >> s) & 1u)
          mbar_wait<false, true>(wdrain,
                                 smem_u32((CTA2 && !issuer) ? (PRE ? &aux->mdone[s] : &aux->empty[s]) : &aux->full[s]),
                                 (fill_par >> s) & 1u, kSiteTeardown);
      for (int kb = 0; kb < bres_issued; ++kb)
        mbar_wait<false, true>(wc, smem_u32(&aux->bres_full[kb]), 0, kSiteTeardown);
      // B multicast: the peer's MMA commits arrive on this CTA's empty
      // barriers; once both CTAs' MMAs have released the last fill of every
      // stage, none of them is still on its way here
      if (MCB)
        for (int s = 0; s < STAGES; ++s)
          if ((filled >> s) & 1u) mbar_wait<false, true>(wc, smem_u32(&aux->empty[s]), (fill_par >> s) & 1u, kSiteTeardown);
    }
  } else if (warp == 1) {
    // ======================= MMA issuer =======================
    // (CTA pair: rank 0 issues for both CTAs; rank 1's warp 1 only holds its
    // share of the tensor memory)
    if (lane == 0 && issuer) {
      uint32_t stage = 0, phase = 0;
      int it = 0;
      bool ok = true;
      for (int k = 0, t = tile_of(0); t < total && ok; t = tile_of(++k)) {
        for (int s = 0; s < S && ok; ++s, ++it) {
          const int buf = it & 1;
          const uint32_t aph = static_cast<uint32_t>(it >> 1) & 1u;
          // with the residual, the epilogue releases each buffer once more
          // up front, after writing the first tile's R into it
          if (!mbar_wait<CTA2>(wc, smem_u32(&aux->acc_empty[buf]), RES ? aph : aph ^ 1u, kSiteMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d0 = tmem_base + static_cast<uint32_t>(buf * BN);
          for (int kb = 0; kb < num_kb; ++kb) {
            if (!mbar_wait(wc, smem_u32(&aux->full[stage]), phase, kSiteMma) ||
                (BRES && it == 0 && !mbar_wait(wc, smem_u32(&aux->bres_full[kb]), 0, kSiteMma))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = base + stage * STAGE_BYTES;
            const uint32_t sb = BRES ? bres_base + kb * Cfg::B_BYTES : sa + A_BYTES;
#pragma unroll
            for (int ks = 0; ks < BK / 16; ++ks) {
              // K-major operand (A; B^T): 128-byte rows, 8-row groups 1024 bytes
              // apart; a K step of 16 elements is 32 bytes inside the swizzled row.
              // MN-major operand (B; A^T): 64-element chunks of 64 k-rows x 128
              // bytes; LBO = chunk stride along M or N, SBO = 8-row group stride
              // along K; a K step of 16 rows is 2048 bytes.
              const uint64_t da = AT ? make_smem_desc(sa + ks * (16 * 128), BK * 128, 1024, kSwizzle128B)
                                     : make_smem_desc(sa + ks * 32, 16, 1024, kSwizzle128B);
              const uint64_t db = BT ? make_smem_desc(sb + ks * 32, 16, 1024, kSwizzle128B)
                                     : make_smem_desc(sb + ks * (16 * 128), BK * 128, 1024, kSwizzle128B);
              umma_bf16<CG>(d0, da, db, Cfg::IDESC, (RES || (kb | ks) != 0) ? 1u : 0u);
            }
            if (CTA2) {
              umma_commit_pair(smem_u32(&aux->empty[stage]), 0x3);  // both CTAs' stage
              // rank 1's norm warps read its A rows once the stage is known complete
              if (PRE) umma_commit_pair(smem_u32(&aux->mdone[stage]), 0x2);
            } else if (MCB) {
              umma_commit_mc(smem_u32(&aux->empty[stage]), 0x3);  // both CTAs' stage (B written by both)
            } else {
              umma_commit(smem_u32(&aux->empty[stage]));
            }
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (ok) {
            if (CTA2) umma_commit_pair(smem_u32(&aux->acc_full[buf]), 0x3);
            else umma_commit(smem_u32(&aux->acc_full[buf]));
          }
        }
      }
      // every MMA issued has completed before tensor memory is released
      umma_commit<CG>(smem_u32(&aux->teardown));
      mbar_wait<false, true>(wc, smem_u32(&aux->teardown), 0, kSiteTeardown);
    }
  } else if (warp < 2 + kEpiWarps) {
    // ======================= epilogue (8 warps) =======================
    const int q = warp & 3;            // TMEM lane quarter this warp may access
    const int h = (warp - 2) >> 2;     // column half of each tile
    const int row = q * 32 + lane;     // tile row of this thread
    const int etid = static_cast<int>(threadIdx.x) - 64;  // 0..255
    const uint32_t stg = stg_base + static_cast<uint32_t>(warp - 2) * (Cfg::STG_BUFS * kBoxBytes);
    uint32_t sbuf = 0;
    int it = 0;


    // stage one [32 rows x 32 columns] bf16 box of this warp's rows (64-byte
    // swizzle) and store it with TMA
    auto store_box = [&](const uint32_t (&w)[16], int col0, int m0) {
      const uint32_t sbase = stg + sbuf * kBoxBytes;
      if (lane == 0) {
        // the store that last used this buffer, STG_BUFS stores ago, has read it
        bulk_wait_read<Cfg::STG_BUFS - 1>();
      }
      __syncwarp();
      // row `lane` of the box: 16-byte chunk ch sits at chunk (ch ^ ((row >> 1) & 3))
      const uint32_t rbase = sbase + static_cast<uint32_t>(lane) * 64u;
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        const uint32_t a = rbase + (static_cast<uint32_t>(ch ^ ((lane >> 1) & 3)) << 4);
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
      sbuf = sbuf + 1u == static_cast<uint32_t>(Cfg::STG_BUFS) ? 0u : sbuf + 1u;
    };

    // give an accumulator buffer back to the MMA issuer (CTA pair: on rank 0's
    // barrier, released at cluster scope; rank 0's MMAs write both CTAs'
    // tensor memory)
    auto release_acc = [&](int b) {
      if (lane == 0) {
        if (CTA2 && !issuer) mbar_arrive_remote(mapa_shared(smem_u32(&aux->acc_empty[b]), 0));
        else mbar_arrive(smem_u32(&aux->acc_empty[b]));
      }
    };

    // barrier of the two epilogue warps that share this TMEM lane quarter
    // (the same 32 rows, one column half each) on an mbarrier, so that it is
    // bounded like every other wait (returns false if it gave up)
    int esn = 0;
    auto esync = [&]() -> bool {
      const int b = esn & 1;
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&aux->ebar[q][b]));
      const bool r =
          mbar_wait_warp(wc, smem_u32(&aux->ebar[q][b]), static_cast<uint32_t>(esn >> 1) & 1u, kSiteEpilogue);
      ++esn;
      return r;
    };

    // combine this row's partial statistics of the two column halves, in
    // half order (identical in both halves)
    auto combine_halves = [&](float& part0, float& part1, float nh0, float nh1) -> bool {
      const int hp = esn & 1;
      aux->hstat[hp][h][row] = make_float2(part0, part1);
      if (!esync()) return false;
      const float2 a = aux->hstat[hp][0][row];
      const float2 b = aux->hstat[hp][1][row];
      if (NBWD) {
        // the norm backward's row reductions are plain sums
        part0 = a.x + b.x;
        part1 = a.y + b.y;
      } else if (LN && nh0 == nh1 && nh0 > 0.0f) {
        // equal halves (every full tile): the combination's weights are
        // exactly 1/2 and nh/2, the same values without its divisions
        const float d = b.x - a.x;
        part0 = a.x + d * 0.5f;
        part1 = a.y + (b.y + d * d * (nh0 * 0.5f));
      } else if (LN) {
        float mean = 0.0f, m2 = 0.0f, n = 0.0f;
        combine_mean_m2(mean, m2, n, a.x, a.y, nh0);
        combine_mean_m2(mean, m2, n, b.x, b.y, nh1);
        part0 = mean;
        part1 = m2;
      } else {
        part0 = a.x + b.x;
        part1 = 0.0f;
      }
      return true;
    };

    // exchange (part0, part1) of this row with the cluster and combine them
    // in rank order; half 0 pushes, both halves wait and combine; returns
    // false if the wait gave up
    auto exchange = [&](float& part0, float& part1, int g, int xit) -> bool {
      if constexpr (!CLUSTER) {
        return true;  // (no cluster: nothing to exchange, no exchange buffers)
      } else {
        const int xp = xit & 1;
        const uint32_t xb = smem_u32(&aux->xbar[xp]);
        if (etid == 0) mbar_arrive_expect_tx(xb, static_cast<uint32_t>(C) * 128u * 8u);
        if (h == 0) {
          const uint32_t mine = smem_u32(&aux->xstat[xp][rank][row]);
          for (int r2 = 0; r2 < C; ++r2) st_async_f32x2(mapa_shared(mine, r2), part0, part1, mapa_shared(xb, r2));
        }
        if (!mbar_wait_warp<true>(wc, xb, static_cast<uint32_t>(xit >> 1) & 1u, kSiteExchange)) return false;
        float n_acc = 0.0f, m_acc = 0.0f, q_acc = 0.0f;
        for (int r2 = 0; r2 < C; ++r2) {
          const float2 v = aux->xstat[xp][r2][row];
          const int nq = min(max(N - (g * C + r2) * cta_cols, 0), cta_cols);
          if (NBWD) {
            m_acc += v.x;
            q_acc += v.y;
          } else if (LN) {
            combine_mean_m2(m_acc, q_acc, n_acc, v.x, v.y, static_cast<float>(nq));
          } else {
            q_acc += v.x;
          }
        }
        part0 = (LN || NBWD) ? m_acc : q_acc;
        part1 = q_acc;
        return true;
      }
    };

    // residual: write R of iteration it2's tile into its accumulator buffer
    // (this warp's lanes and column half); false if there is no such tile
    auto preload_iter = [&](int it2) -> bool {
      const int t2 = cid + (it2 / S) * ncl;
      if (t2 >= total) return false;
      const int g2 = t2 % ngroups;
      const int n0b = (g2 * C + rank) * cta_cols + (it2 % S) * BN;
      const uint32_t tb2 = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                           static_cast<uint32_t>((it2 & 1) * BN + h * HALF);
      preload_residual<NCH>(p, tb2, (t2 / ngroups) * Cfg::BM + row, n0b + h * HALF);
      return true;
    };
    // The first tile's residual by TMA, when a warp's staging buffers hold its
    // half of a tile: each warp loads its [32 x 32] boxes of R (the C store
    // layout, zero-filled past M and N), then every lane moves its row into
    // tensor memory.  One bulk copy per box instead of a 16-byte load per row
    // segment, so the first MMA, which waits for this, is not held up behind
    // the ring's loads.  Returns 1 when loaded, 0 with no tile, -1 if the
    // wait gave up.
    constexpr bool RTMA = RES && !CLUSTER && !SPILL && NCH <= Cfg::STG_BUFS;
    auto preload_first_tma = [&]() -> int {
      if (cid >= total) return 0;
      const int n0b = ((cid % ngroups) * C + rank) * cta_cols + h * HALF;
      const int r0 = (cid / ngroups) * Cfg::BM + q * 32;
      const uint32_t bar = smem_u32(&aux->rload);
      if (lane == 0) {
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(NCH) * kBoxBytes);
#pragma unroll
        for (int c = 0; c < NCH; ++c) tma_load_2d(stg + c * kBoxBytes, &tmR, n0b + c * 32, r0, bar);
      }
      if (!mbar_wait_warp(wc, bar, 0u, kSiteEpilogue)) {
        // gave up (or another role did): the copies in flight land before
        // this CTA can exit (bounded teardown drain)
        if (lane == 0) mbar_wait<false, true>(wc, bar, 0u, kSiteTeardown);
        __syncwarp();
        return -1;
      }
      const uint32_t tb0 = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(h * HALF);
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        // row `lane` of box c: 16-byte chunk ch at chunk ch ^ ((row >> 1) & 3)
        const uint32_t rbase = stg + c * kBoxBytes + static_cast<uint32_t>(lane) * 64u;
        uint32_t v[32];
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t x0, x1, x2, x3;
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(x0), "=r"(x1), "=r"(x2), "=r"(x3)
                       : "r"(rbase + (static_cast<uint32_t>(ch ^ ((lane >> 1) & 3)) << 4))
                       : "memory");
          const uint32_t in[4] = {x0, x1, x2, x3};
#pragma unroll
          for (int hh = 0; hh < 4; ++hh) {
            v[ch * 8 + 2 * hh] = __float_as_uint(bf16_lo(in[hh]));
            v[ch * 8 + 2 * hh + 1] = __float_as_uint(bf16_hi(in[hh]));
          }
        }
        tmem_st_32x32b_x32(tb0 + c * 32, v);
      }
      tmem_st_wait();
      return 1;
    };
    bool preload_ok = true;
    if (RES) {
      // the first two tiles' buffers start out holding their residual
      for (int i2 = 0; i2 < 2; ++i2) {
        if (RTMA && i2 == 0) {
          const int r = preload_first_tma();
          if (r < 0) {
            preload_ok = false;
            break;
          }
          if (r == 0) break;
        } else if (!preload_iter(i2)) {
          break;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&aux->acc_empty[i2]));
      }
    }
    if (POST && !SPILL && !GX) {
      // resident post-norm CTAs own one fixed BN-column slice of every row
      // (after the residual preload, which the first MMA waits for)
      const int n0 = rank * BN;
      for (int j = etid; j < BN; j += 32 * kEpiWarps) {
        const int n = n0 + j;
        aux->gam[j] = (p.gamma != nullptr && n < N) ? __bfloat162float(p.gamma[n]) : 1.0f;
        aux->bet[j] = (p.beta != nullptr && n < N) ? __bfloat162float(p.beta[n]) : 0.0f;
        if (NBWD) {
          // h_hat = (x - beta) / gamma as x * (1/gamma) + (-beta/gamma)
          aux->igam[j] = __frcp_rn(aux->gam[j]);
          aux->bet[j] = -aux->bet[j] * aux->igam[j];
        }
      }
      asm volatile("bar.sync 1, 256;" ::: "memory");  // the eight epilogue warps, before any wait
    }

    // Grid exchange of tile (row block, column group g): the column-half-0
    // warps publish the tile's statistics for its 128 rows and each counts
    // in on the row block's counter (4 arrivals per tile, atomic adds); one
    // lane of the CTA polls the counter until every tile of the row block
    // has arrived and passes that on through an mbarrier, on which the other
    // epilogue warps sleep rather than spin (one poller per CTA keeps the
    // counter's L2 line quiet for the arrivals, and sleeping waiters leave
    // the issue slots to the producer and MMA warps); then every warp
    // combines all the tiles' statistics in tile order (the same arithmetic
    // in every tile of the row, so every tile derives the same mean and
    // rstd).  xk counts this CTA's exchanges; exchange k completes phase k/2
    // of barrier k%2 (a warp cannot be two exchanges behind the poller: the
    // halves meet in combine_halves before every exchange).  False if a wait
    // gave up.
    int xk = 0;
    auto gx_exchange = [&](float& part0, float& part1, int m0_, int g_) -> bool {
      const int rb = m0_ / Cfg::BM;
      if (h == 0) p.gx_part[(static_cast<size_t>(rb) * ngroups + g_) * Cfg::BM + row] = make_float2(part0, part1);
      __syncwarp();
      if (h == 0 && lane == 0) grid_arrive(p.gx_cnt + rb);
      const uint32_t gxb = smem_u32(&aux->gxbar[xk & 1]);
      const uint32_t gxpar = static_cast<uint32_t>(xk >> 1) & 1u;
      ++xk;
      if (warp == 2) {
        bool ready = true;
        if (lane == 0) {
          ready = grid_wait_eq(wc, p.gx_cnt + rb, static_cast<unsigned long long>(4 * ngroups), kSiteGrid);
          // (the arrive releases at CTA scope what this lane acquired at GPU scope)
          if (ready) mbar_arrive(gxb);
        }
        if (!__all_sync(0xffffffffu, ready)) return false;
        __syncwarp();  // lane 0's acquire orders every lane's loads below
      } else if (!mbar_wait_warp(wc, gxb, gxpar, kSiteGrid)) {
        return false;
      }
      // Combine the tiles' statistics in tile order, XB per batch of loads in
      // flight (fewer where the norm warps leave fewer registers).
      // LayerNorm in two passes over them, without a division per step:
      // mean = sum_q n_q mean_q / N, then M2 = sum_q (M2_q + n_q (mean_q - mean)^2).
      constexpr int XB = (Cfg::AUXW || NBWD) ? 8 : 32;
      const float2* src = p.gx_part + static_cast<size_t>(rb) * ngroups * Cfg::BM + row;
      auto nq = [&](int qq) { return static_cast<float>(min(max(N - qq * cta_cols, 0), cta_cols)); };
      if (NBWD) {
        // the norm backward's two row sums: plain sums, in tile order
        float a0 = 0.0f, a1 = 0.0f;
        for (int q0 = 0; q0 < ngroups; q0 += XB) {
          float2 v[XB];
#pragma unroll
          for (int u = 0; u < XB; ++u)
            v[u] = q0 + u < ngroups ? __ldcg(src + static_cast<size_t>(q0 + u) * Cfg::BM) : make_float2(0.f, 0.f);
#pragma unroll
          for (int u = 0; u < XB; ++u) {
            a0 += v[u].x;
            a1 += v[u].y;
          }
        }
        part0 = a0;
        part1 = a1;
        return true;
      }
      float acc = 0.0f;  // LayerNorm: sum n_q mean_q; RMSNorm: sum of squares
      float2 v[XB];
      for (int q0 = 0; q0 < ngroups; q0 += XB) {
#pragma unroll
        for (int u = 0; u < XB; ++u)
          v[u] = q0 + u < ngroups ? __ldcg(src + static_cast<size_t>(q0 + u) * Cfg::BM) : make_float2(0.f, 0.f);
#pragma unroll
        for (int u = 0; u < XB; ++u) acc = LN ? fmaf(nq(q0 + u), v[u].x, acc) : acc + v[u].x;
      }
      if (!LN) {
        part0 = acc;
        part1 = 0.0f;
        return true;
      }
      const float mean = acc * inv_N();
      float m2 = 0.0f;
      for (int q0 = 0; q0 < ngroups; q0 += XB) {
        if (q0 > 0 || ngroups > XB) {  // (one batch: its values are still in registers)
#pragma unroll
          for (int u = 0; u < XB; ++u)
            v[u] = q0 + u < ngroups ? __ldcg(src + static_cast<size_t>(q0 + u) * Cfg::BM) : make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < XB; ++u) {
          const float d = v[u].x - mean;
          m2 += v[u].y + nq(q0 + u) * (d * d);
        }
      }
      part0 = mean;
      part1 = m2;
      return true;
    };

    // spill-layout state: running shifted sums of this half over the current
    // row block, and (inline normalisation only) the pending row block
    float k0 = 0.0f, sum1 = 0.0f, sum2 = 0.0f;
    bool pend = false;
    int pm0 = 0, pc0 = 0, pnext = 0;
    float pmean = 0.0f, prstd = 1.0f;
    int xit = 0;  // row-block statistics completed so far
    bool ok = preload_ok;

    for (int k = 0, t = tile_of(0); t < total && ok; t = tile_of(++k)) {
      const int m0 = (t / ngroups) * RB + prank * Cfg::BM;  // first row of this CTA's tile rows
      const int g = t % ngroups;
      for (int s = 0; s < S && ok; ++s, ++it) {
        const int n0 = (g * C + rank) * cta_cols + s * BN;  // first column of the tile
        const int c0h = n0 + h * HALF;                      // first column of this half
        const int buf = it & 1;
        const uint32_t aph = static_cast<uint32_t>(it >> 1) & 1u;
        // resident grid exchange: this half's gamma (lanes 0-15) and beta
        // (lanes 16-31), 8 columns per lane, loaded while the tile's MMAs run
        uint4 gbv = make_uint4(0x3f803f80u, 0x3f803f80u, 0x3f803f80u, 0x3f803f80u);  // bf16 1.0 pairs
        if (GX) {
          const int col = c0h + (lane & 15) * 8;
          const __nv_bfloat16* src = lane < 16 ? p.gamma : p.beta;
          if (lane >= 16) gbv = make_uint4(0u, 0u, 0u, 0u);
          if (src != nullptr && col < N) gbv = __ldg(reinterpret_cast<const uint4*>(src + col));
        }
        // pre-norm with folded affine: this half's column sums and bias, four
        // columns per lane, loaded while the tile's MMAs run (the epilogue
        // hands them to the lanes by shuffles)
        float4 cs4 = make_float4(0.f, 0.f, 0.f, 0.f), bi4 = make_float4(0.f, 0.f, 0.f, 0.f);
        if (AFF) {
          const int col = c0h + 4 * lane;
          if (4 * lane < HALF && col < N) {
            if (PRE_LN) cs4 = __ldg(reinterpret_cast<const float4*>(p.colsum + col));
            if (p.bias != nullptr) bi4 = __ldg(reinterpret_cast<const float4*>(p.bias + col));
          }
        }
        // dgrad, post-norm backward: this half's X values (and the forward
        // rstd of the row), loaded while the tile's MMAs run
        uint4 xv[(DGRAD || NBWD) ? NCH : 1][4];
        const float rstd_row = (NBWD && m0 + row < M) ? __ldg(p.rstd_in + m0 + row) : 0.0f;
        if (DGRAD || NBWD) {
#pragma unroll
          for (int c = 0; c < NCH; ++c)
#pragma unroll
            for (int g8 = 0; g8 < 4; ++g8) {
              const int col = c0h + c * 32 + g8 * 8;
              xv[c][g8] = make_uint4(0, 0, 0, 0);
              if (m0 + row < M && col < N)
                xv[c][g8] = __ldg(reinterpret_cast<const uint4*>(p.X + static_cast<size_t>(m0 + row) * N + col));
            }
        }
        if (!mbar_wait_warp(wc, smem_u32(&aux->acc_full[buf]), aph, kSiteEpilogue)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                            static_cast<uint32_t>(buf * BN + h * HALF);

        // ---- lazy pre-norm scale: rstd (and, for LayerNorm, mean) of the A row ----
        float pre = 1.0f, pre_mean = 0.0f;
        if (PRE) {
          const int sb = it & 1;
          if (!mbar_wait_warp(wc, smem_u32(&aux->ss_full[sb]), static_cast<uint32_t>(it >> 1) & 1u,
                              kSiteEpilogue)) {
            ok = false;
            break;
          }
          const float ss = Cfg::NPART == 2 ? aux->ss[sb][0][row] + aux->ss[sb][Cfg::NPART - 1][row]
                                           : aux->ss[sb][0][row];
          if (PRE_LN) {
            // LayerNorm of the A row from its shifted sums (shift: ssk)
            const float s1 = Cfg::NPART == 2 ? aux->ss1[sb][0][row] + aux->ss1[sb][Cfg::NPART - 1][row]
                                             : aux->ss1[sb][0][row];
            const float mu = s1 * inv_K();
            pre_mean = aux->ssk[sb][row] + mu;
            const float var = fmaxf(ss * inv_K() - mu * mu, 0.0f);
            pre = rsqrtf(var + p.pre_eps);
          } else {
            pre = rsqrtf(ss * inv_K() + p.pre_eps);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&aux->ss_empty[sb]));
        }
        if (DGRAD) {
          // RMSNorm backward: dA = (rstd * dC) @ B^T + c * X, c = -rstd^2 (dC . C) / N
          const int mr = m0 + row;
          pre_mean = mr < M ? __ldg(p.rowcoef + mr) : 0.0f;
        }
        const int nvh = min(max(N - c0h, 0), HALF);  // valid columns of this half

        if (SPILL) {
          // ---- pass 1: statistics + un-normalised (pre-scaled) bf16 slice to C ----
          if (s == 0) sum1 = sum2 = 0.0f;
          for (int cb = 0; cb < NCH / Cfg::LDB; ++cb) {
            if (cb * Cfg::LDB * 32 >= nvh) break;
            uint32_t r[Cfg::LDB][32];
            tmem_load_batch<Cfg::LDB>(tb + cb * Cfg::LDB * 32, r);
            if (LN && s == 0 && cb == 0) k0 = __uint_as_float(r[0][0]);
#pragma unroll
            for (int b = 0; b < Cfg::LDB; ++b) {
              const int c = cb * Cfg::LDB + b;
              if (c * 32 >= nvh) break;
              float a1[2] = {0.f, 0.f}, a2[2] = {0.f, 0.f};
              accum_stats<LN>(r[b], nvh - c * 32, k0, a1, a2);
              sum1 += a1[0] + a1[1];
              sum2 += a2[0] + a2[1];
              uint32_t w[16];
              scale_pack<PRE>(r[b], pre, w);  // the (pre-scaled) value before the norm
              store_box(w, c0h + c * 32, m0);
            }
          }
          if (RES) preload_iter(it + 2);  // this buffer's next tile starts from its residual
          tc_fence_before();
          __syncwarp();
          release_acc(buf);

          // ---- (inline) one slice of the pending row block's normalisation ----
          if (!NORMW && pend) {
            normalize_slice<LN>(p, pm0 + q * 32 + 16 * h, 16, 16 * h, pc0 + pnext * BN, pmean, prstd, lane);
            if (++pnext == S) pend = false;
          }
          if (s == S - 1) {
            // ---- row block complete: statistics, exchange, then hand it over ----
            const int cbase = (g * C + rank) * cta_cols;
            float nh[2] = {0.f, 0.f};
            for (int s2 = 0; s2 < S; ++s2)
#pragma unroll
              for (int hh = 0; hh < 2; ++hh)
                nh[hh] += static_cast<float>(min(max(N - (cbase + s2 * BN + hh * HALF), 0), HALF));
            const float nmine = nh[h];
            float part0, part1;  // statistics of the pre-scaled values v = pre * u
            if (LN) {
              const float inv_nm = nmine > 0.0f ? 1.0f / nmine : 0.0f;
              part0 = nmine > 0.0f ? pre * (k0 + sum1 * inv_nm) : 0.0f;
              part1 = nmine > 0.0f ? pre * pre * fmaxf(sum2 - sum1 * sum1 * inv_nm, 0.0f) : 0.0f;
            } else {
              part0 = pre * pre * sum2;
              part1 = 0.0f;
            }
            if (!combine_halves(part0, part1, nh[0], nh[1]) || !exchange(part0, part1, g, xit)) {
              ok = false;
              break;
            }
            ++xit;
            const float mean = LN ? part0 : 0.0f;
            const float rstd = rsqrtf((LN ? part1 : part0) * inv_N() + p.eps);
            const int m = m0 + row;
            if (h == 0 && rank == 0 && g == 0 && m < M) {
              if (LN && p.mean_out != nullptr) p.mean_out[m] = mean;
              if (p.rstd_out != nullptr) p.rstd_out[m] = rstd;
              if (PRE && p.pre_rstd_out != nullptr) p.pre_rstd_out[m] = pre;
            }
            if (NORMW) {
              // hand the row block to the normaliser warps
              const int nb = xit - 1;
              const int b = nb & (HD - 1);
              if (!mbar_wait_warp(wc, smem_u32(&aux->nstat_empty[b]), (static_cast<uint32_t>(nb / HD) & 1u) ^ 1u,
                                  kSiteEpilogue)) {
                ok = false;
                break;
              }
              // this warp's un-normalised stores are complete and visible
              // before they are read back
              if (lane == 0) {
                bulk_wait<0>();
                fence_proxy_async_global();
              }
              __syncwarp();
              if (h == 0) aux->nstat[b][row] = make_float2(mean, rstd);
              if (etid == 0) {
                aux->nstat_m0[b] = m0;
                aux->nstat_c0[b] = cbase;
              }
              __syncwarp();
              if (lane == 0) mbar_arrive(smem_u32(&aux->nstat_full[b]));
            } else {
              while (pend) {  // (only when S == 1 would anything remain)
                normalize_slice<LN>(p, pm0 + q * 32 + 16 * h, 16, 16 * h, pc0 + pnext * BN, pmean, prstd, lane);
                if (++pnext == S) pend = false;
              }
              // both halves' stores of this block are complete before either
              // half re-reads rows the other half wrote
              if (lane == 0) {
                bulk_wait<0>();
                fence_proxy_async_global();
              }
              if (!esync()) {
                ok = false;
                break;
              }
              pend = true;
              pm0 = m0;
              pc0 = cbase;
              pnext = 0;
              pmean = mean;
              prstd = rstd;
            }
          }
          continue;
        }

        // ---- resident layouts: statistics straight from tensor memory ----
        constexpr int LDB = Cfg::LDB, NBATCH = NCH / LDB;
        uint32_t r[LDB][32];
        if (Cfg::KEEP) tmem_load_batch<LDB>(tb, r);  // the whole half, once
        // grid exchange: this warp's gamma/beta of the tile into its own
        // shared-memory slice (read back as float4 broadcasts after the
        // exchange; the previous tile's reads of the slice are complete)
        if (GX && !NBWD) {
          float* dst = (lane < 16 ? &aux->wgam[warp - 2][0] : &aux->wbet[warp - 2][0]) + (lane & 15) * 8;
          const uint32_t gw[4] = {gbv.x, gbv.y, gbv.z, gbv.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            dst[2 * e] = bf16_lo(gw[e]);
            dst[2 * e + 1] = bf16_hi(gw[e]);
          }
          __syncwarp();
        } else if (GX) {
          // post-norm backward: gamma and 1/gamma from lanes 0-15, -beta/gamma
          // from lanes 16-31 (which take their columns' gamma from lane - 16)
          const uint32_t gw[4] = {gbv.x, gbv.y, gbv.z, gbv.w};
          uint32_t ow[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) ow[e] = __shfl_xor_sync(0xffffffffu, gw[e], 16);
          const int o = (lane & 15) * 8;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float mine = (e & 1) ? bf16_hi(gw[e >> 1]) : bf16_lo(gw[e >> 1]);
            const float other = (e & 1) ? bf16_hi(ow[e >> 1]) : bf16_lo(ow[e >> 1]);
            if (lane < 16) {
              aux->wgam[warp - 2][o + e] = mine;
              aux->wigam[warp - 2][o + e] = __frcp_rn(mine);
            } else {
              aux->wbet[warp - 2][o + e] = -mine * __frcp_rn(other);
            }
          }
          __syncwarp();
        }
        float mean = 0.0f, rstd = 1.0f, proj = 0.0f;
        if constexpr (NBWD) {
          float part0 = 0.0f, part1 = 0.0f;
          // post-norm backward: the row sums of dh = u * gamma and dh * h_hat,
          // h_hat = (x - beta) / gamma, over this half's columns; the column
          // sums of u * h_hat and u over this warp's 32 rows (u is exactly zero
          // past M and N: those A rows and B columns are zero-filled)
          const int lim0 = m0 + row < M ? nvh : 0;
          const bool cols = p.cpart != nullptr;
#pragma unroll
          for (int c = 0; c < NCH; ++c) {
            if (c * 32 >= nvh) break;
            tmem_load_batch<1>(tb + c * 32, r);
            // (gamma, 1/gamma, -beta/gamma as float4 broadcasts)
            const float4* gm = reinterpret_cast<const float4*>(GX ? &aux->wgam[warp - 2][c * 32]
                                                                  : &aux->gam[h * HALF + c * 32]);
            const float4* be = reinterpret_cast<const float4*>(GX ? &aux->wbet[warp - 2][c * 32]
                                                                  : &aux->bet[h * HALF + c * 32]);
            const float4* ig = reinterpret_cast<const float4*>(GX ? &aux->wigam[warp - 2][c * 32]
                                                                  : &aux->igam[h * HALF + c * 32]);
            float va[32];
#pragma unroll
            for (int j4 = 0; j4 < 8; ++j4) {
              const float4 g4 = gm[j4], b4 = be[j4], i4 = ig[j4];
              const float gv[4] = {g4.x, g4.y, g4.z, g4.w};
              const float bv[4] = {b4.x, b4.y, b4.z, b4.w};
              const float iv[4] = {i4.x, i4.y, i4.z, i4.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int j = 4 * j4 + e;
                const float u = j < lim0 - c * 32 ? __uint_as_float(r[0][j]) : 0.0f;
                const float hh = fmaf(bf16_of(xv[c][j >> 3], j & 7), iv[e], bv[e]);
                const float dh = u * gv[e];
                part0 += dh;
                part1 = fmaf(dh, hh, part1);
                va[j] = u * hh;
                r[0][j] = __float_as_uint(u);
              }
            }
            if (cols) {
              float vb[32];
#pragma unroll
              for (int j = 0; j < 32; ++j) vb[j] = __uint_as_float(r[0][j]);
              const float sg = warp_column_sums(va, lane);
              const float sb = warp_column_sums(vb, lane);
              const int col = c0h + c * 32 + lane;
              if (m0 + q * 32 < M && col < N) {
                float* cp = p.cpart + static_cast<size_t>((m0 >> 5) + q) * 2 * N;
                cp[col] = sg;
                cp[N + col] = sb;
              }
            }
          }
          const float n_h0 = static_cast<float>(min(max(N - n0, 0), HALF));
          const float n_h1 = static_cast<float>(min(max(N - n0 - HALF, 0), HALF));
          if (!combine_halves(part0, part1, n_h0, n_h1)) {
            ok = false;
            break;
          }
          if (CLUSTER) {
            if (!exchange(part0, part1, g, xit)) {
              ok = false;
              break;
            }
            ++xit;
          } else if (GX) {
            if (!gx_exchange(part0, part1, m0, g)) {
              ok = false;
              break;
            }
          }
          // dH = rstd * (dh - mean_n(dh) - h_hat * mean_n(dh * h_hat))
          mean = LN ? part0 * inv_N() : 0.0f;
          proj = part1 * inv_N();
          rstd = rstd_row;
        } else if (POST) {
          float kk = 0.0f;
          float a1[2] = {0.f, 0.f}, a2[2] = {0.f, 0.f};
          for (int cb = 0; cb < NBATCH; ++cb) {
            if (cb * LDB * 32 >= nvh) break;
            if (!Cfg::KEEP) tmem_load_batch<LDB>(tb + cb * LDB * 32, r);
            if (LN && cb == 0) kk = __uint_as_float(r[0][0]);
#pragma unroll
            for (int b = 0; b < LDB; ++b) {
              const int lim = nvh - (cb * LDB + b) * 32;
              if (lim > 0) accum_stats<LN>(r[b], lim, kk, a1, a2);
            }
          }
          const float s1 = a1[0] + a1[1], s2 = a2[0] + a2[1];
          const float nf = static_cast<float>(nvh);
          float part0, part1;  // statistics of the pre-scaled values v = pre * u
          if (LN) {
            const float inv_nf = nvh == HALF ? 1.0f / static_cast<float>(HALF) : (nvh > 0 ? 1.0f / nf : 0.0f);
            part0 = nvh > 0 ? pre * (kk + s1 * inv_nf) : 0.0f;
            part1 = nvh > 0 ? pre * pre * fmaxf(s2 - s1 * s1 * inv_nf, 0.0f) : 0.0f;
          } else {
            part0 = pre * pre * s2;
            part1 = 0.0f;
          }
          const float n_h0 = static_cast<float>(min(max(N - n0, 0), HALF));
          const float n_h1 = static_cast<float>(min(max(N - n0 - HALF, 0), HALF));
          if (!combine_halves(part0, part1, n_h0, n_h1)) {
            ok = false;
            break;
          }
          if (CLUSTER) {
            if (!exchange(part0, part1, g, xit)) {
              ok = false;
              break;
            }
            ++xit;
          } else if (GX && m0 < M) {
            // (B multicast: the second row block of the last pair may lie
            // past M; it has no statistics to exchange and stores nothing)
            if (!gx_exchange(part0, part1, m0, g)) {
              ok = false;
              break;
            }
          }
          if (LN) {
            mean = part0;
            rstd = rsqrtf(part1 * inv_N() + p.eps);
          } else {
            rstd = rsqrtf(part0 * inv_N() + p.eps);
          }
        }

        const int ew = warp - 2;
        // ---- normalise / scale, bf16, stage, TMA store: 32 columns at a time ----
        if constexpr (NBWD) {
          // dH = rstd * (u * gamma - mean_n(dh) - h_hat * mean_n(dh * h_hat))
          const float rm = -rstd * mean, rp = -rstd * proj;
#pragma unroll
          for (int c = 0; c < NCH; ++c) {
            const int col0 = c0h + c * 32;
            if (col0 >= N) break;
            tmem_load_batch<1>(tb + c * 32, r);
            const float4* gm = reinterpret_cast<const float4*>(GX ? &aux->wgam[ew][c * 32]
                                                                  : &aux->gam[h * HALF + c * 32]);
            const float4* be = reinterpret_cast<const float4*>(GX ? &aux->wbet[ew][c * 32]
                                                                  : &aux->bet[h * HALF + c * 32]);
            const float4* ig = reinterpret_cast<const float4*>(GX ? &aux->wigam[ew][c * 32]
                                                                  : &aux->igam[h * HALF + c * 32]);
            uint32_t w[16];
#pragma unroll
            for (int j4 = 0; j4 < 8; ++j4) {
              const float4 g4 = gm[j4], b4 = be[j4], i4 = ig[j4];
              const float gv[4] = {g4.x, g4.y, g4.z, g4.w};
              const float bv[4] = {b4.x, b4.y, b4.z, b4.w};
              const float iv[4] = {i4.x, i4.y, i4.z, i4.w};
              float y[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int j = 4 * j4 + e;
                const float hh = fmaf(bf16_of(xv[c][j >> 3], j & 7), iv[e], bv[e]);
                y[e] = fmaf(__uint_as_float(r[0][j]) * gv[e], rstd, fmaf(hh, rp, rm));
              }
              w[2 * j4] = pack_bf16x2(y[0], y[1]);
              w[2 * j4 + 1] = pack_bf16x2(y[2], y[3]);
            }
            store_box(w, col0, m0);
          }
        } else {
          for (int cb = 0; cb < NBATCH; ++cb) {
            if (c0h + cb * LDB * 32 >= N) break;
            if (!Cfg::KEEP) tmem_load_batch<LDB>(tb + cb * LDB * 32, r);
#pragma unroll
            for (int b = 0; b < LDB; ++b) {
              const int c = cb * LDB + b;
              const int col0 = c0h + c * 32;
              if (col0 >= N) break;
              uint32_t w[16];
              if (POST) {
                // y = (v - mean) * rstd * gamma + beta = (u*a + b) * gamma + beta, v = pre * u
                affine_pack(r[b], pre * rstd, LN ? -mean * rstd : 0.0f,
                            GX ? &aux->wgam[ew][c * 32] : &aux->gam[h * HALF + c * 32],
                            GX ? &aux->wbet[ew][c * 32] : &aux->bet[h * HALF + c * 32], w);
              } else if (DGRAD) {
                // y = u + c * x
                const uint64_t cc = f2(pre_mean, pre_mean);
#pragma unroll
                for (int g8 = 0; g8 < 4; ++g8) {
                  const uint32_t xw[4] = {xv[c][g8].x, xv[c][g8].y, xv[c][g8].z, xv[c][g8].w};
#pragma unroll
                  for (int hh = 0; hh < 4; ++hh) {
                    const int jj = g8 * 8 + 2 * hh;
                    w[jj >> 1] = pack_bf16x2_f2(f2_fma(f2(bf16_lo(xw[hh]), bf16_hi(xw[hh])), cc, f2u(r[b][jj], r[b][jj + 1])));
                  }
                }
              } else if (AFF) {
                // lazy pre-norm with folded affine: y = rstd * (u - mean * colsum_n) + bias_n
                prenorm_pack_lanes<PRE_LN>(r[b], pre, -pre_mean * pre, cs4, bi4, p.bias != nullptr, c * 8, w);
              } else {
                scale_pack<PRE>(r[b], pre, w);
              }
              store_box(w, col0, m0);
            }
          }
        }
        if (RES) preload_iter(it + 2);  // this buffer's next tile starts from its residual
        tc_fence_before();
        __syncwarp();
        release_acc(buf);

        // ---- row statistics ----
        const int m = m0 + row;
        if (h == 0 && m < M) {
          if (POST && !NBWD) {
            if (rank == 0 && (!GX || g == 0)) {
              if (LN && p.mean_out != nullptr) p.mean_out[m] = mean;
              if (p.rstd_out != nullptr) p.rstd_out[m] = rstd;
              if (PRE && p.pre_rstd_out != nullptr) p.pre_rstd_out[m] = pre;
            }
          } else if (PRE) {
            if (g == 0 && p.rstd_out != nullptr) p.rstd_out[m] = pre;
            if (PRE_LN && g == 0 && p.mean_out != nullptr) p.mean_out[m] = pre_mean;
          }
        }
      }
    }
    if (SPILL && !NORMW && ok) {
      while (pend) {  // the last row block
        normalize_slice<LN>(p, pm0 + q * 32 + 16 * h, 16, 16 * h, pc0 + pnext * BN, pmean, prstd, lane);
        if (++pnext == S) pend = false;
      }
    }
    if (lane == 0) bulk_wait_read<0>();  // staging is read; the writes complete with the grid
  } else if (NORMW) {
    // ======================= normaliser warps (spill layout) =======================
    const int k = warp - (2 + kEpiWarps);  // rows 32k..32k+31 of each row block
    int nb = 0;
    for (int t = cid; t < total; t += ncl, ++nb) {
      const int b = nb & (HD - 1);
      if (!mbar_wait_warp(wc, smem_u32(&aux->nstat_full[b]), static_cast<uint32_t>(nb / HD) & 1u, kSiteEpilogue))
        break;
      float2 st = aux->nstat[b][k * 32 + lane];
      const int m0 = aux->nstat_m0[b];
      const int c0 = aux->nstat_c0[b];
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&aux->nstat_empty[b]));
      for (int s = 0; s < S; ++s) normalize_slice<LN>(p, m0 + k * 32, 32, 0, c0 + s * BN, st.x, st.y, lane);
    }
  } else if (PRE) {
    // ======================= norm warps (Lazy Pre-Norm) =======================
    // 4 x NPART warps: warp nw takes row (nw % 4) * 32 + lane and part nw / 4
    // of each staged row's 16-byte chunks
    const int nw = warp - (2 + kEpiWarps);
    const int row = (nw & 3) * 32 + lane;
    const int part = nw >> 2;
    constexpr int ROW_BYTES = BK * 2;
    constexpr int CHUNKS = ROW_BYTES / 16;
    constexpr int CPP = CHUNKS / Cfg::NPART;  // chunks per part
    // swizzle phase of this row: chunk index XOR (row address bits 7..9)
    const int swz = ((row * ROW_BYTES) >> 7) & (CHUNKS - 1);
    uint32_t stage = 0, phase = 0;
    int it = 0;
    bool ok = true;
    // the previous tile's row block and this row's sums over it: a tile of the
    // same row block (the second of a pair) reuses them, still waiting for and
    // releasing every stage as the MMA does
    int held_rb = -1;
    float held_s2 = 0.0f, held_s1 = 0.0f, held_shift = 0.0f;
    for (int k = 0, t = tile_of(0); t < total && ok; t = tile_of(++k)) {
      const bool reuse = PAIRS && t / ngroups == held_rb;
      held_rb = t / ngroups;
      for (int s = 0; s < S && ok; ++s, ++it) {
        // packed pairs of partial sums: acc = sum of squares (of a - shift for
        // the pre-LayerNorm), lsum = sum of (a - shift)
        uint64_t acc[2] = {0ull, 0ull}, lsum[2] = {0ull, 0ull};
        float shift = 0.0f;
        uint64_t sh2 = 0ull;
        for (int kb = 0; kb < num_kb; ++kb) {
          // (CTA pair, rank 1: this CTA's copies complete on rank 0's barrier;
          // the MMAs' commit says the stage is complete)
          if (!mbar_wait_warp(wc, smem_u32((CTA2 && !issuer) ? &aux->mdone[stage] : &aux->full[stage]), phase,
                              kSiteNorm)) {
            ok = false;
            break;
          }
          const uint8_t* arow = smem + stage * STAGE_BYTES + row * ROW_BYTES;
          if (PRE_LN && kb == 0 && !reuse) {
            // the shift is the row's first element, a[row][0] (logical chunk 0),
            // the same for both parts
            shift = bf16_lo(*reinterpret_cast<const uint32_t*>(arow + (swz << 4)));
            sh2 = f2(shift, shift);
          }
#pragma unroll
          for (int c = 0; c < (reuse ? 0 : CPP); ++c) {
            // visit the part's chunks in a bank-conflict-free order (the
            // lanes' rows have distinct swizzle phases); sums do not depend
            // on the order
            const int ch = part * CPP + c;
            const uint4 v = *reinterpret_cast<const uint4*>(arow + ((ch ^ swz) << 4));
            const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const uint64_t x = f2(bf16_lo(wv[e]), bf16_hi(wv[e]));
              if (PRE_LN) {
                // zero-filled K tail: a = 0 contributes (0 - shift), removed below
                const uint64_t d = f2_sub(x, sh2);
                lsum[e & 1] = f2_add(lsum[e & 1], d);
                acc[e & 1] = f2_fma(d, d, acc[e & 1]);
              } else {
                acc[e & 1] = f2_fma(x, x, acc[e & 1]);
              }
            }
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
        if (!mbar_wait_warp(wc, smem_u32(&aux->ss_empty[sb]), (static_cast<uint32_t>(it >> 1) & 1u) ^ 1u,
                            kSiteNorm)) {
          ok = false;
          break;
        }
        float s2t = (f2_lo(acc[0]) + f2_hi(acc[0])) + (f2_lo(acc[1]) + f2_hi(acc[1]));
        float s1t = 0.0f;
        if (PRE_LN) {
          s1t = (f2_lo(lsum[0]) + f2_hi(lsum[0])) + (f2_lo(lsum[1]) + f2_hi(lsum[1]));
          if (part == 0) {
            // the zero-filled tail of the last k-block added (0 - shift) per
            // element to one part or the other; both share the shift, so part
            // 0 removes all of it from the total
            const float pad = static_cast<float>(num_kb * BK - K);
            s1t += pad * shift;
            s2t -= pad * shift * shift;
          }
        }
        if (reuse) {
          s2t = held_s2;
          s1t = held_s1;
          shift = held_shift;
        } else {
          held_s2 = s2t;
          held_s1 = s1t;
          held_shift = shift;
        }
        if (PRE_LN) {
          if (part == 0) aux->ssk[sb][row] = shift;
          aux->ss1[sb][part][row] = s1t;
        }
        aux->ss[sb][part][row] = s2t;
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&aux->ss_full[sb]));
      }
    }
  }

  // ---------------- teardown ----------------
  tc_fence_before();
  __syncthreads();
  // CTA pair: rank 0 reaches this after its last MMA completed, so neither
  // CTA's tensor memory is still being written when it is released
  if (CTA2) cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<CG>(tmem_base, Cfg::TMEM_COLS);
  }
  if (CLUSTER || PAIR) cluster_sync();  // no CTA leaves while a peer may still address it
  if (GX) {
    // the last CTA of the grid to finish zeroes every counter this grid used
    // (and the finish count): the next launch on the workspace starts from
    // zero; every other CTA has finished its waits by then
    if (threadIdx.x == 0) {
      __threadfence();
      aux->gx_last = atomicAdd(p.gx_finish, 1u) == gridDim.x - 1u;
    }
    __syncthreads();
    if (aux->gx_last) {
      const int nrb = (M + Cfg::BM - 1) / Cfg::BM;
      for (int i = static_cast<int>(threadIdx.x); i < nrb; i += static_cast<int>(blockDim.x)) p.gx_cnt[i] = 0ull;
      if (threadIdx.x == 0) *reinterpret_cast<volatile uint32_t*>(p.gx_finish) = 0u;
    }
  }
}

}  // namespace fnorm
