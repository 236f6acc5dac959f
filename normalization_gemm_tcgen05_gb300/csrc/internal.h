// internal.h — host-side declarations shared by the translation units of
// libfnorm (not part of the public C ABI, which is include/fnorm.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "fnorm.h"

namespace fnorm {

// thread-local error message (returned by fnorm_last_error)
void set_error(const char* fmt, ...);
fnorm_status_t cuda_fail(cudaError_t e, const char* what);

struct DeviceInfo {
  int id;
  int num_sms;
  uint32_t* status;  // device status word of this device
};

// Properties of the current device, cached per device.  The first call on a
// device also resolves the address of its status word.
fnorm_status_t current_device(DeviceInfo* out);

uint64_t wait_limit_ns();
int forced_postnorm_cluster();
// programmatic dependent launch for every kernel of the library (environment
// variable FNORM_PDL=0 turns it off)
bool pdl_enabled();
// FNORM_PLAIN_GX_LAUNCH=1: the clustered grid exchange as a plain cluster
// launch instead of a cooperative one (for profilers that replay a
// cooperative launch without its clusters)
bool plain_cluster_grid_exchange();

// 2-D row-major bf16 tensor map: `inner` elements per row (contiguous),
// `outer` rows, `pitch_bytes` between rows; box of box_inner x box_outer.
fnorm_status_t encode_tmap_bf16_2d(CUtensorMap* map, const void* ptr, uint64_t inner, uint64_t outer,
                                   uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_outer,
                                   CUtensorMapSwizzle swizzle);

// Workspace of the grid-exchange post-norm: per-(row block, tile) row
// statistics, per-row-block arrival counters and the finish counter (both
// zero between calls).  Calls that share one must be ordered (one stream).
struct GxScratch {
  float2* part;              // [units][128]
  unsigned long long* cnt;   // [row blocks]
  uint32_t* finish;
  int units_cap;
  int rowblocks_cap;
};

// Bytes of the caller's grid-exchange workspace for an M x N post-norm, and
// its layout over a given buffer (FNORM_ERR_INVALID_ARG if it is too small or
// misaligned).  Nothing is allocated.  The counters have a fixed capacity of
// kGxMaxRowBlocks 128-row blocks (M up to 2^21); taller calls take the
// cluster spill layout.
constexpr size_t kGxHeaderBytes = 256;
constexpr int kGxMaxRowBlocks = 16384;
size_t gx_workspace_bytes(int64_t M, int64_t N);
fnorm_status_t gx_scratch_from(void* workspace, size_t bytes, int64_t M, int64_t N, GxScratch* out);

// The fixed workspace of fnorm_gemm_postnorm_noalloc (a device array, no
// allocation): address taken and counters cleared by the first call per
// device.  Calls sharing it must not overlap.
fnorm_status_t noalloc_scratch(cudaStream_t stream, const GxScratch** out);

struct FusedLaunch {
  const void* A;
  const void* B;
  void* C;
  int M, N, K;
  int mode;     // MODE_* bits of fused_gemm.cuh (cluster/spill/resident-B bits are set by the launcher)
  int bn;       // UMMA N of one accumulator tile (64..256, multiple of 64)
  int slices;   // spill layout: BN-column slices per CTA and row block, else 1
  bool spill;   // post-norm spill layout (rows wider than the cluster's tensor memory)
  bool bres;    // all of B resident in shared memory (N <= bn, K <= 128 KB / (bn * 2), many row blocks)
  int cluster;  // CTAs per cluster along N (post-norm), else 1
  float eps, pre_eps;
  const void* gamma;
  const void* beta;
  float* mean_out;
  float* rstd_out;
  float* pre_rstd_out;
  const float* colsum;  // pre-norm with folded affine: column sums of the folded B (LayerNorm)
  const float* bias;    // pre-norm with folded affine: beta @ B, or NULL
  const void* R;        // residual [M, N] added before the post-norm, or NULL
  // backward: A may be an A^T source ([K, M] row-major) and B a B^T source
  // ([N, K] row-major), as the mode says
  const void* X;          // dgrad: [M, N] forward input combined in the epilogue
  const float* rowcoef;   // dgrad: [M] coefficients c = -rstd^2 (dC . C) / K
  const float* rstd_in;   // post-norm backward: [M] the forward's rstd (X is then the forward output)
  float* cpart;           // post-norm backward: [ceil(M/32)][2][N] column partials, or NULL
  const GxScratch* gx;    // grid-exchange post-norm's workspace
  cudaStream_t stream;
};

// instantiation sets (one translation unit each)
fnorm_status_t launch_fused_plain(const FusedLaunch& L);          // GEMM, Lazy Pre-Norm
fnorm_status_t launch_fused_post_single(const FusedLaunch& L);    // post-norm, one CTA per row block
fnorm_status_t launch_fused_post_cluster(const FusedLaunch& L);   // post-norm over a cluster
fnorm_status_t launch_fused_prenorm_affine(const FusedLaunch& L); // lazy pre-norm, affine folded into B
fnorm_status_t launch_fused_post_residual(const FusedLaunch& L);  // residual + post-norm, one CTA per row block
fnorm_status_t launch_fused_post_residual_cluster(const FusedLaunch& L);  // residual + post-norm over a cluster
fnorm_status_t launch_fused_backward(const FusedLaunch& L);       // backward of the Lazy Pre-RMSNorm GEMM
fnorm_status_t launch_fused_post_grid(const FusedLaunch& L);      // post-norm, grid-wide statistics exchange
fnorm_status_t launch_fused_pair(const FusedLaunch& L);           // GEMM, lazy pre-norms: two-CTA MMA (256-row tiles)
fnorm_status_t launch_fused_mcb(const FusedLaunch& L);            // GEMM, lazy pre-norms: B multicast over a 2-CTA cluster
fnorm_status_t launch_fused_mcb_grid(const FusedLaunch& L);       // grid-exchange post-norm, B multicast
fnorm_status_t launch_fused_norm_backward(const FusedLaunch& L);  // post-norm backward on the dC-producing GEMM

// B' = bf16(gamma_k * B[k, n]), colsum[n] = sum_k B'[k, n], bias[n] = sum_k beta_k * B[k, n]
fnorm_status_t launch_fold_prenorm_affine(const void* B, int K, int N, const void* gamma, const void* beta,
                                          void* B_folded, float* colsum, float* bias, cudaStream_t stream);

// R (optional, [M, N]) is added to X before the norm
fnorm_status_t launch_rownorm(const void* X, const void* R, void* Y, int M, int N, bool layernorm, const void* gamma,
                              const void* beta, float eps, float* mean_out, float* rstd_out,
                              cudaStream_t stream);

// backward row pass: dCs = bf16(rstd * dC) and coef[m] = -rstd^2 (dC . C)[m] / K
fnorm_status_t launch_backward_rows(const void* dC, const void* C, const float* rstd, void* dCs, float* coef, int M,
                                    int N, int K, cudaStream_t stream);
// post-norm backward: dH from dC and the forward output (h_hat = (C - beta) /
// gamma), and dgamma/dbeta through per-64-row partials in part[groups][2][N]
int postnorm_backward_groups(int M);
// dgamma[n] = sum_g part[g][0][n], dbeta[n] = sum_g part[g][1][n] over `groups`
// row groups, in a fixed order (either output may be NULL)
fnorm_status_t launch_column_sum(const float* part, int groups, int N, float* dgamma, float* dbeta,
                                 cudaStream_t stream);
fnorm_status_t launch_postnorm_backward_rows(const void* dC, const void* C, const void* gamma, const void* beta,
                                             const float* rstd, bool layernorm, void* dH, float* part, float* dgamma,
                                             float* dbeta, int M, int N, cudaStream_t stream);
// dX = rstd * dY - rstd^3 * X * sum(dY * X) / N per row (RMSNorm backward, no affine)
fnorm_status_t launch_rmsnorm_backward(const void* dY, const void* X, const float* rstd, void* dX, int M, int N,
                                       cudaStream_t stream);
fnorm_status_t launch_fused_transposed(const FusedLaunch& L);   // plain GEMM with A^T and/or B^T operands
fnorm_status_t launch_fused_transposed_mcb(const FusedLaunch& L);  // the same and the dgrad, B multicast

fnorm_status_t launch_wait_timeout_selftest(uint64_t limit_ns, cudaStream_t stream);
fnorm_status_t launch_cluster_shape_selftest(int cluster, cudaStream_t stream);

}  // namespace fnorm
