// fold.cu — folds a pre-norm's fixed elementwise affine into the weight of
// the GEMM it feeds, so that the lazy pre-norm kernel can apply it after the
// k-loop.  [ATB] section 6.4 (at inference gamma is fixed and can be folded
// into the weights of the following matmul); [FNF-ru] "Lazy Pre-Norm" limits
// (a per-column affine does not commute with the GEMM, so it cannot stay in
// the prologue).
//
//   B'[k, n]  = bf16(gamma_k * B[k, n])       (round to nearest even)
//   colsum[n] = sum_k B'[k, n]               (fp32, of the rounded values the
//                                              GEMM multiplies)
//   bias[n]   = sum_k beta_k * B[k, n]       (fp32)
//
// Memory-bound, one pass over B: a CTA owns 64 columns (eight 16-byte column
// groups) and strides 32 row lanes over K, so a warp reads four 128-byte row
// segments per step.  Partial sums are reduced over the row lanes through
// shared memory in a fixed order: the results are deterministic.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace fnorm {

namespace {

constexpr int kFoldCols = 64;                      // columns per CTA
constexpr int kFoldGroups = kFoldCols / 8;         // 16-byte groups per row segment
constexpr int kFoldLanes = 32;                     // row lanes
constexpr int kFoldThreads = kFoldGroups * kFoldLanes;

__global__ void __launch_bounds__(kFoldThreads) fold_kernel(const __nv_bfloat16* B, int K, int N,
                                                            const __nv_bfloat16* __restrict__ gamma,
                                                            const __nv_bfloat16* __restrict__ beta,
                                                            __nv_bfloat16* Bf, float* __restrict__ colsum,
                                                            float* __restrict__ bias) {
  __shared__ float red_cs[kFoldLanes][kFoldCols + 1];
  __shared__ float red_b[kFoldLanes][kFoldCols + 1];
  grid_dependency_wait();
  if (threadIdx.x == 0) grid_launch_dependents();
  const int grp = threadIdx.x % kFoldGroups;
  const int lane_k = threadIdx.x / kFoldGroups;
  const int n = blockIdx.x * kFoldCols + grp * 8;
  const bool col_ok = n < N;  // N is a multiple of 8: a group is wholly in or out
  float cs[8], bs[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) cs[j] = bs[j] = 0.0f;
  if (col_ok) {
    for (int k = lane_k; k < K; k += kFoldLanes) {
      const size_t off = static_cast<size_t>(k) * N + n;
      const uint4 v = *reinterpret_cast<const uint4*>(B + off);
      const float g = gamma != nullptr ? __bfloat162float(gamma[k]) : 1.0f;
      const float be = beta != nullptr ? __bfloat162float(beta[k]) : 0.0f;
      const uint32_t in[4] = {v.x, v.y, v.z, v.w};
      uint32_t out[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const float b0 = bf16_lo(in[h]), b1 = bf16_hi(in[h]);
        out[h] = pack_bf16x2(g * b0, g * b1);
        cs[2 * h] += bf16_lo(out[h]);
        cs[2 * h + 1] += bf16_hi(out[h]);
        bs[2 * h] = fmaf(be, b0, bs[2 * h]);
        bs[2 * h + 1] = fmaf(be, b1, bs[2 * h + 1]);
      }
      *reinterpret_cast<uint4*>(Bf + off) = make_uint4(out[0], out[1], out[2], out[3]);
    }
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    red_cs[lane_k][grp * 8 + j] = cs[j];
    red_b[lane_k][grp * 8 + j] = bs[j];
  }
  __syncthreads();
  if (threadIdx.x < kFoldCols) {
    const int c = threadIdx.x;
    const int col = blockIdx.x * kFoldCols + c;
    if (col < N) {
      float s = 0.0f, t = 0.0f;
      for (int l = 0; l < kFoldLanes; ++l) {
        s += red_cs[l][c];
        t += red_b[l][c];
      }
      if (colsum != nullptr) colsum[col] = s;
      if (bias != nullptr) bias[col] = t;
    }
  }
}

}  // namespace

fnorm_status_t launch_fold_prenorm_affine(const void* B, int K, int N, const void* gamma, const void* beta,
                                          void* B_folded, float* colsum, float* bias, cudaStream_t stream) {
  DeviceInfo dev;
  fnorm_status_t st = current_device(&dev);
  if (st != FNORM_OK) return st;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3((unsigned)((N + kFoldCols - 1) / kFoldCols), 1, 1);
  cfg.blockDim = dim3(kFoldThreads, 1, 1);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 0;
  if (pdl_enabled()) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 1;
  }
  const cudaError_t e = cudaLaunchKernelEx(
      &cfg, fold_kernel, static_cast<const __nv_bfloat16*>(B), K, N, static_cast<const __nv_bfloat16*>(gamma),
      static_cast<const __nv_bfloat16*>(beta), static_cast<__nv_bfloat16*>(B_folded), colsum, bias);
  if (e != cudaSuccess) return cuda_fail(e, "affine fold launch");
  return FNORM_OK;
}

}  // namespace fnorm
