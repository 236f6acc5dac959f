// rownorm.cu — standalone row RMSNorm / LayerNorm, optionally of X + R (the
// unfused comparison kernels).  [ATB] sections 1.1 (LayerNorm) and 1.2
// (RMSNorm); [FNF-ru] FAQ: a standalone norm reads and writes the whole tensor
// and stays memory-bound; [FNF-ru] "FlashNormAttention" for the residual add.
//
// Memory-bound single pass from registers: a group of `tpr` threads (a power
// of two) owns one row; each thread loads up to VPT 16-byte vectors of it,
// the group reduces with warp shuffles (and shared memory when the group is
// wider than a warp), LayerNorm takes the variance as a second pass over the
// registers, then the row is normalised and written with 16-byte stores.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace fnorm {

namespace {

constexpr int kVPT = 4;  // 16-byte vectors per thread: 32 elements

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// sum over the `tpr` threads of this thread's group (groups are aligned)
__device__ __forceinline__ float group_sum(float v, int tpr, float* red) {
  const int w = tpr < 32 ? tpr : 32;
  for (int o = w >> 1; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (tpr <= 32) return v;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();  // earlier readers of red[] are done
  if (lane == 0) red[warp] = v;
  __syncthreads();
  const int nw = tpr >> 5;
  const int w0 = (static_cast<int>(threadIdx.x) / tpr) * nw;
  float s = 0.0f;
  for (int i = 0; i < nw; ++i) s += red[w0 + i];
  return s;
}

template <bool LN, bool RESID>
__global__ void __launch_bounds__(1024) rownorm_kernel(const __nv_bfloat16* __restrict__ X,
                                                       const __nv_bfloat16* __restrict__ R,
                                                       __nv_bfloat16* __restrict__ Y, int M, int N, int tpr,
                                                       const __nv_bfloat16* __restrict__ gamma,
                                                       const __nv_bfloat16* __restrict__ beta, float eps,
                                                       float* __restrict__ mean_out,
                                                       float* __restrict__ rstd_out) {
  __shared__ float red[32];
  grid_dependency_wait();  // launched with programmatic serialisation: inputs are ready after this
  if (threadIdx.x == 0) grid_launch_dependents();
  const int rpb = blockDim.x / tpr;
  const int row = blockIdx.x * rpb + static_cast<int>(threadIdx.x) / tpr;
  const int t = static_cast<int>(threadIdx.x) % tpr;
  const int nvec = N >> 3;
  const bool row_ok = row < M;
  const __nv_bfloat16* xr = X + static_cast<size_t>(row_ok ? row : 0) * N;
  const __nv_bfloat16* rr = RESID ? R + static_cast<size_t>(row_ok ? row : 0) * N : nullptr;

  float x[kVPT * 8];
#pragma unroll
  for (int i = 0; i < kVPT; ++i) {
    const int vi = t + i * tpr;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (row_ok && vi < nvec) v = ld_stream(xr + vi * 8);
    x[i * 8 + 0] = bf16_lo(v.x); x[i * 8 + 1] = bf16_hi(v.x);
    x[i * 8 + 2] = bf16_lo(v.y); x[i * 8 + 3] = bf16_hi(v.y);
    x[i * 8 + 4] = bf16_lo(v.z); x[i * 8 + 5] = bf16_hi(v.z);
    x[i * 8 + 6] = bf16_lo(v.w); x[i * 8 + 7] = bf16_hi(v.w);
    if (RESID) {  // residual: the row normalised is x + r, summed in fp32
      uint4 u = make_uint4(0, 0, 0, 0);
      if (row_ok && vi < nvec) u = ld_stream(rr + vi * 8);
      x[i * 8 + 0] += bf16_lo(u.x); x[i * 8 + 1] += bf16_hi(u.x);
      x[i * 8 + 2] += bf16_lo(u.y); x[i * 8 + 3] += bf16_hi(u.y);
      x[i * 8 + 4] += bf16_lo(u.z); x[i * 8 + 5] += bf16_hi(u.z);
      x[i * 8 + 6] += bf16_lo(u.w); x[i * 8 + 7] += bf16_hi(u.w);
    }
  }
  const float inv_n = 1.0f / static_cast<float>(N);
  float mean = 0.0f, rstd;
  if (LN) {
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < kVPT * 8; ++j) s += x[j];
    mean = group_sum(s, tpr, red) * inv_n;
    float q = 0.0f;
#pragma unroll
    for (int i = 0; i < kVPT; ++i) {
      const bool ok = (t + i * tpr) < nvec;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float d = x[i * 8 + j] - mean;
        q += ok ? d * d : 0.0f;
      }
    }
    rstd = rsqrtf(group_sum(q, tpr, red) * inv_n + eps);
  } else {
    float q = 0.0f;
#pragma unroll
    for (int j = 0; j < kVPT * 8; ++j) q = fmaf(x[j], x[j], q);
    rstd = rsqrtf(group_sum(q, tpr, red) * inv_n + eps);
  }
  if (!row_ok) return;
  __nv_bfloat16* yr = Y + static_cast<size_t>(row) * N;
#pragma unroll
  for (int i = 0; i < kVPT; ++i) {
    const int vi = t + i * tpr;
    if (vi >= nvec) break;
    float g[8], b[8];
    if (gamma != nullptr) {
      const uint4 gv = *reinterpret_cast<const uint4*>(gamma + vi * 8);
      g[0] = bf16_lo(gv.x); g[1] = bf16_hi(gv.x); g[2] = bf16_lo(gv.y); g[3] = bf16_hi(gv.y);
      g[4] = bf16_lo(gv.z); g[5] = bf16_hi(gv.z); g[6] = bf16_lo(gv.w); g[7] = bf16_hi(gv.w);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) g[j] = 1.0f;
    }
    if (beta != nullptr) {
      const uint4 bv = *reinterpret_cast<const uint4*>(beta + vi * 8);
      b[0] = bf16_lo(bv.x); b[1] = bf16_hi(bv.x); b[2] = bf16_lo(bv.y); b[3] = bf16_hi(bv.y);
      b[4] = bf16_lo(bv.z); b[5] = bf16_hi(bv.z); b[6] = bf16_lo(bv.w); b[7] = bf16_hi(bv.w);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) b[j] = 0.0f;
    }
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
      const float y0 = (x[i * 8 + j] - mean) * rstd * g[j] + b[j];
      const float y1 = (x[i * 8 + j + 1] - mean) * rstd * g[j + 1] + b[j + 1];
      w[j >> 1] = pack_bf16x2(y0, y1);
    }
    *reinterpret_cast<uint4*>(yr + vi * 8) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  if (t == 0) {
    if (LN && mean_out != nullptr) mean_out[row] = mean;
    if (rstd_out != nullptr) rstd_out[row] = rstd;
  }
}

}  // namespace

fnorm_status_t launch_rownorm(const void* X, const void* R, void* Y, int M, int N, bool layernorm, const void* gamma,
                              const void* beta, float eps, float* mean_out, float* rstd_out,
                              cudaStream_t stream) {
  DeviceInfo dev;
  fnorm_status_t st = current_device(&dev);
  if (st != FNORM_OK) return st;
  const int nvec = N / 8;
  const int need = (nvec + kVPT - 1) / kVPT;
  int tpr = 1;
  while (tpr < need) tpr <<= 1;
  if (tpr > 1024) {
    set_error("rows of %d elements exceed the standalone norm kernel's %d", N, 1024 * kVPT * 8);
    return FNORM_ERR_UNSUPPORTED;
  }
  const int block = tpr > 256 ? tpr : 256;
  const int rpb = block / tpr;
  const int grid = (M + rpb - 1) / rpb;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3((unsigned)block, 1, 1);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 0;
  if (pdl_enabled()) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 1;
  }
  const auto* x = static_cast<const __nv_bfloat16*>(X);
  const auto* r = static_cast<const __nv_bfloat16*>(R);
  auto* y = static_cast<__nv_bfloat16*>(Y);
  const auto* g = static_cast<const __nv_bfloat16*>(gamma);
  const auto* b = static_cast<const __nv_bfloat16*>(beta);
  auto kern = layernorm ? (r != nullptr ? rownorm_kernel<true, true> : rownorm_kernel<true, false>)
                        : (r != nullptr ? rownorm_kernel<false, true> : rownorm_kernel<false, false>);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, x, r, y, M, N, tpr, g, b, eps, mean_out, rstd_out);
  if (e != cudaSuccess) return cuda_fail(e, "row norm launch");
  return FNORM_OK;
}

}  // namespace fnorm
