// rownorm.cu — standalone row RMSNorm / LayerNorm, optionally of X + R, and
// the RMSNorm backward (the unfused comparison kernels); the fused backward's
// row pass.  [ATB] sections 1.1 (LayerNorm) and 1.2
// (RMSNorm); [FNF-ru] FAQ: a standalone norm reads and writes the whole tensor
// and stays memory-bound; [FNF-ru] "FlashNormAttention" for the residual add.
//
// Memory-bound single pass from registers: a group of `tpr` threads (a power
// of two) owns one row; each thread loads up to VPT 16-byte vectors of it,
// the group reduces with warp shuffles (and shared memory when the group is
// wider than a warp), LayerNorm takes the variance as a second pass over the
// registers, then the row is normalised and written with 16-byte stores.
#include <cuda_bf16.h>

#include <atomic>

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

// Standalone RMSNorm backward (no affine), the unfused comparison of the
// fused backward: dX = rstd * dY - rstd^3 * X * sum_n(dY * X) / N per row, with
// the forward's rstd given.  Same row layout as rownorm_kernel: a group of tpr
// threads holds the row's dY and X in registers.
__global__ void __launch_bounds__(512) rmsnorm_bwd_kernel(const __nv_bfloat16* __restrict__ dY,
                                                           const __nv_bfloat16* __restrict__ X,
                                                           const float* __restrict__ rstd_in,
                                                           __nv_bfloat16* __restrict__ dX, int M, int N, int tpr) {
  __shared__ float red[32];
  grid_dependency_wait();
  if (threadIdx.x == 0) grid_launch_dependents();
  const int rpb = blockDim.x / tpr;
  const int row = blockIdx.x * rpb + static_cast<int>(threadIdx.x) / tpr;
  const int t = static_cast<int>(threadIdx.x) % tpr;
  const int nvec = N >> 3;
  const bool row_ok = row < M;
  const size_t off = static_cast<size_t>(row_ok ? row : 0) * N;
  uint32_t g[kVPT * 4], x[kVPT * 4];  // bf16 pairs, widened when used
#pragma unroll
  for (int i = 0; i < kVPT; ++i) {
    const int vi = t + i * tpr;
    uint4 u = make_uint4(0, 0, 0, 0), v = make_uint4(0, 0, 0, 0);
    if (row_ok && vi < nvec) {
      u = ld_stream(dY + off + vi * 8);
      v = ld_stream(X + off + vi * 8);
    }
    g[i * 4] = u.x; g[i * 4 + 1] = u.y; g[i * 4 + 2] = u.z; g[i * 4 + 3] = u.w;
    x[i * 4] = v.x; x[i * 4 + 1] = v.y; x[i * 4 + 2] = v.z; x[i * 4 + 3] = v.w;
  }
  float q = 0.0f;
#pragma unroll
  for (int j = 0; j < kVPT * 4; ++j) {
    q = fmaf(bf16_lo(g[j]), bf16_lo(x[j]), q);
    q = fmaf(bf16_hi(g[j]), bf16_hi(x[j]), q);
  }
  const float dot = group_sum(q, tpr, red);
  if (!row_ok) return;
  const float r = rstd_in[row];
  const float c = -r * r * r * dot / static_cast<float>(N);
#pragma unroll
  for (int i = 0; i < kVPT; ++i) {
    const int vi = t + i * tpr;
    if (vi >= nvec) break;
    uint32_t w[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const uint32_t gg = g[i * 4 + h], xx = x[i * 4 + h];
      w[h] = pack_bf16x2(fmaf(bf16_lo(gg), r, c * bf16_lo(xx)), fmaf(bf16_hi(gg), r, c * bf16_hi(xx)));
    }
    *reinterpret_cast<uint4*>(dX + off + vi * 8) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// The backward's row pass over dC and the forward output C, one read of each:
//   dCs[m,n] = bf16(rstd[m] * dC[m,n])       (the rebuilt scale, on dC's side)
//   coef[m]  = -rstd[m]^2 * sum_n dC[m,n] C[m,n] / K
// A group of tpr threads per row, 16-byte loads and stores.
__global__ void __launch_bounds__(256) backward_rows_kernel(const __nv_bfloat16* __restrict__ dC,
                                                            const __nv_bfloat16* __restrict__ C,
                                                            const float* __restrict__ rstd,
                                                            __nv_bfloat16* __restrict__ dCs, float* __restrict__ coef,
                                                            int M, int N, int K, int tpr) {
  __shared__ float red[32];
  grid_dependency_wait();
  if (threadIdx.x == 0) grid_launch_dependents();
  const int rpb = blockDim.x / tpr;
  const int row = blockIdx.x * rpb + static_cast<int>(threadIdx.x) / tpr;
  const int t = static_cast<int>(threadIdx.x) % tpr;
  const int nvec = N >> 3;
  const bool row_ok = row < M;
  const size_t off = static_cast<size_t>(row_ok ? row : 0) * N;
  const float r = row_ok ? rstd[row] : 0.0f;
  float q = 0.0f;
  for (int vi = t; vi < nvec; vi += tpr) {
    uint4 u = make_uint4(0, 0, 0, 0), v = make_uint4(0, 0, 0, 0);
    if (row_ok) {
      u = ld_stream(dC + off + vi * 8);
      v = ld_stream(C + off + vi * 8);
    }
    const uint32_t uw[4] = {u.x, u.y, u.z, u.w}, vw[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      q = fmaf(bf16_lo(uw[h]), bf16_lo(vw[h]), q);
      q = fmaf(bf16_hi(uw[h]), bf16_hi(vw[h]), q);
      o[h] = pack_bf16x2(bf16_lo(uw[h]) * r, bf16_hi(uw[h]) * r);
    }
    if (row_ok) *reinterpret_cast<uint4*>(dCs + off + vi * 8) = make_uint4(o[0], o[1], o[2], o[3]);
  }
  const float s = group_sum(q, tpr, red);
  if (row_ok && t == 0) coef[row] = -r * r * s / static_cast<float>(K);
}

// Post-norm backward.  The forward's normalised rows are rebuilt from its
// output: h_hat = (C - beta) / gamma (gamma != 0).  With dh = dC * gamma:
//   LayerNorm: dH = rstd * (dh - mean_n(dh) - h_hat * mean_n(dh * h_hat))
//   RMSNorm:   dH = rstd * (dh - h_hat * mean_n(dh * h_hat))
//   dgamma = sum_m dC * h_hat,   dbeta = sum_m dC.
// Row pass: one warp per row, two sweeps over the row (sums, then dH; the
// second sweep reads from L2), 16-byte loads, any N.  The first sweep's
// dh * h_hat is dC * (C - beta), with no division; the second multiplies by
// correctly rounded reciprocals of gamma instead of dividing by it.
constexpr int kRowsPerBlock = 8;

__device__ __forceinline__ float bf16_at(const uint4& v, int e) {
  const uint32_t w = e < 2 ? v.x : e < 4 ? v.y : e < 6 ? v.z : v.w;
  return (e & 1) ? bf16_hi(w) : bf16_lo(w);
}

template <bool LN>
__global__ void __launch_bounds__(32 * kRowsPerBlock) postnorm_bwd_rows_kernel(
    const __nv_bfloat16* __restrict__ dC, const __nv_bfloat16* __restrict__ C, const __nv_bfloat16* __restrict__ gamma,
    const __nv_bfloat16* __restrict__ beta, const float* __restrict__ rstd_in, __nv_bfloat16* __restrict__ dH, int M,
    int N) {
  grid_dependency_wait();
  if (threadIdx.x == 0) grid_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * kRowsPerBlock + warp;
  if (row >= M) return;
  const int nvec = N >> 3;
  const size_t off = static_cast<size_t>(row) * N;
  const float r = rstd_in[row];
  float s1 = 0.0f, s2 = 0.0f;
  for (int vi = lane; vi < nvec; vi += 32) {
    const uint4 u = ld_stream(dC + off + vi * 8), v = *reinterpret_cast<const uint4*>(C + off + vi * 8);
    uint4 g = make_uint4(0x3f803f80u, 0x3f803f80u, 0x3f803f80u, 0x3f803f80u), b = make_uint4(0, 0, 0, 0);
    if (gamma != nullptr) g = *reinterpret_cast<const uint4*>(gamma + vi * 8);
    if (beta != nullptr) b = *reinterpret_cast<const uint4*>(beta + vi * 8);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float du = bf16_at(u, e);
      s1 = fmaf(du, bf16_at(g, e), s1);
      s2 = fmaf(du, bf16_at(v, e) - bf16_at(b, e), s2);  // (dC * gamma) * (C - beta) / gamma
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    s1 += __shfl_xor_sync(0xffffffffu, s1, o);
    s2 += __shfl_xor_sync(0xffffffffu, s2, o);
  }
  const float inv_n = 1.0f / static_cast<float>(N);
  const float m1 = LN ? s1 * inv_n : 0.0f, m2 = s2 * inv_n;
  for (int vi = lane; vi < nvec; vi += 32) {
    const uint4 u = *reinterpret_cast<const uint4*>(dC + off + vi * 8);
    const uint4 v = *reinterpret_cast<const uint4*>(C + off + vi * 8);
    uint4 g = make_uint4(0x3f803f80u, 0x3f803f80u, 0x3f803f80u, 0x3f803f80u), b = make_uint4(0, 0, 0, 0);
    if (gamma != nullptr) g = *reinterpret_cast<const uint4*>(gamma + vi * 8);
    if (beta != nullptr) b = *reinterpret_cast<const uint4*>(beta + vi * 8);
    uint32_t o[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      float y[2];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int e = 2 * h + q;
        const float gm = bf16_at(g, e);
        const float hat = (bf16_at(v, e) - bf16_at(b, e)) * __frcp_rn(gm);
        y[q] = r * (bf16_at(u, e) * gm - m1 - hat * m2);
      }
      o[h] = pack_bf16x2(y[0], y[1]);
    }
    *reinterpret_cast<uint4*>(dH + off + vi * 8) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// Column pass: thread t owns 8 adjacent columns and walks kColRows rows,
// accumulating dC * h_hat and dC; part[group][0][n], part[group][1][n].
constexpr int kColRows = 64;

__global__ void __launch_bounds__(256) postnorm_bwd_cols_kernel(const __nv_bfloat16* __restrict__ dC,
                                                                const __nv_bfloat16* __restrict__ C,
                                                                const __nv_bfloat16* __restrict__ gamma,
                                                                const __nv_bfloat16* __restrict__ beta,
                                                                float* __restrict__ part, int M, int N) {
  grid_dependency_wait();
  if (threadIdx.x == 0) grid_launch_dependents();
  const int vi = blockIdx.x * blockDim.x + threadIdx.x;  // 8-column group
  const int grp = blockIdx.y;                            // 64-row group
  if (vi >= (N >> 3)) return;
  uint4 g = make_uint4(0x3f803f80u, 0x3f803f80u, 0x3f803f80u, 0x3f803f80u), b = make_uint4(0, 0, 0, 0);
  if (gamma != nullptr) g = *reinterpret_cast<const uint4*>(gamma + vi * 8);
  if (beta != nullptr) b = *reinterpret_cast<const uint4*>(beta + vi * 8);
  float ig[8], bt[8], ag[8], ab[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    ig[e] = __frcp_rn(bf16_at(g, e));
    bt[e] = bf16_at(b, e);
    ag[e] = ab[e] = 0.0f;
  }
  const int m_end = min(M, (grp + 1) * kColRows);
  constexpr int kU = 8;  // rows of loads in flight
  for (int m0 = grp * kColRows; m0 < m_end; m0 += kU) {
    uint4 u[kU], v[kU];
#pragma unroll
    for (int k = 0; k < kU; ++k) {
      u[k] = v[k] = make_uint4(0, 0, 0, 0);  // rows past M add zero
      if (m0 + k < m_end) {
        const size_t o = static_cast<size_t>(m0 + k) * N + vi * 8;
        u[k] = ld_stream(dC + o);
        v[k] = ld_stream(C + o);
      }
    }
#pragma unroll
    for (int k = 0; k < kU; ++k)
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float dc = bf16_at(u[k], e);
        ag[e] = fmaf(dc, (bf16_at(v[k], e) - bt[e]) * ig[e], ag[e]);
        ab[e] += dc;
      }
  }
  float* pg = part + static_cast<size_t>(grp) * 2 * N + vi * 8;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    pg[e] = ag[e];
    pg[N + e] = ab[e];
  }
}

// Row and column passes in one (N <= 1024, both wanted).  A block takes one
// kColRows-row group and a warp every kRowsPerBlock-th row of it; a lane keeps
// its columns' dC and C of the current row in registers between the two
// sweeps (each read once), and adds its columns' dgamma/dbeta contributions
// into its warp's own slice of shared memory.  The block then sums the
// warps' slices in warp order into part[group] (the column pass's layout).
template <bool LN, int VPL>
__global__ void __launch_bounds__(32 * kRowsPerBlock, 2) postnorm_bwd_fused_kernel(
    const __nv_bfloat16* __restrict__ dC, const __nv_bfloat16* __restrict__ C, const __nv_bfloat16* __restrict__ gamma,
    const __nv_bfloat16* __restrict__ beta, const float* __restrict__ rstd_in, __nv_bfloat16* __restrict__ dH,
    float* __restrict__ part, int M, int N) {
  extern __shared__ float red[];  // [kRowsPerBlock][2][N]
  grid_dependency_wait();
  if (threadIdx.x == 0) grid_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = blockIdx.x;
  const int nvec = N >> 3;
  float* pw = red + static_cast<size_t>(warp) * 2 * N;
  for (int n = lane; n < 2 * N; n += 32) pw[n] = 0.0f;
  __syncwarp();
  // gamma and beta of this lane's columns, re-read each row through the
  // read-only cache rather than held in registers
  auto gb = [&](int j, uint4& g, uint4& b) {
    const int vi = lane + 32 * j;
    g = make_uint4(0x3f803f80u, 0x3f803f80u, 0x3f803f80u, 0x3f803f80u);
    b = make_uint4(0, 0, 0, 0);
    if (vi < nvec && gamma != nullptr) g = __ldg(reinterpret_cast<const uint4*>(gamma + vi * 8));
    if (vi < nvec && beta != nullptr) b = __ldg(reinterpret_cast<const uint4*>(beta + vi * 8));
  };
  const float inv_n = 1.0f / static_cast<float>(N);
  for (int i = warp; i < kColRows; i += kRowsPerBlock) {
    const int row = grp * kColRows + i;
    if (row >= M) break;
    const size_t off = static_cast<size_t>(row) * N;
    uint4 u[VPL], v[VPL];
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      const int vi = lane + 32 * j;
      u[j] = v[j] = make_uint4(0, 0, 0, 0);  // columns past N add zero
      if (vi < nvec) {
        u[j] = ld_stream(dC + off + vi * 8);
        v[j] = ld_stream(C + off + vi * 8);
      }
    }
    float s1 = 0.0f, s2 = 0.0f;
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      uint4 g, b;
      gb(j, g, b);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float du = bf16_at(u[j], e);
        s1 = fmaf(du, bf16_at(g, e), s1);
        s2 = fmaf(du, bf16_at(v[j], e) - bf16_at(b, e), s2);  // (dC * gamma) * (C - beta) / gamma
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      s1 += __shfl_xor_sync(0xffffffffu, s1, o);
      s2 += __shfl_xor_sync(0xffffffffu, s2, o);
    }
    const float r = rstd_in[row];
    const float m1 = LN ? s1 * inv_n : 0.0f, m2 = s2 * inv_n;
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      const int vi = lane + 32 * j;
      if (vi >= nvec) continue;
      uint4 g, b;
      gb(j, g, b);
      float hat[8];
      uint32_t o[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        float y[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int e = 2 * h + q;
          const float gm = bf16_at(g, e);
          hat[e] = (bf16_at(v[j], e) - bf16_at(b, e)) * __frcp_rn(gm);
          y[q] = r * (bf16_at(u[j], e) * gm - m1 - hat[e] * m2);
        }
        o[h] = pack_bf16x2(y[0], y[1]);
      }
      *reinterpret_cast<uint4*>(dH + off + vi * 8) = make_uint4(o[0], o[1], o[2], o[3]);
      float4* pg = reinterpret_cast<float4*>(pw + vi * 8);
      float4* pb = reinterpret_cast<float4*>(pw + N + vi * 8);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float4 ga = pg[hh], ba = pb[hh];
        ga.x = fmaf(bf16_at(u[j], 4 * hh), hat[4 * hh], ga.x);
        ga.y = fmaf(bf16_at(u[j], 4 * hh + 1), hat[4 * hh + 1], ga.y);
        ga.z = fmaf(bf16_at(u[j], 4 * hh + 2), hat[4 * hh + 2], ga.z);
        ga.w = fmaf(bf16_at(u[j], 4 * hh + 3), hat[4 * hh + 3], ga.w);
        ba.x += bf16_at(u[j], 4 * hh);
        ba.y += bf16_at(u[j], 4 * hh + 1);
        ba.z += bf16_at(u[j], 4 * hh + 2);
        ba.w += bf16_at(u[j], 4 * hh + 3);
        pg[hh] = ga;
        pb[hh] = ba;
      }
    }
  }
  __syncthreads();
  float* pgo = part + static_cast<size_t>(grp) * 2 * N;
  for (int n = threadIdx.x; n < 2 * N; n += blockDim.x) {
    float acc = 0.0f;
    for (int w = 0; w < kRowsPerBlock; ++w) acc += red[static_cast<size_t>(w) * 2 * N + n];
    pgo[n] = acc;
  }
}

// dgamma[n] = sum_g part[g][0][n], dbeta[n] = sum_g part[g][1][n].  A block
// takes kSumCols columns; each of its kSumRows thread rows sums every
// kSumRows-th group (loads coalesced along n, several in flight), and the
// rows' sums are then added in row order, so the result is the same on every
// run.
constexpr int kSumCols = 32, kSumRows = 32;

__global__ void __launch_bounds__(kSumCols * kSumRows) column_sum_kernel(const float* __restrict__ part, int ngroups,
                                                                         int N, float* __restrict__ dgamma,
                                                                         float* __restrict__ dbeta) {
  __shared__ float ra[kSumRows][kSumCols + 1], rb[kSumRows][kSumCols + 1];
  grid_dependency_wait();
  if (threadIdx.x == 0) grid_launch_dependents();
  const int tx = static_cast<int>(threadIdx.x) % kSumCols, ty = static_cast<int>(threadIdx.x) / kSumCols;
  const int n = blockIdx.x * kSumCols + tx;
  float a = 0.0f, b = 0.0f;
  if (n < N) {
#pragma unroll 4
    for (int k = ty; k < ngroups; k += kSumRows) {
      a += part[static_cast<size_t>(k) * 2 * N + n];
      b += part[static_cast<size_t>(k) * 2 * N + N + n];
    }
  }
  ra[ty][tx] = a;
  rb[ty][tx] = b;
  __syncthreads();
  if (ty == 0 && n < N) {
    float sa = 0.0f, sb = 0.0f;
    for (int r = 0; r < kSumRows; ++r) {
      sa += ra[r][tx];
      sb += rb[r][tx];
    }
    if (dgamma != nullptr) dgamma[n] = sa;
    if (dbeta != nullptr) dbeta[n] = sb;
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

fnorm_status_t launch_backward_rows(const void* dC, const void* C, const float* rstd, void* dCs, float* coef, int M,
                                    int N, int K, cudaStream_t stream) {
  DeviceInfo dev;
  fnorm_status_t st = current_device(&dev);
  if (st != FNORM_OK) return st;
  // a group of up to 256 threads per row, about four 16-byte vectors each
  const int nvec = N / 8;
  int tpr = 1;
  while (tpr < 256 && tpr * 4 < nvec) tpr <<= 1;
  const int block = 256;
  const int rpb = block / tpr;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3((unsigned)((M + rpb - 1) / rpb), 1, 1);
  cfg.blockDim = dim3((unsigned)block, 1, 1);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 0;
  if (pdl_enabled()) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 1;
  }
  const cudaError_t e = cudaLaunchKernelEx(&cfg, backward_rows_kernel, static_cast<const __nv_bfloat16*>(dC),
                                           static_cast<const __nv_bfloat16*>(C), rstd,
                                           static_cast<__nv_bfloat16*>(dCs), coef, M, N, K, tpr);
  if (e != cudaSuccess) return cuda_fail(e, "backward row pass launch");
  return FNORM_OK;
}

namespace {
cudaLaunchConfig_t small_cfg(dim3 grid, dim3 block, cudaStream_t stream, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 0;
  if (pdl_enabled()) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 1;
  }
  return cfg;
}
}  // namespace

int postnorm_backward_groups(int M) { return (M + kColRows - 1) / kColRows; }

namespace {
// the fused row and column pass: 64 N bytes of shared memory (opted in once
// per device, up to 64 KB at N = 1024)
template <bool LN, int VPL>
cudaError_t launch_postnorm_fused(cudaLaunchConfig_t& cfg, int dev_id, const __nv_bfloat16* dc,
                                  const __nv_bfloat16* c, const __nv_bfloat16* g, const __nv_bfloat16* b,
                                  const float* rstd, __nv_bfloat16* dh, float* part, int M, int N) {
  auto kern = postnorm_bwd_fused_kernel<LN, VPL>;
  static std::atomic<uint64_t> configured{0};  // one bit per device
  if (!((configured.load(std::memory_order_acquire) >> dev_id) & 1ull)) {
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 65536);
    if (e != cudaSuccess) return e;
    configured.fetch_or(1ull << dev_id, std::memory_order_acq_rel);
  }
  cfg.dynamicSmemBytes = static_cast<size_t>(kRowsPerBlock) * 2 * N * sizeof(float);
  return cudaLaunchKernelEx(&cfg, kern, dc, c, g, b, rstd, dh, part, M, N);
}
}  // namespace

fnorm_status_t launch_postnorm_backward_rows(const void* dC, const void* C, const void* gamma, const void* beta,
                                             const float* rstd, bool layernorm, void* dH, float* part, float* dgamma,
                                             float* dbeta, int M, int N, cudaStream_t stream) {
  DeviceInfo dev;
  fnorm_status_t st = current_device(&dev);
  if (st != FNORM_OK) return st;
  const auto* dc = static_cast<const __nv_bfloat16*>(dC);
  const auto* c = static_cast<const __nv_bfloat16*>(C);
  const auto* g = static_cast<const __nv_bfloat16*>(gamma);
  const auto* b = static_cast<const __nv_bfloat16*>(beta);
  cudaLaunchAttribute attr[1];
  const bool cols = dgamma != nullptr || dbeta != nullptr;
  if (dH != nullptr && cols && N <= 1024) {
    // both passes in one kernel (each row of dC and C read once), then the column sum
    const int groups = postnorm_backward_groups(M);
    const int vpl = (N / 8 + 31) / 32;
    cudaLaunchConfig_t cfg = small_cfg(dim3((unsigned)groups), dim3(32 * kRowsPerBlock), stream, attr);
    auto* dh = static_cast<__nv_bfloat16*>(dH);
    cudaError_t e;
    if (vpl <= 1)
      e = layernorm ? launch_postnorm_fused<true, 1>(cfg, dev.id, dc, c, g, b, rstd, dh, part, M, N)
                    : launch_postnorm_fused<false, 1>(cfg, dev.id, dc, c, g, b, rstd, dh, part, M, N);
    else if (vpl <= 2)
      e = layernorm ? launch_postnorm_fused<true, 2>(cfg, dev.id, dc, c, g, b, rstd, dh, part, M, N)
                    : launch_postnorm_fused<false, 2>(cfg, dev.id, dc, c, g, b, rstd, dh, part, M, N);
    else
      e = layernorm ? launch_postnorm_fused<true, 4>(cfg, dev.id, dc, c, g, b, rstd, dh, part, M, N)
                    : launch_postnorm_fused<false, 4>(cfg, dev.id, dc, c, g, b, rstd, dh, part, M, N);
    if (e != cudaSuccess) return cuda_fail(e, "post-norm backward row and column pass launch");
    cfg = small_cfg(dim3((unsigned)((N + kSumCols - 1) / kSumCols)), dim3(kSumCols * kSumRows), stream, attr);
    e = cudaLaunchKernelEx(&cfg, column_sum_kernel, static_cast<const float*>(part), groups, N, dgamma, dbeta);
    if (e != cudaSuccess) return cuda_fail(e, "column sum launch");
    return FNORM_OK;
  }
  if (dH != nullptr) {
    cudaLaunchConfig_t cfg =
        small_cfg(dim3((unsigned)((M + kRowsPerBlock - 1) / kRowsPerBlock)), dim3(32 * kRowsPerBlock), stream, attr);
    const cudaError_t e =
        layernorm ? cudaLaunchKernelEx(&cfg, postnorm_bwd_rows_kernel<true>, dc, c, g, b, rstd,
                                       static_cast<__nv_bfloat16*>(dH), M, N)
                  : cudaLaunchKernelEx(&cfg, postnorm_bwd_rows_kernel<false>, dc, c, g, b, rstd,
                                       static_cast<__nv_bfloat16*>(dH), M, N);
    if (e != cudaSuccess) return cuda_fail(e, "post-norm backward row pass launch");
  }
  if (cols) {
    const int groups = postnorm_backward_groups(M);
    cudaLaunchConfig_t cfg = small_cfg(dim3((unsigned)((N / 8 + 255) / 256), (unsigned)groups), dim3(256), stream, attr);
    cudaError_t e = cudaLaunchKernelEx(&cfg, postnorm_bwd_cols_kernel, dc, c, g, b, part, M, N);
    if (e != cudaSuccess) return cuda_fail(e, "post-norm backward column pass launch");
    cfg = small_cfg(dim3((unsigned)((N + kSumCols - 1) / kSumCols)), dim3(kSumCols * kSumRows), stream, attr);
    e = cudaLaunchKernelEx(&cfg, column_sum_kernel, static_cast<const float*>(part), groups, N, dgamma, dbeta);
    if (e != cudaSuccess) return cuda_fail(e, "column sum launch");
  }
  return FNORM_OK;
}

fnorm_status_t launch_column_sum(const float* part, int groups, int N, float* dgamma, float* dbeta,
                                 cudaStream_t stream) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg =
      small_cfg(dim3((unsigned)((N + kSumCols - 1) / kSumCols)), dim3(kSumCols * kSumRows), stream, attr);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, column_sum_kernel, part, groups, N, dgamma, dbeta);
  if (e != cudaSuccess) return cuda_fail(e, "column sum launch");
  return FNORM_OK;
}

fnorm_status_t launch_rmsnorm_backward(const void* dY, const void* X, const float* rstd, void* dX, int M, int N,
                                       cudaStream_t stream) {
  DeviceInfo dev;
  fnorm_status_t st = current_device(&dev);
  if (st != FNORM_OK) return st;
  const int nvec = N / 8;
  const int need = (nvec + kVPT - 1) / kVPT;
  int tpr = 1;
  while (tpr < need) tpr <<= 1;
  if (tpr > 512) {  // two row slices in registers: 512 threads a row at most
    set_error("rows of %d elements exceed the RMSNorm backward kernel's %d", N, 512 * kVPT * 8);
    return FNORM_ERR_UNSUPPORTED;
  }
  const int block = tpr > 256 ? tpr : 256;
  const int rpb = block / tpr;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3((unsigned)((M + rpb - 1) / rpb), 1, 1);
  cfg.blockDim = dim3((unsigned)block, 1, 1);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 0;
  if (pdl_enabled()) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 1;
  }
  const cudaError_t e = cudaLaunchKernelEx(&cfg, rmsnorm_bwd_kernel, static_cast<const __nv_bfloat16*>(dY),
                                           static_cast<const __nv_bfloat16*>(X), rstd,
                                           static_cast<__nv_bfloat16*>(dX), M, N, tpr);
  if (e != cudaSuccess) return cuda_fail(e, "RMSNorm backward launch");
  return FNORM_OK;
}

}  // namespace fnorm
