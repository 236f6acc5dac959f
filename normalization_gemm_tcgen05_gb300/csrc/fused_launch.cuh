// fused_launch.cuh — host launch of one instantiation of fused_gemm_kernel:
// tensor maps, persistent grid sizing (one CTA per SM, or as many clusters as
// can be co-resident), cluster and programmatic-dependent-launch attributes.
#pragma once

#include <atomic>

#include "fused_gemm.cuh"
#include "internal.h"

namespace fnorm {

template <class Cfg>
fnorm_status_t launch_cfg(const FusedLaunch& L) {
  DeviceInfo dev;
  fnorm_status_t st = current_device(&dev);
  if (st != FNORM_OK) return st;
  auto kern = fused_gemm_kernel<Cfg>;

  static std::atomic<uint64_t> configured{0};  // one bit per device
  if (!((configured.load(std::memory_order_acquire) >> dev.id) & 1ull)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg::SMEM_BYTES);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(max dynamic shared memory)");
    configured.fetch_or(1ull << dev.id, std::memory_order_acq_rel);
  }
  if (Cfg::BRES && (L.N > Cfg::BN || (L.K + Cfg::BK - 1) / Cfg::BK > Cfg::KB_MAX)) {
    set_error("internal: resident-B kernel given N %d, K %d", L.N, L.K);
    return FNORM_ERR_UNSUPPORTED;
  }

  // A [M,K] in [128 x 64] boxes (A^T source [K,M]: [64 x 64] boxes); B [K,N]
  // in [64 x 64] boxes, MN-major for the MMA (B^T source [N,K]: [BN x 64]
  // boxes, K-major; with B multicast each CTA loads half of them, [BN/2 x 64]);
  // C [M,N] in [32 x 32] store boxes (64-byte rows)
  CUtensorMap ta, tb, tc;
  if (Cfg::AT)
    st = encode_tmap_bf16_2d(&ta, L.A, (uint64_t)L.M, (uint64_t)L.K, (uint64_t)L.M * 2, 64, Cfg::BK,
                             CU_TENSOR_MAP_SWIZZLE_128B);
  else
    st = encode_tmap_bf16_2d(&ta, L.A, (uint64_t)L.K, (uint64_t)L.M, (uint64_t)L.K * 2, Cfg::BK, Cfg::BM,
                             CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != FNORM_OK) return st;
  if (Cfg::BT)
    st = encode_tmap_bf16_2d(&tb, L.B, (uint64_t)L.K, (uint64_t)L.N, (uint64_t)L.K * 2, Cfg::BK,
                             Cfg::MCB ? Cfg::BN / 2 : Cfg::BN,
                             CU_TENSOR_MAP_SWIZZLE_128B);
  else
    st = encode_tmap_bf16_2d(&tb, L.B, (uint64_t)L.N, (uint64_t)L.K, (uint64_t)L.N * 2, 64, Cfg::BK,
                             CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != FNORM_OK) return st;
  st = encode_tmap_bf16_2d(&tc, L.C, (uint64_t)L.N, (uint64_t)L.M, (uint64_t)L.N * 2, 32, 32,
                           CU_TENSOR_MAP_SWIZZLE_64B);
  if (st != FNORM_OK) return st;
  // the residual R [M,N] in the same [32 x 32] boxes (read by the first tile
  // of the single-CTA residual layouts); otherwise unused
  CUtensorMap tr = tc;
  if (Cfg::RES) {
    st = encode_tmap_bf16_2d(&tr, L.R, (uint64_t)L.N, (uint64_t)L.M, (uint64_t)L.N * 2, 32, 32,
                             CU_TENSOR_MAP_SWIZZLE_64B);
    if (st != FNORM_OK) return st;
  }

  FusedParams p;
  p.M = L.M;
  p.N = L.N;
  p.K = L.K;
  p.cluster = Cfg::CLUSTER ? L.cluster : 1;
  p.slices = Cfg::SPILL ? L.slices : 1;
  p.wave = dev.num_sms / 2 > 0 ? dev.num_sms / 2 : 1;
  {
    // the backward GEMMs' L2 policy: none within one wave of tiles (no later
    // wave re-reads B); else A evict_first, and B evict_last where it fits
    // in half of L2
    const int64_t tiles = (static_cast<int64_t>(L.M) + Cfg::BM - 1) / Cfg::BM *
                          ((static_cast<int64_t>(L.N) + Cfg::BN - 1) / Cfg::BN);
    p.l2_hints = tiles <= dev.num_sms ? 0 : static_cast<int64_t>(L.K) * L.N * 2 <= (int64_t{64} << 20) ? 2 : 1;
  }
  p.eps = L.eps;
  p.pre_eps = L.pre_eps;
  p.gamma = static_cast<const __nv_bfloat16*>(L.gamma);
  p.beta = static_cast<const __nv_bfloat16*>(L.beta);
  p.C = static_cast<__nv_bfloat16*>(L.C);
  p.mean_out = L.mean_out;
  p.rstd_out = L.rstd_out;
  p.pre_rstd_out = L.pre_rstd_out;
  p.colsum = L.colsum;
  p.bias = L.bias;
  p.R = static_cast<const __nv_bfloat16*>(L.R);
  p.rowcoef = L.rowcoef;
  if (Cfg::GX) {
    const int units = ((L.M + Cfg::BM - 1) / Cfg::BM) * ((L.N + Cfg::BN - 1) / Cfg::BN);
    if (L.gx == nullptr || units > L.gx->units_cap || (L.M + Cfg::BM - 1) / Cfg::BM > L.gx->rowblocks_cap) {
      set_error("internal: grid-exchange workspace missing or too small");
      return FNORM_ERR_UNSUPPORTED;
    }
    p.gx_part = L.gx->part;
    p.gx_cnt = L.gx->cnt;
    p.gx_finish = L.gx->finish;
  }
  p.X = static_cast<const __nv_bfloat16*>(L.X);
  p.rstd_in = L.rstd_in;
  p.cpart = L.cpart;
  p.status = dev.status;
  p.wait_limit_ns = wait_limit_ns();

  const int C = p.cluster;
  const int num_m = (L.M + Cfg::RB - 1) / Cfg::RB;
  const int group_cols = Cfg::BN * p.slices * C;
  const int ngroups = (L.N + group_cols - 1) / group_cols;
  const long long total = (long long)num_m * ngroups;

  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[3];
  cfg.blockDim = dim3(Cfg::NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
  cfg.stream = L.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 0;
  // The grid exchange waits on other CTAs, so all of them must be resident at
  // once: the grid never exceeds what the device holds at a time (one CTA
  // per SM, or the co-resident clusters), and the launch is cooperative, so
  // that the driver starts it only when all of its CTAs fit, whatever runs
  // on other streams.  FNORM_PLAIN_GX_LAUNCH=1 makes the clustered form (B
  // multicast) a plain cluster launch with programmatic stream
  // serialisation: profilers replay a cooperative launch of clusters without
  // its clusters (the kernel then reports the mismatch and does nothing).  A
  // plain launch's CTAs are all resident once the kernels before it in the
  // stream have finished, unless work on other streams holds SMs.
  const bool coop = Cfg::GX && !(Cfg::PAIR && plain_cluster_grid_exchange());
  if (pdl_enabled() && !coop) {
    // the kernel's set-up may overlap the previous grid; its first global
    // access waits for that grid (griddepcontrol.wait)
    attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
    ++cfg.numAttrs;
  }
  if (coop) {
    attr[cfg.numAttrs].id = cudaLaunchAttributeCooperative;
    attr[cfg.numAttrs].val.cooperative = 1;
    ++cfg.numAttrs;
  }
  if (Cfg::CLUSTER || Cfg::PAIR) {
    // post-norm: C CTAs along N; two-CTA MMA and B multicast: the CTA pair of
    // each 256-row unit
    const int CL = Cfg::PAIR ? 2 : C;
    if (Cfg::CLUSTER && (C < 1 || C > Cfg::CLMAX)) {
      set_error("cluster size %d outside 1..%d for this kernel", C, Cfg::CLMAX);
      return FNORM_ERR_UNSUPPORTED;
    }
    cudaLaunchAttribute& ca = attr[cfg.numAttrs++];
    ca.id = cudaLaunchAttributeClusterDimension;
    ca.val.clusterDim.x = (unsigned)CL;
    ca.val.clusterDim.y = 1;
    ca.val.clusterDim.z = 1;
    // co-resident clusters, cached per device and cluster size
    static std::atomic<int> max_clusters[64][9];
    int mc = max_clusters[dev.id][CL].load(std::memory_order_relaxed);
    if (mc == 0) {
      cudaLaunchConfig_t q = cfg;  // occupancy query: the cluster attribute only
      q.gridDim = dim3((unsigned)CL, 1, 1);
      q.attrs = &ca;
      q.numAttrs = 1;
      cudaError_t e = cudaOccupancyMaxActiveClusters(&mc, (void*)kern, &q);
      if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveClusters");
      if (mc <= 0) {
        set_error("no cluster of %d CTAs (%u bytes of shared memory each) fits on this device", CL,
                  Cfg::SMEM_BYTES);
        return FNORM_ERR_UNSUPPORTED;
      }
      max_clusters[dev.id][CL].store(mc, std::memory_order_relaxed);
    }
    const long long nclusters = total < mc ? total : mc;
    if (Cfg::GX && ngroups > nclusters) {
      set_error("internal: a grid exchange over %d tiles per row needs as many clusters (%lld)", ngroups, nclusters);
      return FNORM_ERR_UNSUPPORTED;
    }
    cfg.gridDim = dim3((unsigned)(nclusters * CL), 1, 1);
  } else {
    const long long grid = total < dev.num_sms ? total : dev.num_sms;
    if (Cfg::GX && ngroups > grid) {
      // every tile of a row block must be able to publish while the others
      // wait: no CTA may hold two tiles of one row block
      set_error("internal: a grid exchange over %d tiles per row needs as many CTAs (grid %lld)", ngroups, grid);
      return FNORM_ERR_UNSUPPORTED;
    }
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
  }
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, ta, tb, tc, tr, p);
  if (e != cudaSuccess && Cfg::GX && Cfg::PAIR &&
      (e == cudaErrorNotSupported || e == cudaErrorInvalidValue || e == cudaErrorInvalidConfiguration ||
       e == cudaErrorCooperativeLaunchTooLarge)) {
    // a clustered grid exchange refused before anything ran: the caller
    // takes the one-CTA grid exchange
    (void)cudaGetLastError();
    set_error("clustered grid exchange not available: %s", cudaGetErrorString(e));
    return FNORM_ERR_UNSUPPORTED;
  }
  if (e != cudaSuccess) return cuda_fail(e, "fused GEMM launch");
  return FNORM_OK;
}

}  // namespace fnorm
