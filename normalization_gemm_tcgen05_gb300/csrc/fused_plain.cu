// fused_plain.cu — instantiations of the fused kernel for the plain GEMM and
// the Lazy Pre-RMSNorm GEMM (one CTA per 128 x BN tile, persistent).
#include "fused_launch.cuh"

namespace fnorm {

fnorm_status_t launch_fused_plain(const FusedLaunch& L) {
  const bool pre = (L.mode & MODE_PRE) != 0;
  if (L.nsub != 1 || (L.mode & ~MODE_PRE) != 0) {
    set_error("internal: unexpected plain-GEMM plan (mode %d, nsub %d)", L.mode, L.nsub);
    return FNORM_ERR_UNSUPPORTED;
  }
  switch (L.bn_sub) {
    case 64:  return pre ? launch_cfg<KCfg<64, 1, 64, MODE_PRE>>(L) : launch_cfg<KCfg<64, 1, 64, 0>>(L);
    case 128: return pre ? launch_cfg<KCfg<128, 1, 64, MODE_PRE>>(L) : launch_cfg<KCfg<128, 1, 64, 0>>(L);
    case 256: return pre ? launch_cfg<KCfg<256, 1, 64, MODE_PRE>>(L) : launch_cfg<KCfg<256, 1, 64, 0>>(L);
    default: break;
  }
  set_error("internal: no plain-GEMM kernel with tile width %d", L.bn_sub);
  return FNORM_ERR_UNSUPPORTED;
}

}  // namespace fnorm
