// fused_post_residual.cu — instantiations of the fused kernel for the
// residual-add post-norm, C = norm(A @ B + R) * gamma + beta, when one CTA
// tile spans the whole row (N <= 256), with B streamed or resident.
#include "fused_launch.cuh"

namespace fnorm {

namespace {
template <int BN, int X>
fnorm_status_t by_mode_x(const FusedLaunch& L) {
  switch (L.mode) {
    case MODE_POST | MODE_RES:           return launch_cfg<KCfg<BN, MODE_POST | MODE_RES | X>>(L);
    case MODE_POST | MODE_LN | MODE_RES: return launch_cfg<KCfg<BN, MODE_POST | MODE_LN | MODE_RES | X>>(L);
    default: break;
  }
  set_error("internal: unexpected residual post-norm mode %d", L.mode);
  return FNORM_ERR_UNSUPPORTED;
}

template <int BN>
fnorm_status_t by_mode(const FusedLaunch& L) {
  return L.bres ? by_mode_x<BN, MODE_BRES>(L) : by_mode_x<BN, 0>(L);
}
}  // namespace

fnorm_status_t launch_fused_post_residual(const FusedLaunch& L) {
  if (L.cluster != 1 || L.spill) {
    set_error("internal: unexpected single-CTA residual post-norm plan");
    return FNORM_ERR_UNSUPPORTED;
  }
  switch (L.bn) {
    case 64:  return by_mode<64>(L);
    case 128: return by_mode<128>(L);
    case 192: return by_mode<192>(L);
    case 256: return by_mode<256>(L);
    default: break;
  }
  set_error("internal: no single-CTA residual post-norm kernel with tile width %d", L.bn);
  return FNORM_ERR_UNSUPPORTED;
}

}  // namespace fnorm
