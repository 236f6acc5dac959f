// fused_post_single.cu — instantiations of the fused kernel for the epilogue
// post-norm when one CTA tile spans the whole row (N <= 256).
#include "fused_launch.cuh"

namespace fnorm {

namespace {
template <int BN>
fnorm_status_t by_mode(const FusedLaunch& L) {
  switch (L.mode) {
    case MODE_POST:                      return launch_cfg<KCfg<BN, 1, 64, MODE_POST>>(L);
    case MODE_POST | MODE_LN:            return launch_cfg<KCfg<BN, 1, 64, MODE_POST | MODE_LN>>(L);
    case MODE_POST | MODE_PRE:           return launch_cfg<KCfg<BN, 1, 64, MODE_POST | MODE_PRE>>(L);
    case MODE_POST | MODE_LN | MODE_PRE: return launch_cfg<KCfg<BN, 1, 64, MODE_POST | MODE_LN | MODE_PRE>>(L);
    default: break;
  }
  set_error("internal: unexpected post-norm mode %d", L.mode);
  return FNORM_ERR_UNSUPPORTED;
}
}  // namespace

fnorm_status_t launch_fused_post_single(const FusedLaunch& L) {
  if (L.nsub != 1 || L.cluster != 1) {
    set_error("internal: unexpected single-CTA post-norm plan");
    return FNORM_ERR_UNSUPPORTED;
  }
  switch (L.bn_sub) {
    case 64:  return by_mode<64>(L);
    case 128: return by_mode<128>(L);
    case 192: return by_mode<192>(L);
    case 256: return by_mode<256>(L);
    default: break;
  }
  set_error("internal: no single-CTA post-norm kernel with tile width %d", L.bn_sub);
  return FNORM_ERR_UNSUPPORTED;
}

}  // namespace fnorm
