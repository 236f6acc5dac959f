// fused_post_single.cu — instantiations of the fused kernel for the epilogue
// post-norm when one CTA tile spans the whole row (N <= 256), with B streamed
// per k-block or resident in shared memory.
#include "fused_launch.cuh"

namespace fnorm {

static_assert(KCfg<128, MODE_POST | MODE_LN>::STAGES >= 5 && KCfg<64, MODE_POST | MODE_LN>::STAGES >= 8,
              "post-norm, narrow tiles");
static_assert(KCfg<256, MODE_POST | MODE_LN | MODE_PRE | MODE_BRES>::STAGES >= 4, "pre + post-norm, resident B");

namespace {
template <int BN, int X>
fnorm_status_t by_mode_x(const FusedLaunch& L) {
  switch (L.mode) {
    case MODE_POST:                      return launch_cfg<KCfg<BN, MODE_POST | X>>(L);
    case MODE_POST | MODE_LN:            return launch_cfg<KCfg<BN, MODE_POST | MODE_LN | X>>(L);
    case MODE_POST | MODE_PRE:           return launch_cfg<KCfg<BN, MODE_POST | MODE_PRE | X>>(L);
    case MODE_POST | MODE_LN | MODE_PRE: return launch_cfg<KCfg<BN, MODE_POST | MODE_LN | MODE_PRE | X>>(L);
    default: break;
  }
  set_error("internal: unexpected post-norm mode %d", L.mode);
  return FNORM_ERR_UNSUPPORTED;
}

template <int BN>
fnorm_status_t by_mode(const FusedLaunch& L) {
  return L.bres ? by_mode_x<BN, MODE_BRES>(L) : by_mode_x<BN, 0>(L);
}
}  // namespace

fnorm_status_t launch_fused_post_single(const FusedLaunch& L) {
  if (L.cluster != 1 || L.spill) {
    set_error("internal: unexpected single-CTA post-norm plan");
    return FNORM_ERR_UNSUPPORTED;
  }
  switch (L.bn) {
    case 64:  return by_mode<64>(L);
    case 128: return by_mode<128>(L);
    case 192: return by_mode<192>(L);
    case 256: return by_mode<256>(L);
    default: break;
  }
  set_error("internal: no single-CTA post-norm kernel with tile width %d", L.bn);
  return FNORM_ERR_UNSUPPORTED;
}

}  // namespace fnorm
