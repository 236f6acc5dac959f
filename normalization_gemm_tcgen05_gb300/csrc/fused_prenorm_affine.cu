// fused_prenorm_affine.cu — instantiations of the fused kernel for the lazy
// pre-norm with its elementwise affine folded into B: RMSNorm with a bias row,
// or LayerNorm with the mean removed by a column-sum correction (one CTA per
// 128 x BN tile, persistent; B streamed per k-block or resident).
#include "fused_launch.cuh"

namespace fnorm {

static_assert(KCfg<256, MODE_PRE | MODE_PRE_LN | MODE_AFF>::STAGES >= 4, "pre-LayerNorm, 256-column tiles");

namespace {
template <int BN, int X>
fnorm_status_t by_mode_x(const FusedLaunch& L) {
  switch (L.mode) {
    case MODE_PRE | MODE_AFF:               return launch_cfg<KCfg<BN, MODE_PRE | MODE_AFF | X>>(L);
    case MODE_PRE | MODE_PRE_LN | MODE_AFF: return launch_cfg<KCfg<BN, MODE_PRE | MODE_PRE_LN | MODE_AFF | X>>(L);
    default: break;
  }
  set_error("internal: unexpected folded-affine pre-norm mode %d", L.mode);
  return FNORM_ERR_UNSUPPORTED;
}

template <int BN>
fnorm_status_t by_mode(const FusedLaunch& L) {
  return L.bres ? by_mode_x<BN, MODE_BRES>(L) : by_mode_x<BN, 0>(L);
}
}  // namespace

fnorm_status_t launch_fused_prenorm_affine(const FusedLaunch& L) {
  if (L.spill || L.cluster != 1) {
    set_error("internal: unexpected folded-affine pre-norm plan");
    return FNORM_ERR_UNSUPPORTED;
  }
  switch (L.bn) {
    case 64:  return by_mode<64>(L);
    case 128: return by_mode<128>(L);
    case 256: return by_mode<256>(L);
    default: break;
  }
  set_error("internal: no folded-affine pre-norm kernel with tile width %d", L.bn);
  return FNORM_ERR_UNSUPPORTED;
}

}  // namespace fnorm
