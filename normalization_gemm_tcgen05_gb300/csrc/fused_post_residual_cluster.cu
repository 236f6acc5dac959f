// fused_post_residual_cluster.cu — instantiations of the fused kernel for the
// residual-add post-norm with rows split over a thread-block cluster along N
// (resident slices of 128 or 256 columns, or the spill layout for wider rows).
#include "fused_launch.cuh"

namespace fnorm {

static_assert(KCfg<256, MODE_POST | MODE_CLUSTER | MODE_RES, 4>::STAGES >= 4, "resident cluster ring");
static_assert(KCfg<256, MODE_POST | MODE_LN | MODE_CLUSTER | MODE_SPILL | MODE_RES, 4>::STAGES >= 4, "spill ring");

namespace {
template <int BN, int EXTRA, int CLMAX>
fnorm_status_t by_mode(const FusedLaunch& L) {
  constexpr int CL = MODE_CLUSTER | MODE_RES | EXTRA;
  switch (L.mode) {
    case MODE_POST | MODE_RES:           return launch_cfg<KCfg<BN, MODE_POST | CL, CLMAX>>(L);
    case MODE_POST | MODE_LN | MODE_RES: return launch_cfg<KCfg<BN, MODE_POST | MODE_LN | CL, CLMAX>>(L);
    default: break;
  }
  set_error("internal: unexpected residual post-norm mode %d", L.mode);
  return FNORM_ERR_UNSUPPORTED;
}
}  // namespace

fnorm_status_t launch_fused_post_residual_cluster(const FusedLaunch& L) {
  if (L.spill) {
    if (L.bn == 256) return by_mode<256, MODE_SPILL, 4>(L);
  } else {
    if (L.bn == 128) return by_mode<128, 0, 8>(L);
    if (L.bn == 256) return by_mode<256, 0, 4>(L);
  }
  set_error("internal: no cluster residual post-norm kernel for tile width %d", L.bn);
  return FNORM_ERR_UNSUPPORTED;
}

}  // namespace fnorm
