// fused_post_cluster.cu — instantiations of the fused kernel for the epilogue
// post-norm with rows split over a thread-block cluster along N and the row
// statistics exchanged through distributed shared memory.
//   one accumulator subtile per CTA (128 or 256 columns), clusters of <= 8;
//   two subtiles of 256 (512 columns, K tile 32), clusters of <= 16.
#include "fused_launch.cuh"

namespace fnorm {

namespace {
template <int BN, int NSUB, int BK, int CLBIT>
fnorm_status_t by_mode(const FusedLaunch& L) {
  switch (L.mode) {
    case MODE_POST:
      return launch_cfg<KCfg<BN, NSUB, BK, MODE_POST | CLBIT>>(L);
    case MODE_POST | MODE_LN:
      return launch_cfg<KCfg<BN, NSUB, BK, MODE_POST | MODE_LN | CLBIT>>(L);
    case MODE_POST | MODE_PRE:
      return launch_cfg<KCfg<BN, NSUB, BK, MODE_POST | MODE_PRE | CLBIT>>(L);
    case MODE_POST | MODE_LN | MODE_PRE:
      return launch_cfg<KCfg<BN, NSUB, BK, MODE_POST | MODE_LN | MODE_PRE | CLBIT>>(L);
    default: break;
  }
  set_error("internal: unexpected post-norm mode %d", L.mode);
  return FNORM_ERR_UNSUPPORTED;
}
}  // namespace

fnorm_status_t launch_fused_post_cluster(const FusedLaunch& L) {
  if (L.nsub == 1 && L.bn_sub == 128) return by_mode<128, 1, 64, MODE_CLUSTER>(L);
  if (L.nsub == 1 && L.bn_sub == 256) return by_mode<256, 1, 64, MODE_CLUSTER>(L);
  if (L.nsub == 2 && L.bn_sub == 256) return by_mode<256, 2, 32, MODE_CL16>(L);
  set_error("internal: no cluster post-norm kernel for %d x %d columns", L.nsub, L.bn_sub);
  return FNORM_ERR_UNSUPPORTED;
}

}  // namespace fnorm
