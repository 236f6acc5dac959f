// fused_post_grid.cu — instantiations of the fused kernel for the epilogue
// post-norm of rows wider than a cluster holds: the plain GEMM's 256-column
// tiles stay in tensor memory while the tiles of each row block, on any CTAs
// of the grid, exchange their per-row partial statistics through a global
// workspace; each tile then combines all of them in tile order and normalises
// itself.  ([FNF-ru] "Multi-CTA Norm Fusion": the CTAs sharing a row combine
// one pair of scalars per row; here any CTAs of the grid instead of one
// cluster, so that a row of any width keeps every tile double buffered.)
#include "fused_launch.cuh"

namespace fnorm {

static_assert(KCfg<256, MODE_POST | MODE_LN | MODE_GX>::STAGES >= 4, "grid-exchange ring");
static_assert(KCfg<256, MODE_POST | MODE_LN | MODE_PRE | MODE_GX>::STAGES >= 4, "grid-exchange ring, pre-norm");

fnorm_status_t launch_fused_post_grid(const FusedLaunch& L) {
  if (L.spill || L.cluster != 1 || L.bn != 256 || L.bres || L.gx == nullptr) {
    set_error("internal: unexpected grid-exchange plan");
    return FNORM_ERR_UNSUPPORTED;
  }
  switch (L.mode) {
    case MODE_POST:                      return launch_cfg<KCfg<256, MODE_POST | MODE_GX>>(L);
    case MODE_POST | MODE_LN:            return launch_cfg<KCfg<256, MODE_POST | MODE_LN | MODE_GX>>(L);
    case MODE_POST | MODE_PRE:           return launch_cfg<KCfg<256, MODE_POST | MODE_PRE | MODE_GX>>(L);
    case MODE_POST | MODE_LN | MODE_PRE: return launch_cfg<KCfg<256, MODE_POST | MODE_LN | MODE_PRE | MODE_GX>>(L);
    default: break;
  }
  set_error("internal: unexpected grid-exchange post-norm mode %d", L.mode);
  return FNORM_ERR_UNSUPPORTED;
}

}  // namespace fnorm
