// fused_post_grid.cu — instantiations of the fused kernel for the epilogue
// post-norm of wide rows with the row statistics exchanged grid-wide: each
// CTA takes (row block, column chunk) units of S 256-column slices, writes
// the un-normalised slices and publishes its chunk's row statistics to global
// memory; its normaliser warps wait for the row block's other chunks, combine
// them in chunk order and normalise the unit in place.  ([FNF-ru] "Multi-CTA
// Norm Fusion": the CTAs sharing a row combine one pair of scalars per row;
// here any CTAs of the grid instead of one cluster.)
#include "fused_launch.cuh"

namespace fnorm {

static_assert(KCfg<256, MODE_POST | MODE_LN | MODE_SPILL | MODE_GX>::STAGES >= 4, "grid-exchange ring");

fnorm_status_t launch_fused_post_grid(const FusedLaunch& L) {
  if (!L.spill || L.cluster != 1 || L.bn != 256 || L.gx == nullptr) {
    set_error("internal: unexpected grid-exchange plan");
    return FNORM_ERR_UNSUPPORTED;
  }
  switch (L.mode) {
    case MODE_POST:           return launch_cfg<KCfg<256, MODE_POST | MODE_SPILL | MODE_GX>>(L);
    case MODE_POST | MODE_LN: return launch_cfg<KCfg<256, MODE_POST | MODE_LN | MODE_SPILL | MODE_GX>>(L);
    default: break;
  }
  set_error("internal: unexpected grid-exchange post-norm mode %d", L.mode);
  return FNORM_ERR_UNSUPPORTED;
}

}  // namespace fnorm
