// fused_multicast_grid.cu — instantiations of the grid-exchange post-norm
// (resident 256-column tiles, row statistics exchanged grid-wide through a
// workspace) with B shared by a 2-CTA cluster along M through TMA multicast.
// ([FNF-ru] "Multi-CTA Norm Fusion" for the exchange; the cluster here shares
// operand loads, not statistics.)
#include "fused_launch.cuh"

namespace fnorm {

static_assert(KCfg<256, MODE_POST | MODE_LN | MODE_GX | MODE_MCB>::STAGES >= 4, "B multicast grid exchange");

fnorm_status_t launch_fused_mcb_grid(const FusedLaunch& L) {
  if (L.spill || L.cluster != 1 || L.bn != 256 || L.bres || L.gx == nullptr) {
    set_error("internal: unexpected grid-exchange plan");
    return FNORM_ERR_UNSUPPORTED;
  }
  constexpr int X = MODE_GX | MODE_MCB;
  switch (L.mode) {
    case MODE_POST:                      return launch_cfg<KCfg<256, MODE_POST | X>>(L);
    case MODE_POST | MODE_LN:            return launch_cfg<KCfg<256, MODE_POST | MODE_LN | X>>(L);
    case MODE_POST | MODE_PRE:           return launch_cfg<KCfg<256, MODE_POST | MODE_PRE | X>>(L);
    case MODE_POST | MODE_LN | MODE_PRE: return launch_cfg<KCfg<256, MODE_POST | MODE_LN | MODE_PRE | X>>(L);
    default: break;
  }
  set_error("internal: unexpected grid-exchange post-norm mode %d", L.mode);
  return FNORM_ERR_UNSUPPORTED;
}

}  // namespace fnorm
