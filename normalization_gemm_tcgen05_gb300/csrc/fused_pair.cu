// fused_pair.cu — instantiations of the fused kernel with the two-CTA MMA
// (tcgen05 cta_group::2): a 2-CTA cluster computes each [256 x 256] tile, each
// CTA staging its 128 rows of A and 128 of B's 256 columns, for the plain
// GEMM, the Lazy Pre-RMSNorm GEMM and the lazy pre-norms with the affine
// folded into B (persistent clusters over the tiles).
#include "fused_launch.cuh"

namespace fnorm {

static_assert(KCfg<256, MODE_CTA2>::STAGES >= 6, "two-CTA GEMM: [128 x 64] A + [64 x 128] B stages");
static_assert(KCfg<256, MODE_CTA2 | MODE_PRE | MODE_PRE_LN | MODE_AFF>::STAGES >= 5, "two-CTA pre-LayerNorm");

fnorm_status_t launch_fused_pair(const FusedLaunch& L) {
  if (L.bn != 256 || L.bres || L.spill || L.cluster != 1) {
    set_error("internal: unexpected two-CTA GEMM plan (tile width %d)", L.bn);
    return FNORM_ERR_UNSUPPORTED;
  }
  switch (L.mode) {
    case 0:                                 return launch_cfg<KCfg<256, MODE_CTA2>>(L);
    case MODE_PRE:                          return launch_cfg<KCfg<256, MODE_CTA2 | MODE_PRE>>(L);
    case MODE_PRE | MODE_AFF:               return launch_cfg<KCfg<256, MODE_CTA2 | MODE_PRE | MODE_AFF>>(L);
    case MODE_PRE | MODE_PRE_LN | MODE_AFF: return launch_cfg<KCfg<256, MODE_CTA2 | MODE_PRE | MODE_PRE_LN | MODE_AFF>>(L);
    default: break;
  }
  set_error("internal: no two-CTA GEMM kernel for mode %d", L.mode);
  return FNORM_ERR_UNSUPPORTED;
}

}  // namespace fnorm
