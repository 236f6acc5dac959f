// fused_multicast.cu — instantiations of the fused kernel with B shared by a
// 2-CTA cluster along M (TMA multicast): the plain GEMM, the Lazy
// Pre-RMSNorm GEMM and the lazy pre-norms with the affine folded into B, on
// 256-column tiles.  The two CTAs of a cluster compute the tiles of two
// neighbouring 128-row blocks at the same columns with their own one-CTA
// MMAs; each loads half of every stage's B tile into both, so each SM reads
// 32 KB from L2 per 64-deep k-block instead of 48 KB.
#include "fused_launch.cuh"

namespace fnorm {

static_assert(KCfg<256, MODE_MCB>::STAGES >= 4, "B multicast: [128 x 64] A + [64 x 256] B stages");
static_assert(KCfg<256, MODE_MCB | MODE_PRE | MODE_PRE_LN | MODE_AFF>::STAGES >= 4, "B multicast pre-LayerNorm");

fnorm_status_t launch_fused_mcb(const FusedLaunch& L) {
  if (L.bn != 256 || L.bres || L.spill || L.cluster != 1) {
    set_error("internal: unexpected B-multicast GEMM plan (tile width %d)", L.bn);
    return FNORM_ERR_UNSUPPORTED;
  }
  switch (L.mode) {
    case 0:                                 return launch_cfg<KCfg<256, MODE_MCB>>(L);
    case MODE_PRE:                          return launch_cfg<KCfg<256, MODE_MCB | MODE_PRE>>(L);
    case MODE_PRE | MODE_AFF:               return launch_cfg<KCfg<256, MODE_MCB | MODE_PRE | MODE_AFF>>(L);
    case MODE_PRE | MODE_PRE_LN | MODE_AFF: return launch_cfg<KCfg<256, MODE_MCB | MODE_PRE | MODE_PRE_LN | MODE_AFF>>(L);
    default: break;
  }
  set_error("internal: no B-multicast GEMM kernel for mode %d", L.mode);
  return FNORM_ERR_UNSUPPORTED;
}

}  // namespace fnorm
