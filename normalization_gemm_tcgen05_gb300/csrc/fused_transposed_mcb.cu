// fused_transposed_mcb.cu — instantiations of the GEMMs with transposed
// operands (fused_transposed.cu) and of the Lazy Pre-RMSNorm backward's dgrad
// (fused_backward.cu) with B shared by a 2-CTA cluster along M: the two CTAs
// compute neighbouring 128-row blocks at the same 256 columns, and each loads
// half of every k-block's B tile into both CTAs' shared memory with one TMA
// multicast.  B read as stored: MN-major boxes of a [K, N] array, or, for the
// B^T operand, half of the [256 x 64] K-major box of an [N, K] array each.
#include "fused_launch.cuh"

namespace fnorm {

static_assert(KCfg<256, MODE_AT | MODE_MCB>::STAGES >= 4, "wgrad ring with B multicast");
static_assert(KCfg<256, MODE_DGRAD | MODE_BT | MODE_MCB>::STAGES >= 4, "dgrad ring with B multicast");

fnorm_status_t launch_fused_transposed_mcb(const FusedLaunch& L) {
  if (L.spill || L.cluster != 1 || L.bres || L.bn != 256) {
    set_error("internal: unexpected transposed-GEMM plan for B multicast");
    return FNORM_ERR_UNSUPPORTED;
  }
  switch (L.mode) {
    case MODE_AT:               return launch_cfg<KCfg<256, MODE_AT | MODE_MCB>>(L);
    case MODE_BT:               return launch_cfg<KCfg<256, MODE_BT | MODE_MCB>>(L);
    case MODE_AT | MODE_BT:     return launch_cfg<KCfg<256, MODE_AT | MODE_BT | MODE_MCB>>(L);
    case MODE_DGRAD | MODE_BT:  return launch_cfg<KCfg<256, MODE_DGRAD | MODE_BT | MODE_MCB>>(L);
    default: break;
  }
  set_error("internal: unexpected transposed-GEMM mode %d for B multicast", L.mode);
  return FNORM_ERR_UNSUPPORTED;
}

}  // namespace fnorm
