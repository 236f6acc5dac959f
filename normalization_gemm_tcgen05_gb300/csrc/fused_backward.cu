// fused_backward.cu — instantiations of the fused kernel for the dgrad of the
// Lazy Pre-RMSNorm GEMM's backward ([FNF-ru] "Lazy Pre-Norm" limits: the
// backward has to rebuild what the forward never materialised):
//   dA = (rstd * dC) @ B^T + c * A,  c = -rstd^2 (dC . C) / K per row,
// B^T read K-major straight from B, the RMSNorm backward's row term added to
// the accumulator in the epilogue.  The wgrad, dB = A^T @ (rstd * dC), is the
// plain transposed GEMM of fused_transposed.cu on the same rstd * dC.
#include "fused_launch.cuh"

namespace fnorm {

static_assert(KCfg<256, MODE_DGRAD | MODE_BT>::STAGES >= 4, "dgrad ring");
static_assert(KCfg<256, MODE_AT>::STAGES >= 4, "wgrad ring");

fnorm_status_t launch_fused_backward(const FusedLaunch& L) {
  if (L.spill || L.cluster != 1 || L.bres) {
    set_error("internal: unexpected backward plan");
    return FNORM_ERR_UNSUPPORTED;
  }
  if (L.mode == (MODE_DGRAD | MODE_BT)) {
    switch (L.bn) {
      case 64:  return launch_cfg<KCfg<64, MODE_DGRAD | MODE_BT>>(L);
      case 128: return launch_cfg<KCfg<128, MODE_DGRAD | MODE_BT>>(L);
      case 256: return launch_cfg<KCfg<256, MODE_DGRAD | MODE_BT>>(L);
      default: break;
    }
  }
  set_error("internal: no backward kernel for mode %d, tile width %d", L.mode, L.bn);
  return FNORM_ERR_UNSUPPORTED;
}

}  // namespace fnorm
