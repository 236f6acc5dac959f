// fused_backward.cu — instantiations of the fused kernel for the backward of
// the Lazy Pre-RMSNorm GEMM ([FNF-ru] "Lazy Pre-Norm" limits: the backward
// rebuilds the normalised tensor the forward never materialised):
//   dgrad: dA = rstd * (dC @ B^T) - rstd^2 (dC . C) / K * A, B^T read K-major
//          from B, the row dots (dC . C) taken by the norm warps from the
//          staged tiles, the combination in the epilogue;
//   wgrad: dB = (A * rstd)^T @ dC, A^T read MN-major from A, its rows scaled
//          by rstd in shared memory by the norm warps before the MMA.
#include "fused_launch.cuh"

namespace fnorm {

static_assert(KCfg<256, MODE_PRE | MODE_DGRAD | MODE_BT>::STAGES >= 3, "dgrad ring (64 KB stages)");
static_assert(KCfg<256, MODE_AT | MODE_ASCALE>::STAGES >= 4, "wgrad ring");

fnorm_status_t launch_fused_backward(const FusedLaunch& L) {
  if (L.spill || L.cluster != 1 || L.bres) {
    set_error("internal: unexpected backward plan");
    return FNORM_ERR_UNSUPPORTED;
  }
  if (L.mode == (MODE_PRE | MODE_DGRAD | MODE_BT)) {
    switch (L.bn) {
      case 64:  return launch_cfg<KCfg<64, MODE_PRE | MODE_DGRAD | MODE_BT>>(L);
      case 128: return launch_cfg<KCfg<128, MODE_PRE | MODE_DGRAD | MODE_BT>>(L);
      case 256: return launch_cfg<KCfg<256, MODE_PRE | MODE_DGRAD | MODE_BT>>(L);
      default: break;
    }
  } else if (L.mode == (MODE_AT | MODE_ASCALE)) {
    switch (L.bn) {
      case 64:  return launch_cfg<KCfg<64, MODE_AT | MODE_ASCALE>>(L);
      case 128: return launch_cfg<KCfg<128, MODE_AT | MODE_ASCALE>>(L);
      case 256: return launch_cfg<KCfg<256, MODE_AT | MODE_ASCALE>>(L);
      default: break;
    }
  }
  set_error("internal: no backward kernel for mode %d, tile width %d", L.mode, L.bn);
  return FNORM_ERR_UNSUPPORTED;
}

}  // namespace fnorm
