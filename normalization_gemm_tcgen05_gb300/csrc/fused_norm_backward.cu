// fused_norm_backward.cu — instantiations of the fused kernel for the
// post-norm's backward regrouped onto the GEMM that produces the norm's output
// gradient ([TFN] "fusion regrouping": in the backward the norm is fused with
// the consuming layer's data-gradient GEMM, dC = G @ op(W), instead of with
// the GEMM it followed in the forward).  The accumulator holds dC; the
// epilogue writes dH and the column partials of dgamma and dbeta.  Rows of up
// to 256 columns sit in one CTA's tile, rows of up to 1024 over a cluster of
// 2 or 4 CTAs with the two row sums exchanged through distributed shared
// memory, wider rows in resident 256-column tiles with the row sums exchanged
// grid-wide through the caller's workspace (a cooperative launch).  The
// consumer's weight is read as stored: W [N, J] as the B^T operand (K-major),
// or W [J, N] as the plain B operand.
#include "fused_launch.cuh"

namespace fnorm {

static_assert(KCfg<256, MODE_POST | MODE_LN | MODE_NBWD | MODE_CLUSTER | MODE_BT, 4>::STAGES >= 4,
              "post-norm backward ring");

namespace {
template <int BN, int X, int CLMAX>
fnorm_status_t by_norm(const FusedLaunch& L) {
  switch (L.mode & ~MODE_BT) {
    case MODE_POST | MODE_NBWD:           return launch_cfg<KCfg<BN, MODE_POST | MODE_NBWD | X, CLMAX>>(L);
    case MODE_POST | MODE_NBWD | MODE_LN: return launch_cfg<KCfg<BN, MODE_POST | MODE_NBWD | MODE_LN | X, CLMAX>>(L);
    default: break;
  }
  set_error("internal: unexpected post-norm backward mode %d", L.mode);
  return FNORM_ERR_UNSUPPORTED;
}

template <int X>
fnorm_status_t by_layout(const FusedLaunch& L) {
  if (L.gx != nullptr) {
    if (L.cluster == 1 && L.bn == 256) return by_norm<256, X | MODE_GX, 0>(L);
    set_error("internal: the grid-exchange post-norm backward takes one-CTA tiles of 256 columns");
    return FNORM_ERR_UNSUPPORTED;
  }
  if (L.cluster == 1 && L.bn == 128) return by_norm<128, X, 0>(L);
  if (L.cluster == 1 && L.bn == 256) return by_norm<256, X, 0>(L);
  if (L.cluster > 1 && L.bn == 256) return by_norm<256, X | MODE_CLUSTER, 4>(L);
  set_error("internal: no post-norm backward kernel for a cluster of %d, tile width %d", L.cluster, L.bn);
  return FNORM_ERR_UNSUPPORTED;
}
}  // namespace

fnorm_status_t launch_fused_norm_backward(const FusedLaunch& L) {
  if (L.spill || L.bres) {
    set_error("internal: unexpected post-norm backward plan");
    return FNORM_ERR_UNSUPPORTED;
  }
  return (L.mode & MODE_BT) ? by_layout<MODE_BT>(L) : by_layout<0>(L);
}

}  // namespace fnorm
