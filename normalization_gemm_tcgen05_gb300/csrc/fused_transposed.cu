// fused_transposed.cu — instantiations of the plain GEMM with transposed
// operands, C = op(A) @ op(B): A read MN-major from a [K, M] array (A^T) and/or
// B read K-major from an [N, K] array (B^T), straight from their row-major
// layouts.  The backward's unfused comparison (dC @ B^T and A_hat^T @ dC) and a
// general-purpose entry point (fnorm_gemm_ex).
#include "fused_launch.cuh"

namespace fnorm {

namespace {
template <int BN>
fnorm_status_t by_mode(const FusedLaunch& L) {
  switch (L.mode) {
    case MODE_AT:           return launch_cfg<KCfg<BN, MODE_AT>>(L);
    case MODE_BT:           return launch_cfg<KCfg<BN, MODE_BT>>(L);
    case MODE_AT | MODE_BT: return launch_cfg<KCfg<BN, MODE_AT | MODE_BT>>(L);
    default: break;
  }
  set_error("internal: unexpected transposed-GEMM mode %d", L.mode);
  return FNORM_ERR_UNSUPPORTED;
}
}  // namespace

fnorm_status_t launch_fused_transposed(const FusedLaunch& L) {
  if (L.spill || L.cluster != 1 || L.bres) {
    set_error("internal: unexpected transposed-GEMM plan");
    return FNORM_ERR_UNSUPPORTED;
  }
  switch (L.bn) {
    case 64:  return by_mode<64>(L);
    case 128: return by_mode<128>(L);
    case 256: return by_mode<256>(L);
    default: break;
  }
  set_error("internal: no transposed-GEMM kernel with tile width %d", L.bn);
  return FNORM_ERR_UNSUPPORTED;
}

}  // namespace fnorm
