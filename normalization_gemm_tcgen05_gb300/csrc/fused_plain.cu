// fused_plain.cu — instantiations of the fused kernel for the plain GEMM and
// the Lazy Pre-RMSNorm GEMM (one CTA per 128 x BN tile, persistent), with B
// streamed per k-block or, for N <= BN and short K, resident in shared memory.
#include "fused_launch.cuh"

namespace fnorm {

// Pipeline depths the streaming kernels are tuned for (stage = A + B tile).
static_assert(KCfg<256, MODE_PRE>::STAGES >= 4, "Lazy Pre-Norm, 256-column tiles");
static_assert(KCfg<128, 0>::STAGES >= 5 && KCfg<64, 0>::STAGES >= 8, "GEMM, narrow tiles");

namespace {
template <int BN>
fnorm_status_t by_mode(const FusedLaunch& L, bool pre) {
  if (L.bres) return pre ? launch_cfg<KCfg<BN, MODE_PRE | MODE_BRES>>(L) : launch_cfg<KCfg<BN, MODE_BRES>>(L);
  return pre ? launch_cfg<KCfg<BN, MODE_PRE>>(L) : launch_cfg<KCfg<BN, 0>>(L);
}
}  // namespace

fnorm_status_t launch_fused_plain(const FusedLaunch& L) {
  const bool pre = (L.mode & MODE_PRE) != 0;
  if ((L.mode & ~MODE_PRE) != 0 || L.spill || L.cluster != 1) {
    set_error("internal: unexpected plain-GEMM plan (mode %d)", L.mode);
    return FNORM_ERR_UNSUPPORTED;
  }
  switch (L.bn) {
    case 64:  return by_mode<64>(L, pre);
    case 128: return by_mode<128>(L, pre);
    case 256: return by_mode<256>(L, pre);
    default: break;
  }
  set_error("internal: no plain-GEMM kernel with tile width %d", L.bn);
  return FNORM_ERR_UNSUPPORTED;
}

}  // namespace fnorm
