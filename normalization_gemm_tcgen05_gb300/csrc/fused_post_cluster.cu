// fused_post_cluster.cu — instantiations of the fused kernel for the epilogue
// post-norm with rows split over a thread-block cluster along N and the row
// statistics exchanged through distributed shared memory:
//   resident: one 128-column slice per CTA (clusters of up to 8) or one
//             256-column slice (clusters of up to 4) kept in tensor memory;
//   spill:    S slices of 256 columns per CTA, normalised from L2 (clusters
//             of up to 4).
// The cluster bound sizes the statistics exchange buffers, which share the
// CTA's shared memory with the pipeline stages.
#include "fused_launch.cuh"

namespace fnorm {

// Pipeline depth the compute-bound cluster kernels are tuned for: a 4-stage
// ring of 48 KB stages (one staging box per epilogue warp makes room for it).
static_assert(KCfg<256, MODE_POST | MODE_LN | MODE_CLUSTER, 4>::STAGES >= 4, "resident cluster ring");
static_assert(KCfg<256, MODE_POST | MODE_LN | MODE_CLUSTER | MODE_SPILL, 4>::STAGES >= 4, "spill ring");

namespace {
template <int BN, int EXTRA, int CLMAX>
fnorm_status_t by_mode(const FusedLaunch& L) {
  constexpr int CL = MODE_CLUSTER | EXTRA;
  switch (L.mode) {
    case MODE_POST:                      return launch_cfg<KCfg<BN, MODE_POST | CL, CLMAX>>(L);
    case MODE_POST | MODE_LN:            return launch_cfg<KCfg<BN, MODE_POST | MODE_LN | CL, CLMAX>>(L);
    case MODE_POST | MODE_PRE:           return launch_cfg<KCfg<BN, MODE_POST | MODE_PRE | CL, CLMAX>>(L);
    case MODE_POST | MODE_LN | MODE_PRE:
      return launch_cfg<KCfg<BN, MODE_POST | MODE_LN | MODE_PRE | CL, CLMAX>>(L);
    default: break;
  }
  set_error("internal: unexpected post-norm mode %d", L.mode);
  return FNORM_ERR_UNSUPPORTED;
}
}  // namespace

fnorm_status_t launch_fused_post_cluster(const FusedLaunch& L) {
  if (L.spill) {
    if (L.bn == 256) return by_mode<256, MODE_SPILL, 4>(L);
  } else {
    if (L.bn == 128) return by_mode<128, 0, 8>(L);
    if (L.bn == 256) return by_mode<256, 0, 4>(L);
  }
  set_error("internal: no cluster post-norm kernel for tile width %d", L.bn);
  return FNORM_ERR_UNSUPPORTED;
}

}  // namespace fnorm
