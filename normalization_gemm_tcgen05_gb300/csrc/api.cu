// api.cu — the extern "C" entry points of libfnorm (declared in
// include/fnorm.h): argument validation, the plan (tile widths, cluster size)
// and dispatch to the kernels.  No entry point allocates memory or
// synchronises the host, except fnorm_check_status, whose job is to.
#include <atomic>
#include <cmath>
#include <cstdint>

#include "fused_gemm.cuh"
#include "internal.h"

namespace fnorm {
const char* last_error_cstr();
void clear_error();
void set_wait_limit(uint64_t ns);
fnorm_status_t read_and_clear_status(cudaStream_t stream);

namespace {
std::atomic<int> g_forced_cluster{0};
std::atomic<int> g_pair_mode{-1};  // fnorm_set_pair_mma: -1 automatic, 0 never, 1 whenever eligible
std::atomic<int> g_mcb_mode{-1};   // fnorm_set_b_multicast: -1 automatic, 0 never, 1 whenever eligible

constexpr int64_t kMaxDim = 0x7fffffffLL;

fnorm_status_t bad(const char* msg) {
  set_error("%s", msg);
  return FNORM_ERR_INVALID_ARG;
}

fnorm_status_t check_mnk(int64_t M, int64_t N, int64_t K) {
  if (M < 0 || M > kMaxDim) return bad("M must be in [0, 2^31)");
  if (N < 8 || N > kMaxDim || N % 8 != 0) return bad("N must be a multiple of 8 in [8, 2^31)");
  if (K < 8 || K > kMaxDim || K % 8 != 0) return bad("K must be a multiple of 8 in [8, 2^31)");
  return FNORM_OK;
}

fnorm_status_t check_eps(float eps, const char* name) {
  if (!(eps > 0.0f) || !std::isfinite(eps)) {
    set_error("%s must be finite and > 0", name);
    return FNORM_ERR_INVALID_ARG;
  }
  return FNORM_OK;
}

fnorm_status_t check_ptr(const void* p, const char* name, uintptr_t align, bool optional) {
  if (p == nullptr) {
    if (optional) return FNORM_OK;
    set_error("%s must not be NULL", name);
    return FNORM_ERR_INVALID_ARG;
  }
  if (reinterpret_cast<uintptr_t>(p) % align != 0) {
    set_error("%s must be %u-byte aligned", name, (unsigned)align);
    return FNORM_ERR_INVALID_ARG;
  }
  return FNORM_OK;
}

#define FN_TRY(expr)                      \
  do {                                    \
    fnorm_status_t s_ = (expr);           \
    if (s_ != FNORM_OK) return s_;        \
  } while (0)

int round64(int64_t x) { return static_cast<int>((x + 63) / 64 * 64); }

int gemm_tile_n(int64_t N) { return N <= 64 ? 64 : (N <= 128 ? 128 : 256); }

// Tile width for the transposed and backward GEMMs: the widest tile that
// covers N, halved while a grid of such tiles fills less than one wave of
// SMs and the halved one still fits in one.  (A [2048 x 1024] weight
// gradient: 64 tiles of 128 x 256 would leave 88 of 152 SMs idle.)
int fill_tile_n(int64_t M, int64_t N) {
  int bn = gemm_tile_n(N);
  DeviceInfo dev;
  if (current_device(&dev) != FNORM_OK) return bn;
  auto tiles = [&](int b) { return ((M + 127) / 128) * ((N + b - 1) / b); };
  while (bn > 64 && tiles(bn) < dev.num_sms && tiles(bn / 2) <= dev.num_sms) bn /= 2;
  return bn;
}

// Keep all of B in shared memory when it is one tile wide (N <= bn), at most
// 128 KB, and each CTA will visit several row blocks (more row blocks than
// SMs), so B is read once per CTA instead of once per tile.
bool want_resident_b(int64_t M, int64_t N, int64_t K, int bn) {
  DeviceInfo dev;
  if (current_device(&dev) != FNORM_OK) return false;
  const int64_t kb_max = 131072 / (64LL * bn * 2);
  return N <= bn && (K + 63) / 64 <= kb_max && (M + 127) / 128 > dev.num_sms;
}

// Two-CTA MMA for a 256-column GEMM tile, on request only (fnorm_set_pair_mma).
// The pair halves what each SM takes in per tile, but on GB300 it measured no
// faster than the one-CTA tile on any shape tried (8192 x 4096 x 4096: 160 us
// against 158 us; 16384 x 4096 x 2048: 188 us against 177 us): the one-CTA
// mainloop waits on the latency of its loads, not on their bytes, and the
// pair's loads complete later.  Automatic selection therefore keeps one CTA.
bool want_pair(int bn, bool bres) {
  return g_pair_mode.load(std::memory_order_relaxed) == 1 && bn == 256 && !bres;
}

// B shared by a 2-CTA cluster along M (TMA multicast) for 256-column tiles
// with B streamed: each SM then reads a third less from L2 per k-block.
// Automatic selection takes it whenever there are two row blocks to pair.
bool want_mcb(int64_t M, int bn, bool bres) {
  const int mode = g_mcb_mode.load(std::memory_order_relaxed);
  return mode != 0 && bn == 256 && !bres && (mode == 1 || M > 128);
}

// How a post-norm row of width N is laid out over the CTAs.
//   N <= 256:     one CTA per row block holds the whole row in tensor memory
//                 (tile width N rounded up to 64);
//   N <= 1024:    resident cluster of 2 or 4 CTAs, each holding one 128- or
//                 256-column slice in tensor memory;
//   wider rows:   with a grid-exchange workspace (fnorm_gemm_postnorm_ws,
//                 fnorm_gemm_postnorm_noalloc), the plain GEMM's 256-column
//                 tiles over the whole grid, resident in tensor memory, the
//                 row statistics exchanged through the workspace; without
//                 one (fnorm_gemm_postnorm), the spill layout on a cluster of
//                 kSpillCluster CTAs, each owning S = ceil(N / (cluster *
//                 256)) slices of 256 columns.
// A forced cluster size c keeps the resident layout when each CTA's share fits
// one tile (256 columns for c <= 4, 128 for c = 8), else uses the spill layout
// (c <= 4).
constexpr int kSpillCluster = 4;

struct PostPlan {
  int cluster, bn, slices;
  bool spill, gx;
};

fnorm_status_t plan_postnorm(int64_t N, int forced, PostPlan* pl, bool allow_gx) {
  pl->gx = false;
  auto resident = [&](int c) -> bool {
    const int64_t w = (N + c - 1) / c;  // columns per CTA
    if (w > 256 || (c > 4 && w > 128)) return false;
    pl->cluster = c;
    pl->bn = (c == 1) ? round64(w) : (w <= 128 ? 128 : 256);
    pl->slices = 1;
    pl->spill = false;
    return true;
  };
  auto spill = [&](int c) -> bool {
    const int64_t s = (N + 256LL * c - 1) / (256LL * c);
    if (c > 4 || s > (1 << 20)) return false;
    pl->cluster = c, pl->bn = 256, pl->slices = static_cast<int>(s), pl->spill = true;
    return true;
  };
  if (forced != 0) {
    if (resident(forced) || spill(forced)) return FNORM_OK;
    set_error("a row of %lld columns does not fit a forced cluster of %d CTAs", (long long)N, forced);
    return FNORM_ERR_UNSUPPORTED;
  }
  for (int c : {1, 2, 4})
    if (resident(c)) return FNORM_OK;
  if (allow_gx) {
    pl->cluster = 1, pl->bn = 256, pl->slices = 1, pl->spill = false, pl->gx = true;
    return FNORM_OK;
  }
  if (spill(kSpillCluster)) return FNORM_OK;
  set_error("post-norm row of %lld columns is too wide", (long long)N);
  return FNORM_ERR_UNSUPPORTED;
}

FusedLaunch base_launch(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K, void* stream) {
  FusedLaunch L{};
  L.A = A;
  L.B = B;
  L.C = C;
  L.M = static_cast<int>(M);
  L.N = static_cast<int>(N);
  L.K = static_cast<int>(K);
  L.slices = 1;
  L.spill = false;
  L.bres = false;
  L.cluster = 1;
  L.eps = 1.0f;
  L.pre_eps = 1.0f;
  L.stream = static_cast<cudaStream_t>(stream);
  return L;
}

}  // namespace

int forced_postnorm_cluster() { return g_forced_cluster.load(std::memory_order_relaxed); }

}  // namespace fnorm

using namespace fnorm;

extern "C" {

fnorm_status_t fnorm_gemm(const fnorm_bf16* A, const fnorm_bf16* B, fnorm_bf16* C, int64_t M, int64_t N,
                          int64_t K, void* stream) {
  clear_error();
  FN_TRY(check_mnk(M, N, K));
  if (M == 0) return FNORM_OK;
  FN_TRY(check_ptr(A, "A", 16, false));
  FN_TRY(check_ptr(B, "B", 16, false));
  FN_TRY(check_ptr(C, "C", 16, false));
  FusedLaunch L = base_launch(A, B, C, M, N, K, stream);
  L.mode = 0;
  L.bn = gemm_tile_n(N);
  L.bres = want_resident_b(M, N, K, L.bn);
  if (want_pair(L.bn, L.bres)) return launch_fused_pair(L);
  if (want_mcb(M, L.bn, L.bres)) return launch_fused_mcb(L);
  return launch_fused_plain(L);
}

fnorm_status_t fnorm_gemm_ex(const fnorm_bf16* A, const fnorm_bf16* B, fnorm_bf16* C, int64_t M, int64_t N,
                             int64_t K, int trans_a, int trans_b, void* stream) {
  clear_error();
  FN_TRY(check_mnk(M, N, K));
  if ((trans_a != 0 && trans_a != 1) || (trans_b != 0 && trans_b != 1)) return bad("trans_a, trans_b must be 0 or 1");
  if (trans_a && M % 8 != 0) return bad("with trans_a, M must be a multiple of 8 (the [K, M] row pitch)");
  if (M == 0) return FNORM_OK;
  FN_TRY(check_ptr(A, "A", 16, false));
  FN_TRY(check_ptr(B, "B", 16, false));
  FN_TRY(check_ptr(C, "C", 16, false));
  if (!trans_a && !trans_b) return fnorm_gemm(A, B, C, M, N, K, stream);
  FusedLaunch L = base_launch(A, B, C, M, N, K, stream);
  L.mode = (trans_a ? MODE_AT : 0) | (trans_b ? MODE_BT : 0);
  L.bn = fill_tile_n(M, N);
  return want_mcb(M, L.bn, false) ? launch_fused_transposed_mcb(L) : launch_fused_transposed(L);
}

fnorm_status_t fnorm_lazy_prenorm_gemm(const fnorm_bf16* A, const fnorm_bf16* B, fnorm_bf16* C, int64_t M,
                                       int64_t N, int64_t K, float eps, float* rstd_out, void* stream) {
  clear_error();
  FN_TRY(check_mnk(M, N, K));
  FN_TRY(check_eps(eps, "eps"));
  if (M == 0) return FNORM_OK;
  FN_TRY(check_ptr(A, "A", 16, false));
  FN_TRY(check_ptr(B, "B", 16, false));
  FN_TRY(check_ptr(C, "C", 16, false));
  FN_TRY(check_ptr(rstd_out, "rstd_out", 4, true));
  FusedLaunch L = base_launch(A, B, C, M, N, K, stream);
  L.mode = MODE_PRE;
  L.bn = gemm_tile_n(N);
  L.bres = want_resident_b(M, N, K, L.bn);
  L.pre_eps = eps;
  L.rstd_out = rstd_out;
  if (want_pair(L.bn, L.bres)) return launch_fused_pair(L);
  if (want_mcb(M, L.bn, L.bres)) return launch_fused_mcb(L);
  return launch_fused_plain(L);
}

}  // extern "C"

namespace fnorm {
namespace {
// Where the wide-row grid exchange keeps its statistics: nowhere (the call
// takes the cluster spill layout), the caller's workspace, or the library's
// fixed device array.
enum class Ws { kNone, kCaller, kFixed };

// fnorm_gemm_postnorm and its workspace and allocation-free twins: they
// differ only in where the wide-row grid exchange keeps its statistics
fnorm_status_t gemm_postnorm_impl(const fnorm_bf16* A, const fnorm_bf16* B, fnorm_bf16* C, int64_t M, int64_t N,
                                  int64_t K, fnorm_norm_t norm, const fnorm_bf16* gamma, const fnorm_bf16* beta,
                                  float eps, int pre_rmsnorm, float pre_eps, float* mean_out, float* rstd_out,
                                  float* pre_rstd_out, void* workspace, size_t workspace_bytes, void* stream, Ws ws) {
  clear_error();
  FN_TRY(check_mnk(M, N, K));
  if (norm != FNORM_RMSNORM && norm != FNORM_LAYERNORM) return bad("norm must be FNORM_RMSNORM or FNORM_LAYERNORM");
  if (pre_rmsnorm != 0 && pre_rmsnorm != 1) return bad("pre_rmsnorm must be 0 or 1");
  FN_TRY(check_eps(eps, "eps"));
  if (pre_rmsnorm) FN_TRY(check_eps(pre_eps, "pre_eps"));
  if (norm == FNORM_RMSNORM && mean_out != nullptr) return bad("mean_out is only defined for LayerNorm");
  if (!pre_rmsnorm && pre_rstd_out != nullptr) return bad("pre_rstd_out needs pre_rmsnorm = 1");
  if (ws == Ws::kCaller && workspace == nullptr) ws = Ws::kNone;
  PostPlan plan{};
  FN_TRY(plan_postnorm(N, forced_postnorm_cluster(), &plan, ws != Ws::kNone));
  if (M == 0) return FNORM_OK;
  FN_TRY(check_ptr(A, "A", 16, false));
  FN_TRY(check_ptr(B, "B", 16, false));
  FN_TRY(check_ptr(C, "C", 16, false));
  FN_TRY(check_ptr(gamma, "gamma", 16, true));
  FN_TRY(check_ptr(beta, "beta", 16, true));
  FN_TRY(check_ptr(mean_out, "mean_out", 4, true));
  FN_TRY(check_ptr(rstd_out, "rstd_out", 4, true));
  FN_TRY(check_ptr(pre_rstd_out, "pre_rstd_out", 4, true));
  FusedLaunch L = base_launch(A, B, C, M, N, K, stream);
  GxScratch caller_gx{};
  if (plan.gx && ws == Ws::kCaller && (M + 127) / 128 <= kGxMaxRowBlocks)
    FN_TRY(gx_scratch_from(workspace, workspace_bytes, M, N, &caller_gx));
  if (plan.gx) {
    // one CTA per tile of a row at least (no CTA may hold two tiles of the
    // row block it waits on); a row with more tiles than SMs takes the
    // cluster spill layout instead
    DeviceInfo dev;
    FN_TRY(current_device(&dev));
    if ((N + 255) / 256 > dev.num_sms || (M + 127) / 128 > kGxMaxRowBlocks) {
      FN_TRY(plan_postnorm(N, forced_postnorm_cluster(), &plan, false));
    } else if (ws == Ws::kFixed) {
      const GxScratch* gx = nullptr;
      FN_TRY(noalloc_scratch(L.stream, &gx));
      const int64_t rb = (M + 127) / 128, units = rb * ((N + 255) / 256);
      if (units > gx->units_cap || rb > gx->rowblocks_cap) {
        set_error("fnorm_gemm_postnorm_noalloc: %lld tiles of 128 x 256 (%lld row blocks) exceed its fixed "
                  "workspace (%d tiles, %d row blocks); use fnorm_gemm_postnorm or fnorm_gemm_postnorm_ws",
                  (long long)units, (long long)rb, gx->units_cap, gx->rowblocks_cap);
        return FNORM_ERR_UNSUPPORTED;
      }
      L.gx = gx;
    } else {
      L.gx = &caller_gx;
    }
  }
  L.mode = MODE_POST | (norm == FNORM_LAYERNORM ? MODE_LN : 0) | (pre_rmsnorm ? MODE_PRE : 0);
  L.bn = plan.bn;
  L.slices = plan.slices;
  L.spill = plan.spill;
  L.cluster = plan.cluster;
  L.bres = (plan.cluster == 1 && !plan.spill && !plan.gx) && want_resident_b(M, N, K, plan.bn);
  L.eps = eps;
  L.pre_eps = pre_rmsnorm ? pre_eps : 1.0f;
  L.gamma = gamma;
  L.beta = beta;
  L.mean_out = mean_out;
  L.rstd_out = rstd_out;
  L.pre_rstd_out = pre_rstd_out;
  if (plan.gx) {
    // The grid exchange shares B over 2-CTA clusters like the plain GEMM
    // (2.5-4.2 % faster at N = 4096 and 8192); a device that will not launch
    // that grid of clusters takes the one-CTA kernel.
    if (want_mcb(M, L.bn, L.bres)) {
      const fnorm_status_t st = launch_fused_mcb_grid(L);
      if (st != FNORM_ERR_UNSUPPORTED) return st;
      clear_error();
    }
    return launch_fused_post_grid(L);
  }
  return (plan.cluster == 1 && !plan.spill) ? launch_fused_post_single(L) : launch_fused_post_cluster(L);
}
}  // namespace
}  // namespace fnorm

extern "C" {

fnorm_status_t fnorm_gemm_postnorm(const fnorm_bf16* A, const fnorm_bf16* B, fnorm_bf16* C, int64_t M,
                                   int64_t N, int64_t K, fnorm_norm_t norm, const fnorm_bf16* gamma,
                                   const fnorm_bf16* beta, float eps, int pre_rmsnorm, float pre_eps,
                                   float* mean_out, float* rstd_out, float* pre_rstd_out, void* stream) {
  return gemm_postnorm_impl(A, B, C, M, N, K, norm, gamma, beta, eps, pre_rmsnorm, pre_eps, mean_out, rstd_out,
                            pre_rstd_out, nullptr, 0, stream, Ws::kNone);
}

fnorm_status_t fnorm_gemm_postnorm_ws(const fnorm_bf16* A, const fnorm_bf16* B, fnorm_bf16* C, int64_t M,
                                      int64_t N, int64_t K, fnorm_norm_t norm, const fnorm_bf16* gamma,
                                      const fnorm_bf16* beta, float eps, int pre_rmsnorm, float pre_eps,
                                      float* mean_out, float* rstd_out, float* pre_rstd_out, void* workspace,
                                      size_t workspace_bytes, void* stream) {
  return gemm_postnorm_impl(A, B, C, M, N, K, norm, gamma, beta, eps, pre_rmsnorm, pre_eps, mean_out, rstd_out,
                            pre_rstd_out, workspace, workspace_bytes, stream, Ws::kCaller);
}

fnorm_status_t fnorm_postnorm_workspace_size(int64_t M, int64_t N, size_t* bytes) {
  clear_error();
  if (bytes == nullptr) return bad("bytes must not be NULL");
  FN_TRY(check_mnk(M, N, 8));
  PostPlan plan{};
  FN_TRY(plan_postnorm(N, forced_postnorm_cluster(), &plan, true));
  *bytes = (plan.gx && M > 0 && (M + 127) / 128 <= kGxMaxRowBlocks) ? gx_workspace_bytes(M, N) : 0;
  return FNORM_OK;
}

fnorm_status_t fnorm_gemm_postnorm_noalloc(const fnorm_bf16* A, const fnorm_bf16* B, fnorm_bf16* C, int64_t M,
                                           int64_t N, int64_t K, fnorm_norm_t norm, const fnorm_bf16* gamma,
                                           const fnorm_bf16* beta, float eps, int pre_rmsnorm, float pre_eps,
                                           float* mean_out, float* rstd_out, float* pre_rstd_out, void* stream) {
  return gemm_postnorm_impl(A, B, C, M, N, K, norm, gamma, beta, eps, pre_rmsnorm, pre_eps, mean_out, rstd_out,
                            pre_rstd_out, nullptr, 0, stream, Ws::kFixed);
}


fnorm_status_t fnorm_fold_prenorm_affine(const fnorm_bf16* B, int64_t K, int64_t N, const fnorm_bf16* gamma,
                                         const fnorm_bf16* beta, fnorm_bf16* B_folded, float* colsum, float* bias,
                                         void* stream) {
  clear_error();
  FN_TRY(check_mnk(0, N, K));
  if ((beta == nullptr) != (bias == nullptr)) return bad("bias must be given exactly when beta is");
  FN_TRY(check_ptr(B, "B", 16, false));
  FN_TRY(check_ptr(B_folded, "B_folded", 16, false));
  FN_TRY(check_ptr(gamma, "gamma", 2, true));
  FN_TRY(check_ptr(beta, "beta", 2, true));
  FN_TRY(check_ptr(colsum, "colsum", 16, true));
  FN_TRY(check_ptr(bias, "bias", 16, true));
  {
    // B_folded may be B itself (in place) but no other overlap
    const auto b0 = reinterpret_cast<uintptr_t>(B), f0 = reinterpret_cast<uintptr_t>(B_folded);
    const uintptr_t bytes = static_cast<uintptr_t>(K) * static_cast<uintptr_t>(N) * 2u;
    if (b0 != f0 && b0 < f0 + bytes && f0 < b0 + bytes) return bad("B_folded overlaps B without being B");
  }
  return launch_fold_prenorm_affine(B, static_cast<int>(K), static_cast<int>(N), gamma, beta, B_folded, colsum,
                                    bias, static_cast<cudaStream_t>(stream));
}

fnorm_status_t fnorm_prenorm_gemm(const fnorm_bf16* A, const fnorm_bf16* B_folded, fnorm_bf16* C, int64_t M,
                                  int64_t N, int64_t K, fnorm_norm_t norm, const float* colsum, const float* bias,
                                  float eps, float* mean_out, float* rstd_out, void* stream) {
  clear_error();
  FN_TRY(check_mnk(M, N, K));
  if (norm != FNORM_RMSNORM && norm != FNORM_LAYERNORM) return bad("norm must be FNORM_RMSNORM or FNORM_LAYERNORM");
  FN_TRY(check_eps(eps, "eps"));
  const bool ln = norm == FNORM_LAYERNORM;
  if (!ln && mean_out != nullptr) return bad("mean_out is only defined for LayerNorm");
  if (ln && colsum == nullptr) return bad("LayerNorm needs the column sums of the folded B (colsum)");
  if (M == 0) return FNORM_OK;
  FN_TRY(check_ptr(A, "A", 16, false));
  FN_TRY(check_ptr(B_folded, "B_folded", 16, false));
  FN_TRY(check_ptr(C, "C", 16, false));
  FN_TRY(check_ptr(colsum, "colsum", 16, true));
  FN_TRY(check_ptr(bias, "bias", 16, true));
  FN_TRY(check_ptr(mean_out, "mean_out", 4, true));
  FN_TRY(check_ptr(rstd_out, "rstd_out", 4, true));
  FusedLaunch L = base_launch(A, B_folded, C, M, N, K, stream);
  L.bn = gemm_tile_n(N);
  L.bres = want_resident_b(M, N, K, L.bn);
  L.pre_eps = eps;
  L.rstd_out = rstd_out;
  if (!ln && bias == nullptr) {
    // RMSNorm with gamma only: the folded B makes it the plain lazy pre-norm
    L.mode = MODE_PRE;
    if (want_pair(L.bn, L.bres)) return launch_fused_pair(L);
    if (want_mcb(M, L.bn, L.bres)) return launch_fused_mcb(L);
    return launch_fused_plain(L);
  }
  L.mode = MODE_PRE | MODE_AFF | (ln ? MODE_PRE_LN : 0);
  L.colsum = ln ? colsum : nullptr;
  L.bias = bias;
  L.mean_out = ln ? mean_out : nullptr;
  if (want_pair(L.bn, L.bres)) return launch_fused_pair(L);
  if (want_mcb(M, L.bn, L.bres)) return launch_fused_mcb(L);
  return launch_fused_prenorm_affine(L);
}

fnorm_status_t fnorm_gemm_add_postnorm(const fnorm_bf16* A, const fnorm_bf16* B, const fnorm_bf16* R, fnorm_bf16* C,
                                       int64_t M, int64_t N, int64_t K, fnorm_norm_t norm, const fnorm_bf16* gamma,
                                       const fnorm_bf16* beta, float eps, float* mean_out, float* rstd_out,
                                       void* stream) {
  clear_error();
  FN_TRY(check_mnk(M, N, K));
  if (norm != FNORM_RMSNORM && norm != FNORM_LAYERNORM) return bad("norm must be FNORM_RMSNORM or FNORM_LAYERNORM");
  FN_TRY(check_eps(eps, "eps"));
  if (norm == FNORM_RMSNORM && mean_out != nullptr) return bad("mean_out is only defined for LayerNorm");
  PostPlan plan{};
  FN_TRY(plan_postnorm(N, forced_postnorm_cluster(), &plan, false));
  if (M == 0) return FNORM_OK;
  FN_TRY(check_ptr(A, "A", 16, false));
  FN_TRY(check_ptr(B, "B", 16, false));
  FN_TRY(check_ptr(R, "R", 16, false));
  FN_TRY(check_ptr(C, "C", 16, false));
  FN_TRY(check_ptr(gamma, "gamma", 16, true));
  FN_TRY(check_ptr(beta, "beta", 16, true));
  FN_TRY(check_ptr(mean_out, "mean_out", 4, true));
  FN_TRY(check_ptr(rstd_out, "rstd_out", 4, true));
  {
    const auto r0 = reinterpret_cast<uintptr_t>(R), c0 = reinterpret_cast<uintptr_t>(C);
    const uintptr_t bytes = static_cast<uintptr_t>(M) * static_cast<uintptr_t>(N) * 2u;
    if (r0 < c0 + bytes && c0 < r0 + bytes) return bad("R must not overlap C");
  }
  FusedLaunch L = base_launch(A, B, C, M, N, K, stream);
  L.mode = MODE_POST | MODE_RES | (norm == FNORM_LAYERNORM ? MODE_LN : 0);
  L.bn = plan.bn;
  L.slices = plan.slices;
  L.spill = plan.spill;
  L.cluster = plan.cluster;
  L.bres = (plan.cluster == 1 && !plan.spill) && want_resident_b(M, N, K, plan.bn);
  L.eps = eps;
  L.gamma = gamma;
  L.beta = beta;
  L.mean_out = mean_out;
  L.rstd_out = rstd_out;
  L.R = R;
  return (plan.cluster == 1 && !plan.spill) ? launch_fused_post_residual(L) : launch_fused_post_residual_cluster(L);
}

fnorm_status_t fnorm_lazy_prenorm_gemm_backward(const fnorm_bf16* A, const fnorm_bf16* B, const fnorm_bf16* C,
                                                const fnorm_bf16* dC, const float* rstd, fnorm_bf16* dA,
                                                fnorm_bf16* dB, fnorm_bf16* dCs, float* rowcoef, int64_t M,
                                                int64_t N, int64_t K, void* stream) {
  clear_error();
  FN_TRY(check_mnk(M, N, K));
  if (dA == nullptr && dB == nullptr) return bad("at least one of dA, dB must be given");
  FN_TRY(check_ptr(dA, "dA", 16, true));
  FN_TRY(check_ptr(dB, "dB", 16, true));
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (M == 0) {
    // an empty batch contributes nothing: dB = 0
    if (dB != nullptr) {
      cudaError_t e = cudaMemsetAsync(dB, 0, static_cast<size_t>(K) * static_cast<size_t>(N) * 2, st);
      if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(dB)");
    }
    return FNORM_OK;
  }
  if (M % 8 != 0 && dB != nullptr) return bad("dB needs M to be a multiple of 8 (the [M, K] rows are read as A^T)");
  FN_TRY(check_ptr(A, "A", 16, false));
  FN_TRY(check_ptr(B, "B", 16, dA == nullptr));
  FN_TRY(check_ptr(C, "C", 16, false));
  FN_TRY(check_ptr(dC, "dC", 16, false));
  FN_TRY(check_ptr(rstd, "rstd", 4, false));
  FN_TRY(check_ptr(dCs, "dCs", 16, false));
  FN_TRY(check_ptr(rowcoef, "rowcoef", 4, false));
  {
    const auto a0 = reinterpret_cast<uintptr_t>(dCs), b0 = reinterpret_cast<uintptr_t>(dC);
    const uintptr_t bytes = static_cast<uintptr_t>(M) * static_cast<uintptr_t>(N) * 2u;
    if (a0 < b0 + bytes && b0 < a0 + bytes) return bad("dCs must not overlap dC");
  }
  // one pass over the rows: dCs = rstd * dC, rowcoef = -rstd^2 (dC . C) / K
  FN_TRY(launch_backward_rows(dC, C, rstd, dCs, rowcoef, static_cast<int>(M), static_cast<int>(N),
                              static_cast<int>(K), st));
  if (dA != nullptr) {
    // dA [M,K] = dCs @ B^T + rowcoef * A: a GEMM over N with the RMSNorm
    // backward's row term in its epilogue
    FusedLaunch L = base_launch(dCs, B, dA, M, K, N, stream);
    L.mode = MODE_DGRAD | MODE_BT;
    L.bn = fill_tile_n(M, K);
    L.X = A;
    L.rowcoef = rowcoef;
    FN_TRY(want_mcb(M, L.bn, false) ? launch_fused_transposed_mcb(L) : launch_fused_backward(L));
  }
  if (dB != nullptr) {
    // dB [K,N] = A^T @ dCs: a GEMM over M reading A^T straight from A
    FusedLaunch L = base_launch(A, dCs, dB, K, N, M, stream);
    L.mode = MODE_AT;
    L.bn = fill_tile_n(K, N);
    FN_TRY(want_mcb(K, L.bn, false) ? launch_fused_transposed_mcb(L) : launch_fused_transposed(L));
  }
  return FNORM_OK;
}

fnorm_status_t fnorm_gemm_postnorm_backward(const fnorm_bf16* A, const fnorm_bf16* B, const fnorm_bf16* C,
                                           const fnorm_bf16* dC, fnorm_norm_t norm, const fnorm_bf16* gamma,
                                           const fnorm_bf16* beta, const float* rstd, fnorm_bf16* dA, fnorm_bf16* dB,
                                           float* dgamma, float* dbeta, fnorm_bf16* dH, float* part, int64_t M,
                                           int64_t N, int64_t K, void* stream) {
  clear_error();
  FN_TRY(check_mnk(M, N, K));
  if (norm != FNORM_RMSNORM && norm != FNORM_LAYERNORM) return bad("norm must be FNORM_RMSNORM or FNORM_LAYERNORM");
  if (dA == nullptr && dB == nullptr && dgamma == nullptr && dbeta == nullptr && dH == nullptr)
    return bad("no gradient asked for");
  FN_TRY(check_ptr(dA, "dA", 16, true));
  FN_TRY(check_ptr(dB, "dB", 16, true));
  FN_TRY(check_ptr(dgamma, "dgamma", 4, true));
  FN_TRY(check_ptr(dbeta, "dbeta", 4, true));
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool need_dh = dA != nullptr || dB != nullptr || dH != nullptr;
  const bool need_cols = dgamma != nullptr || dbeta != nullptr;
  if (M == 0) {
    // an empty batch: zero dB, dgamma, dbeta
    struct Z {
      void* p;
      size_t n;
    } z[3] = {{dB, static_cast<size_t>(K) * N * 2}, {dgamma, static_cast<size_t>(N) * 4},
              {dbeta, static_cast<size_t>(N) * 4}};
    for (auto& e : z)
      if (e.p != nullptr) {
        cudaError_t err = cudaMemsetAsync(e.p, 0, e.n, st);
        if (err != cudaSuccess) return cuda_fail(err, "cudaMemsetAsync");
      }
    return FNORM_OK;
  }
  if (dB != nullptr && M % 8 != 0) return bad("dB needs M to be a multiple of 8 (dH is read transposed)");
  FN_TRY(check_ptr(A, "A", 16, dB == nullptr));
  FN_TRY(check_ptr(B, "B", 16, dA == nullptr));
  FN_TRY(check_ptr(C, "C", 16, false));
  FN_TRY(check_ptr(dC, "dC", 16, false));
  FN_TRY(check_ptr(gamma, "gamma", 16, true));
  FN_TRY(check_ptr(beta, "beta", 16, true));
  FN_TRY(check_ptr(rstd, "rstd", 4, !need_dh));
  FN_TRY(check_ptr(dH, "dH", 16, dA == nullptr && dB == nullptr));
  FN_TRY(check_ptr(part, "part", 16, !need_cols));
  FN_TRY(launch_postnorm_backward_rows(dC, C, gamma, beta, rstd, norm == FNORM_LAYERNORM, need_dh ? dH : nullptr,
                                       part, dgamma, dbeta, static_cast<int>(M), static_cast<int>(N), st));
  if (dA != nullptr) FN_TRY(fnorm_gemm_ex(dH, B, dA, M, K, N, 0, 1, stream));   // dH @ B^T
  if (dB != nullptr) FN_TRY(fnorm_gemm_ex(A, dH, dB, K, N, M, 1, 0, stream));   // A^T @ dH
  return FNORM_OK;
}

fnorm_status_t fnorm_gemm_postnorm_backward_regrouped(const fnorm_bf16* G, const fnorm_bf16* W, int64_t J,
                                                     int trans_w, const fnorm_bf16* A, const fnorm_bf16* B,
                                                     const fnorm_bf16* C, fnorm_norm_t norm,
                                                     const fnorm_bf16* gamma, const fnorm_bf16* beta,
                                                     const float* rstd, fnorm_bf16* dA, fnorm_bf16* dB,
                                                     float* dgamma, float* dbeta, fnorm_bf16* dH, float* part,
                                                     void* workspace, size_t workspace_bytes, int64_t M, int64_t N,
                                                     int64_t K, void* stream) {
  clear_error();
  FN_TRY(check_mnk(M, N, K));
  if (J < 8 || J > kMaxDim || J % 8 != 0) return bad("J must be a multiple of 8 in [8, 2^31)");
  if (trans_w != 0 && trans_w != 1) return bad("trans_w must be 0 or 1");
  if (norm != FNORM_RMSNORM && norm != FNORM_LAYERNORM) return bad("norm must be FNORM_RMSNORM or FNORM_LAYERNORM");
  FN_TRY(check_ptr(dA, "dA", 16, true));
  FN_TRY(check_ptr(dB, "dB", 16, true));
  FN_TRY(check_ptr(dgamma, "dgamma", 4, true));
  FN_TRY(check_ptr(dbeta, "dbeta", 4, true));
  // rows of up to 256 columns in one CTA's tile; up to 1024 over a cluster
  // of 2 or 4 CTAs of 256 columns (the two row sums exchanged through
  // distributed shared memory); wider rows in one-CTA tiles of 256 columns
  // with the row sums exchanged grid-wide through the caller's workspace
  const int forced = forced_postnorm_cluster();
  const bool gx = forced == 0 && N > 1024;
  const int c = forced != 0 ? forced : (N <= 256 ? 1 : (N <= 512 ? 2 : 4));
  if (!gx && ((c != 1 && c != 2 && c != 4) || (N + c - 1) / c > 256)) {
    set_error("a cluster size forced to %d does not fit the regrouped post-norm backward of %lld columns (1, 2 or 4 "
              "CTAs of at most 256 columns)", c, (long long)N);
    return FNORM_ERR_UNSUPPORTED;
  }
  GxScratch gxs{};
  if (gx) {
    if (workspace == nullptr) {
      set_error("rows of %lld columns: the regrouped post-norm backward exchanges their row sums grid-wide and needs "
                "a workspace of fnorm_postnorm_workspace_size(M, N) bytes", (long long)N);
      return FNORM_ERR_UNSUPPORTED;
    }
    if ((M + 127) / 128 > kGxMaxRowBlocks) {
      set_error("the regrouped post-norm backward's grid exchange takes at most %d row blocks of 128", kGxMaxRowBlocks);
      return FNORM_ERR_UNSUPPORTED;
    }
    FN_TRY(gx_scratch_from(workspace, workspace_bytes, M, N, &gxs));
  }
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool cols = dgamma != nullptr || dbeta != nullptr;
  if (M == 0) {
    // an empty batch: zero dB, dgamma, dbeta
    struct Z {
      void* p;
      size_t n;
    } z[3] = {{dB, static_cast<size_t>(K) * N * 2}, {dgamma, static_cast<size_t>(N) * 4},
              {dbeta, static_cast<size_t>(N) * 4}};
    for (auto& e : z)
      if (e.p != nullptr) {
        cudaError_t err = cudaMemsetAsync(e.p, 0, e.n, st);
        if (err != cudaSuccess) return cuda_fail(err, "cudaMemsetAsync");
      }
    return FNORM_OK;
  }
  if (dB != nullptr && M % 8 != 0) return bad("dB needs M to be a multiple of 8 (dH is read transposed)");
  FN_TRY(check_ptr(G, "G", 16, false));
  FN_TRY(check_ptr(W, "W", 16, false));
  FN_TRY(check_ptr(A, "A", 16, dB == nullptr));
  FN_TRY(check_ptr(B, "B", 16, dA == nullptr));
  FN_TRY(check_ptr(C, "C", 16, false));
  FN_TRY(check_ptr(gamma, "gamma", 16, true));
  FN_TRY(check_ptr(beta, "beta", 16, true));
  FN_TRY(check_ptr(rstd, "rstd", 4, false));
  FN_TRY(check_ptr(dH, "dH", 16, false));
  FN_TRY(check_ptr(part, "part", 16, !cols));
  if (gx) {
    // one CTA per tile of a row at least (no CTA may hold two tiles of the
    // row block it waits on)
    DeviceInfo dev;
    FN_TRY(current_device(&dev));
    if ((N + 255) / 256 > dev.num_sms) {
      set_error("a row of %lld columns has more 256-column tiles than the device has SMs (%d)", (long long)N,
                dev.num_sms);
      return FNORM_ERR_UNSUPPORTED;
    }
  }
  // dC = G @ op(W)^T in the accumulator: W [N, J] is the B^T operand, W [J, N] the plain one
  FusedLaunch L = base_launch(G, W, dH, M, N, J, stream);
  L.mode = MODE_POST | MODE_NBWD | (norm == FNORM_LAYERNORM ? MODE_LN : 0) | (trans_w ? 0 : MODE_BT);
  L.cluster = gx ? 1 : c;
  L.bn = (!gx && c == 1 && N <= 128) ? 128 : 256;
  L.gx = gx ? &gxs : nullptr;
  L.gamma = gamma;
  L.beta = beta;
  L.X = C;
  L.rstd_in = rstd;
  L.cpart = cols ? part : nullptr;
  FN_TRY(launch_fused_norm_backward(L));
  if (cols) FN_TRY(launch_column_sum(part, static_cast<int>((M + 31) / 32), static_cast<int>(N), dgamma, dbeta, st));
  if (dA != nullptr) FN_TRY(fnorm_gemm_ex(dH, B, dA, M, K, N, 0, 1, stream));   // dH @ B^T
  if (dB != nullptr) FN_TRY(fnorm_gemm_ex(A, dH, dB, K, N, M, 1, 0, stream));   // A^T @ dH
  return FNORM_OK;
}

fnorm_status_t fnorm_rmsnorm(const fnorm_bf16* X, fnorm_bf16* Y, int64_t M, int64_t N, const fnorm_bf16* gamma,
                             float eps, float* rstd_out, void* stream) {
  clear_error();
  if (M < 0 || M > kMaxDim) return bad("M must be in [0, 2^31)");
  if (N < 8 || N % 8 != 0 || N > 32768) return bad("N must be a multiple of 8 in [8, 32768]");
  FN_TRY(check_eps(eps, "eps"));
  if (M == 0) return FNORM_OK;
  FN_TRY(check_ptr(X, "X", 16, false));
  FN_TRY(check_ptr(Y, "Y", 16, false));
  FN_TRY(check_ptr(gamma, "gamma", 16, true));
  FN_TRY(check_ptr(rstd_out, "rstd_out", 4, true));
  return launch_rownorm(X, nullptr, Y, static_cast<int>(M), static_cast<int>(N), false, gamma, nullptr, eps, nullptr,
                        rstd_out, static_cast<cudaStream_t>(stream));
}

fnorm_status_t fnorm_layernorm(const fnorm_bf16* X, fnorm_bf16* Y, int64_t M, int64_t N, const fnorm_bf16* gamma,
                               const fnorm_bf16* beta, float eps, float* mean_out, float* rstd_out,
                               void* stream) {
  clear_error();
  if (M < 0 || M > kMaxDim) return bad("M must be in [0, 2^31)");
  if (N < 8 || N % 8 != 0 || N > 32768) return bad("N must be a multiple of 8 in [8, 32768]");
  FN_TRY(check_eps(eps, "eps"));
  if (M == 0) return FNORM_OK;
  FN_TRY(check_ptr(X, "X", 16, false));
  FN_TRY(check_ptr(Y, "Y", 16, false));
  FN_TRY(check_ptr(gamma, "gamma", 16, true));
  FN_TRY(check_ptr(beta, "beta", 16, true));
  FN_TRY(check_ptr(mean_out, "mean_out", 4, true));
  FN_TRY(check_ptr(rstd_out, "rstd_out", 4, true));
  return launch_rownorm(X, nullptr, Y, static_cast<int>(M), static_cast<int>(N), true, gamma, beta, eps, mean_out,
                        rstd_out, static_cast<cudaStream_t>(stream));
}

fnorm_status_t fnorm_add_rownorm(const fnorm_bf16* X, const fnorm_bf16* R, fnorm_bf16* Y, int64_t M, int64_t N,
                                 fnorm_norm_t norm, const fnorm_bf16* gamma, const fnorm_bf16* beta, float eps,
                                 float* mean_out, float* rstd_out, void* stream) {
  clear_error();
  if (M < 0 || M > kMaxDim) return bad("M must be in [0, 2^31)");
  if (N < 8 || N % 8 != 0 || N > 32768) return bad("N must be a multiple of 8 in [8, 32768]");
  if (norm != FNORM_RMSNORM && norm != FNORM_LAYERNORM) return bad("norm must be FNORM_RMSNORM or FNORM_LAYERNORM");
  FN_TRY(check_eps(eps, "eps"));
  if (norm == FNORM_RMSNORM && mean_out != nullptr) return bad("mean_out is only defined for LayerNorm");
  if (M == 0) return FNORM_OK;
  FN_TRY(check_ptr(X, "X", 16, false));
  FN_TRY(check_ptr(R, "R", 16, false));
  FN_TRY(check_ptr(Y, "Y", 16, false));
  FN_TRY(check_ptr(gamma, "gamma", 16, true));
  FN_TRY(check_ptr(beta, "beta", 16, true));
  FN_TRY(check_ptr(mean_out, "mean_out", 4, true));
  FN_TRY(check_ptr(rstd_out, "rstd_out", 4, true));
  return launch_rownorm(X, R, Y, static_cast<int>(M), static_cast<int>(N), norm == FNORM_LAYERNORM, gamma, beta,
                        eps, mean_out, rstd_out, static_cast<cudaStream_t>(stream));
}

fnorm_status_t fnorm_rmsnorm_backward(const fnorm_bf16* dY, const fnorm_bf16* X, const float* rstd, fnorm_bf16* dX,
                                     int64_t M, int64_t N, void* stream) {
  clear_error();
  if (M < 0 || M > kMaxDim) return bad("M must be in [0, 2^31)");
  if (N < 8 || N % 8 != 0 || N > 16384) return bad("N must be a multiple of 8 in [8, 16384]");
  if (M == 0) return FNORM_OK;
  FN_TRY(check_ptr(dY, "dY", 16, false));
  FN_TRY(check_ptr(X, "X", 16, false));
  FN_TRY(check_ptr(rstd, "rstd", 4, false));
  FN_TRY(check_ptr(dX, "dX", 16, false));
  return launch_rmsnorm_backward(dY, X, rstd, dX, static_cast<int>(M), static_cast<int>(N),
                                 static_cast<cudaStream_t>(stream));
}

fnorm_status_t fnorm_check_status(void* stream) {
  clear_error();
  return read_and_clear_status(static_cast<cudaStream_t>(stream));
}

const char* fnorm_last_error(void) { return last_error_cstr(); }

fnorm_status_t fnorm_set_wait_limit_ns(uint64_t ns) {
  clear_error();
  if (ns == 0) ns = 2000000000ull;
  if (ns < 1000ull) ns = 1000ull;
  if (ns > 60000000000ull) ns = 60000000000ull;
  set_wait_limit(ns);
  return FNORM_OK;
}

fnorm_status_t fnorm_postnorm_plan(int64_t N, int* cluster, int* cols_per_cta) {
  clear_error();
  if (cluster == nullptr || cols_per_cta == nullptr) return bad("output pointers must not be NULL");
  if (N < 8 || N > kMaxDim || N % 8 != 0) return bad("N must be a multiple of 8 in [8, 2^31)");
  PostPlan plan{};
  FN_TRY(plan_postnorm(N, forced_postnorm_cluster(), &plan, false));
  *cluster = plan.cluster;
  *cols_per_cta = plan.bn * plan.slices;
  return FNORM_OK;
}

fnorm_status_t fnorm_set_postnorm_cluster(int cluster_size) {
  clear_error();
  if (cluster_size != 0 && cluster_size != 1 && cluster_size != 2 && cluster_size != 4 && cluster_size != 8)
    return bad("cluster size must be 0 (automatic), 1, 2, 4 or 8");
  g_forced_cluster.store(cluster_size, std::memory_order_relaxed);
  return FNORM_OK;
}

fnorm_status_t fnorm_set_pair_mma(int mode) {
  clear_error();
  if (mode < -1 || mode > 1) return bad("pair MMA mode must be -1 (automatic), 0 (never) or 1 (whenever eligible)");
  g_pair_mode.store(mode, std::memory_order_relaxed);
  return FNORM_OK;
}

fnorm_status_t fnorm_set_b_multicast(int mode) {
  clear_error();
  if (mode < -1 || mode > 1) return bad("B multicast mode must be -1 (automatic), 0 (never) or 1 (whenever eligible)");
  g_mcb_mode.store(mode, std::memory_order_relaxed);
  return FNORM_OK;
}

fnorm_status_t fnorm_debug_wait_timeout(uint64_t limit_ns, void* stream) {
  clear_error();
  if (limit_ns < 1000ull) limit_ns = 1000ull;
  if (limit_ns > 10000000000ull) limit_ns = 10000000000ull;
  return launch_wait_timeout_selftest(limit_ns, static_cast<cudaStream_t>(stream));
}

fnorm_status_t fnorm_debug_cluster_shape(int cluster, void* stream) {
  clear_error();
  if (cluster != 1 && cluster != 2) return bad("cluster must be 1 or 2");
  return launch_cluster_shape_selftest(cluster, static_cast<cudaStream_t>(stream));
}

int fnorm_version(void) { return 100; }

}  // extern "C"
