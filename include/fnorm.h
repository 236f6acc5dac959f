/*
 * fnorm.h — C ABI of libfnorm: row normalization fused into a tcgen05 GEMM
 * on GB300 (sm_103a).
 *
 * Sources, cited by page title and section:
 *   [FNF-ru] "Free normalization fusion" (aixai.ru blog, Russian summary of
 *            the PyTorch post "Towards Free Normalization").
 *   [FNF-es] "PyTorch: normalización casi gratis fusionando kernels"
 *            (noticias.mechatronicstore.cl).
 *   [TFN]    "Towards Free Normalization: Fusing Normalization into GEMM and
 *            Attention Kernels – PyTorch" (news.8syncdev.com abstract).
 *   [ATB]    Ascend ATB RMSNorm-fusion article (gsyq.cn), sections 1.1-1.2
 *            (textbook LayerNorm and RMSNorm definitions).
 *
 * Conventions shared by every entry point
 *   - Matrices are row-major and contiguous.  A is [M,K], B is [K,N],
 *     C is [M,N], X and Y are [M,N].  Element type is bfloat16, passed as its
 *     16-bit storage (fnorm_bf16).  Accumulation is fp32; row statistics are
 *     fp32 arrays of length M.
 *   - Every pointer is DEVICE memory on the current CUDA device, owned by
 *     the caller.  The library never frees or retains caller memory, and no
 *     call allocates device memory or synchronises the host (except
 *     fnorm_check_status, whose job is to synchronise).  Workspaces are the
 *     caller's and passed in (fnorm_gemm_postnorm_ws and the backward
 *     entry points).  Base addresses of A, B, C, X, Y, gamma and beta must be 16-byte
 *     aligned; fp32 statistic outputs 4-byte aligned.  A misaligned pointer
 *     is an argument error.
 *   - Sizes: M >= 0 (M == 0 is a valid empty call that does nothing);
 *     N >= 8 and K >= 8, both multiples of 8 (16-byte row pitch for the
 *     tensor-memory-access engine); M, N, K < 2^31.
 *   - eps > 0 and finite.
 *   - stream is a cudaStream_t (NULL = the legacy default stream).  Calls are
 *     asynchronous on that stream: no host synchronisation happens inside
 *     them and they can be captured into a CUDA graph after the first call on
 *     a device has returned (that first call loads the device code).  Kernels
 *     are launched with programmatic stream serialisation: their set-up may
 *     overlap the previous kernel in the stream, and every global memory
 *     access waits for that kernel to complete (environment variable
 *     FNORM_PDL=0 turns this off), except the cooperative grid exchange.
 *   - Profiling: profilers that replay a cooperative launch of clusters run
 *     it without its clusters; set FNORM_PLAIN_GX_LAUNCH=1 when profiling
 *     wide-row post-norms (fnorm_gemm_postnorm_ws).  Every clustered kernel
 *     checks its cluster size first, so a mismatch is reported
 *     (fnorm_check_status: FNORM_ERR_CUDA), never run.
 *   - A call returns FNORM_OK once its kernels are enqueued.  Argument errors
 *     return FNORM_ERR_INVALID_ARG and launch nothing; shapes the kernels do
 *     not implement return FNORM_ERR_UNSUPPORTED; CUDA launch errors return
 *     FNORM_ERR_CUDA.  fnorm_last_error() then describes the failure.
 *   - Every wait inside the kernels is bounded (fnorm_set_wait_limit_ns).  A
 *     wait that runs out makes the kernel stop early and record a device
 *     status word; fnorm_check_status() reports it as FNORM_ERR_TIMEOUT.
 *   - NaN and Inf inputs are not supported (results are unspecified).
 */
#ifndef FNORM_H
#define FNORM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t fnorm_bf16;  /* bfloat16 storage */

typedef enum {
  FNORM_OK = 0,
  FNORM_ERR_INVALID_ARG = 1,
  FNORM_ERR_UNSUPPORTED = 2,
  FNORM_ERR_CUDA = 3,
  FNORM_ERR_TIMEOUT = 4
} fnorm_status_t;

typedef enum {
  FNORM_RMSNORM = 0,
  FNORM_LAYERNORM = 1
} fnorm_norm_t;

/*
 * fnorm_gemm — C = A @ B, bf16 in and out, fp32 accumulate.
 *   The plain tiled GEMM ([FNF-ru] "Why normalization is a performance
 *   problem": the GEMM tiles over M and N, so no tile sees a whole row).  It
 *   shares the tcgen05 mainloop with the fused kernels and is the GEMM half
 *   of the unfused comparison.
 */
fnorm_status_t fnorm_gemm(const fnorm_bf16* A, const fnorm_bf16* B, fnorm_bf16* C,
                          int64_t M, int64_t N, int64_t K, void* stream);

/*
 * fnorm_gemm_ex — C = op(A) @ op(B), C [M,N], bf16 in and out, fp32 accumulate.
 *   op(A) is A [M,K] (trans_a = 0) or the transpose of a [K,M] array
 *   (trans_a = 1, read MN-major straight from its row-major layout; M must then
 *   be a multiple of 8); op(B) is B [K,N] (trans_b = 0) or the transpose of an
 *   [N,K] array (trans_b = 1, read K-major).  The same tcgen05 mainloop as
 *   fnorm_gemm; the GEMM half of the backward's unfused comparison
 *   (dC @ B^T, A_hat^T @ dC).
 */
fnorm_status_t fnorm_gemm_ex(const fnorm_bf16* A, const fnorm_bf16* B, fnorm_bf16* C, int64_t M, int64_t N,
                             int64_t K, int trans_a, int trans_b, void* stream);

/*
 * fnorm_lazy_prenorm_gemm — C = rmsnorm(A) @ B, RMSNorm without affine,
 * computed as (A @ B) * rstd(A).
 *   [FNF-ru] "Lazy Pre-Norm"; [FNF-es] "Lazy Pre-Norm: el truco matemático".
 *   rstd[m] = 1 / sqrt((1/K) * sum_k A[m,k]^2 + eps), summed in fp32 from the
 *   A tiles already staged in shared memory while the tensor cores run, and
 *   applied to the fp32 accumulator before the bf16 rounding of C.
 *   rstd_out: [M] fp32 device array, or NULL to skip it.
 *   There is deliberately no gamma/beta: a per-column affine does not commute
 *   with the GEMM ([FNF-ru] "Lazy Pre-Norm" limits and FAQ).
 */
fnorm_status_t fnorm_lazy_prenorm_gemm(const fnorm_bf16* A, const fnorm_bf16* B, fnorm_bf16* C,
                                       int64_t M, int64_t N, int64_t K, float eps,
                                       float* rstd_out, void* stream);

/*
 * fnorm_gemm_postnorm — C = norm(A @ B) * gamma + beta (epilogue post-norm).
 *   [FNF-ru] "Multi-CTA Norm Fusion"; [FNF-es] "El problema del tiling";
 *   definitions from [ATB] 1.1 (LayerNorm, biased variance) and 1.2 (RMSNorm).
 *   The row statistics are taken over the fp32 accumulator of each row.  When
 *   N is wider than one CTA's tile, the CTAs of a thread-block cluster that
 *   share a 128-row block split the row along N, exchange per-row partial
 *   statistics through distributed shared memory and each normalises its own
 *   slice (fnorm_postnorm_plan reports the split).  Rows wider than the
 *   cluster's tensor memory (N > 1024 by default) use a spill layout: each
 *   CTA of a 4-CTA cluster writes its un-normalised slices to C in bf16, then
 *   normalises them in place once the statistics are known; those outputs
 *   are normalised from bf16-rounded values (relative error <= 2^-9 of the
 *   value before the norm), and C is therefore also read by this call.  This
 *   entry point needs no workspace; fnorm_gemm_postnorm_ws takes one and
 *   computes wide rows faster, without the spill.
 *   norm:        FNORM_LAYERNORM or FNORM_RMSNORM.
 *   gamma, beta: [N] bf16 device arrays, or NULL (gamma = 1, beta = 0).
 *   eps:         epsilon of the post-norm, inside the square root.
 *   pre_rmsnorm: 0 or 1.  With 1 the kernel first applies a lazy pre-RMSNorm
 *                of A without affine (epsilon pre_eps), i.e. it computes
 *                norm(rmsnorm(A) @ B) in one kernel; pre_eps is ignored with 0.
 *   mean_out:    [M] fp32, LayerNorm only (must be NULL for RMSNorm), or NULL.
 *   rstd_out:    [M] fp32 rstd of the post-norm, or NULL.
 *   pre_rstd_out:[M] fp32 rstd of the pre-norm (pre_rmsnorm == 1 only), or NULL.
 */
fnorm_status_t fnorm_gemm_postnorm(const fnorm_bf16* A, const fnorm_bf16* B, fnorm_bf16* C,
                                   int64_t M, int64_t N, int64_t K, fnorm_norm_t norm,
                                   const fnorm_bf16* gamma, const fnorm_bf16* beta, float eps,
                                   int pre_rmsnorm, float pre_eps,
                                   float* mean_out, float* rstd_out, float* pre_rstd_out,
                                   void* stream);

/*
 * fnorm_gemm_postnorm_ws — fnorm_gemm_postnorm with a caller-owned workspace
 * for the statistics exchange of wide rows.
 *   [FNF-ru] "Multi-CTA Norm Fusion" (the CTAs that share a row combine one
 *   pair of scalars per row), with the exchange made grid-wide: for a row of
 *   more than 1024 columns, every 256-column tile of the plain GEMM stays in
 *   tensor memory; the tiles of a 128-row block, on any CTAs of the grid,
 *   publish their per-row partial statistics (mean and sum of squared
 *   deviations for LayerNorm, sum of squares for RMSNorm) to the workspace
 *   and count in on the row block's counter; each tile then combines all of
 *   them in tile order (so every tile of a row derives the same statistics)
 *   and normalises itself straight from the fp32 accumulator.  Nothing is
 *   written to C before it is normalised.  All CTAs of the kernel must be
 *   resident at once, so it is a cooperative launch, which the driver
 *   starts only when all of its CTAs fit; for more than one row block the
 *   tiles of two neighbouring row blocks share B over a 2-CTA cluster
 *   (fnorm_set_b_multicast).  Profilers that replay a cooperative launch of
 *   clusters run it without its clusters; the kernel then writes nothing
 *   and fnorm_check_status reports FNORM_ERR_CUDA.  With the environment
 *   variable FNORM_PLAIN_GX_LAUNCH=1 (read once per process) the clustered
 *   form is a plain cluster launch instead, which profilers replay as
 *   launched; its CTAs are all resident once the kernels before it in the
 *   stream have finished, but work on other streams that holds SMs past the
 *   wait limit (another such call, for instance) makes it end in
 *   FNORM_ERR_TIMEOUT.  A row of more tiles than the device has SMs
 *   (N > 256 * SMs) or more than 2^21 rows take fnorm_gemm_postnorm's spill
 *   layout instead, as do rows of at most 1024 columns, which need no
 *   workspace.
 *   workspace:       device memory of at least workspace_bytes, 16-byte
 *                    aligned, owned by the caller, or NULL (then this is
 *                    fnorm_gemm_postnorm).  fnorm_postnorm_workspace_size
 *                    gives the bytes an M x N call needs (0: none used).  It
 *                    must be zero-filled before its first use (for instance
 *                    cudaMemsetAsync on the calls' stream); each call leaves
 *                    its counters zero again, so it is cleared once, not per
 *                    call.  Calls that share a
 *                    workspace must not overlap in time (order them on one
 *                    stream); after a call that ended in FNORM_ERR_TIMEOUT
 *                    it must be cleared again.
 *   workspace_bytes: its size; smaller than the call needs is
 *                    FNORM_ERR_INVALID_ARG.
 *   Other arguments and results as fnorm_gemm_postnorm.
 */
fnorm_status_t fnorm_gemm_postnorm_ws(const fnorm_bf16* A, const fnorm_bf16* B, fnorm_bf16* C,
                                      int64_t M, int64_t N, int64_t K, fnorm_norm_t norm,
                                      const fnorm_bf16* gamma, const fnorm_bf16* beta, float eps,
                                      int pre_rmsnorm, float pre_eps,
                                      float* mean_out, float* rstd_out, float* pre_rstd_out,
                                      void* workspace, size_t workspace_bytes, void* stream);

/*
 * fnorm_postnorm_workspace_size — bytes of the workspace fnorm_gemm_postnorm_ws
 * uses for an M x N post-norm, into *bytes: 256 + 8 * 16384 (a header and
 * the counters of up to 16384 row blocks, at the same place whatever the
 * call's shape) plus 1024 per (128-row block, 256-column tile); 0 when the
 * call needs no exchange workspace (N <= 1024, M == 0, M > 2^21 rows, or a
 * forced cluster size).  A workspace sized for M x N serves every call with
 * at most as many (row block, tile) pairs, whatever their shapes.  Host only;
 * launches nothing.
 */
fnorm_status_t fnorm_postnorm_workspace_size(int64_t M, int64_t N, size_t* bytes);

/*
 * fnorm_lazy_prenorm_gemm_backward — gradients of C = rmsnorm(A) @ B
 * (fnorm_lazy_prenorm_gemm) with respect to A and B, given dC = dL/dC:
 *   dB = (A * rstd)^T @ dC = A^T @ (rstd * dC)                      [K,N]
 *   dA = rstd * (dC @ B^T) - rstd^2 * (dC . C) / K * A              [M,K]
 *   with rstd the forward's row rstd and (dC . C) the dot of row m of dC with
 *   row m of the forward output C.  [FNF-ru] "Lazy Pre-Norm" limits (the
 *   forward never materialises the normalised A, so the backward has to
 *   rebuild it) and [TFN] (fusion regrouping: the backward's norm work rides
 *   on the GEMMs).  The second term of dA is the RMSNorm backward,
 *   r^3 * A * sum_k(dA_hat * A) / K with dA_hat = dC @ B^T, rewritten through
 *   sum_k dA_hat[m,k] A[m,k] = (dC . C)[m] / rstd[m], because C = (A @ B) * rstd.
 *   The row scale moves to dC's side (A^T @ (rstd * dC)), so the normalised A
 *   is never built; rstd * dC is rounded to bf16 once.  Three launches: one
 *   memory-bound pass over the rows of dC and C writes dCs = rstd * dC and the
 *   row coefficients; the dgrad GEMM over N reads B^T straight from B and its
 *   epilogue adds coefficient * A to the accumulator; the wgrad GEMM over M
 *   reads A^T straight from A.
 *   A:    [M,K] forward input.   B: [K,N] forward weight.
 *   C:    [M,N] forward output (bf16, as fnorm_lazy_prenorm_gemm wrote it).
 *   dC:   [M,N] gradient of the loss with respect to C.
 *   rstd: [M] fp32 forward rstd (fnorm_lazy_prenorm_gemm's rstd_out).
 *   dA:   [M,K] output, or NULL to skip it (then B may be NULL).
 *   dB:   [K,N] output, or NULL to skip it (M must then be a multiple of 8).
 *         With M == 0, dB is zeroed.
 *   dCs:  [M,N] bf16 caller-owned workspace; receives rstd * dC.  Must not
 *         overlap dC.
 *   rowcoef: [M] fp32 caller-owned workspace; receives -rstd^2 (dC . C) / K.
 *   The sizes are the forward's.  eps is not needed: rstd carries it.
 */
fnorm_status_t fnorm_lazy_prenorm_gemm_backward(const fnorm_bf16* A, const fnorm_bf16* B, const fnorm_bf16* C,
                                                const fnorm_bf16* dC, const float* rstd, fnorm_bf16* dA,
                                                fnorm_bf16* dB, fnorm_bf16* dCs, float* rowcoef, int64_t M,
                                                int64_t N, int64_t K, void* stream);

/*
 * fnorm_gemm_postnorm_noalloc — fnorm_gemm_postnorm_ws (same arguments but
 * the workspace, same results) that allocates nothing, ever, and needs no
 * workspace from the caller.  The pages have no counterpart: it exists for
 * callers that must not allocate device memory at all, not even through
 * their own allocator, and so have no workspace to hand over.
 *   The wide-row grid exchange keeps its statistics in a fixed device array
 *   of the library (2048 (row block, 256-column tile) units, 8192 row
 *   blocks: about 2.1 MB) instead of the caller's workspace.  A shape whose
 *   grid exchange needs more is rejected with FNORM_ERR_UNSUPPORTED and a
 *   message naming the limit (fnorm_gemm_postnorm and fnorm_gemm_postnorm_ws
 *   take it).  Shapes that need no exchange workspace (N <= 1024) run
 *   exactly as fnorm_gemm_postnorm.
 *   The first call on a device takes the array's address and clears its
 *   counters (on the call's stream): make it before capturing a stream into
 *   a CUDA graph.  All calls of a device share the array: calls that
 *   overlap in time (different streams, or graphs replayed concurrently)
 *   race and give wrong results; order them on one stream.
 */
fnorm_status_t fnorm_gemm_postnorm_noalloc(const fnorm_bf16* A, const fnorm_bf16* B, fnorm_bf16* C,
                                           int64_t M, int64_t N, int64_t K, fnorm_norm_t norm,
                                           const fnorm_bf16* gamma, const fnorm_bf16* beta, float eps,
                                           int pre_rmsnorm, float pre_eps, float* mean_out, float* rstd_out,
                                           float* pre_rstd_out, void* stream);

/*
 * fnorm_gemm_postnorm_backward — gradients of C = norm(A @ B) * gamma + beta
 * (fnorm_gemm_postnorm without the pre-norm) given dC = dL/dC.  The forward
 * never materialised H = A @ B; its normalised rows are rebuilt from the
 * output, h_hat = (C - beta) / gamma (every gamma must be nonzero), then with
 * dh = dC * gamma:
 *   LayerNorm: dH = rstd * (dh - mean_n(dh) - h_hat * mean_n(dh * h_hat))
 *   RMSNorm:   dH = rstd * (dh - h_hat * mean_n(dh * h_hat))
 *   dgamma = sum_m dC * h_hat;  dbeta = sum_m dC;
 *   dA = dH @ B^T;  dB = A^T @ dH.
 *   [TFN] (the backward of a post-norm fused with a GEMM through "fusion
 *   regrouping"); [ATB] 1.1, 1.2 for the norms differentiated.  One row pass
 *   (one warp per row) writes dH; a column pass and a fixed-order sum give
 *   dgamma and dbeta (deterministic); the two GEMMs read dH in place, B^T and
 *   dH^T through fnorm_gemm_ex.
 *   A, B: forward inputs; C: [M,N] forward output; dC: [M,N].
 *   gamma, beta: the forward's [N] bf16 (NULL: 1 and 0).
 *   rstd: [M] fp32 forward rstd (rstd_out).  The mean is not needed.
 *   dA [M,K], dB [K,N], dgamma [N] fp32, dbeta [N] fp32: outputs, each NULL
 *   to skip (dB needs M to be a multiple of 8; with M == 0 dB, dgamma and
 *   dbeta are zeroed).
 *   dH: [M,N] bf16, receives dH whenever given; needed with dA or dB (their
 *   GEMMs read it).
 *   part: fp32 workspace of 2 * N * ceil(M / 64) values, needed with dgamma
 *   or dbeta.
 */
fnorm_status_t fnorm_gemm_postnorm_backward(const fnorm_bf16* A, const fnorm_bf16* B, const fnorm_bf16* C,
                                           const fnorm_bf16* dC, fnorm_norm_t norm, const fnorm_bf16* gamma,
                                           const fnorm_bf16* beta, const float* rstd, fnorm_bf16* dA, fnorm_bf16* dB,
                                           float* dgamma, float* dbeta, fnorm_bf16* dH, float* part, int64_t M,
                                           int64_t N, int64_t K, void* stream);

/*
 * fnorm_gemm_postnorm_backward_regrouped — fnorm_gemm_postnorm_backward when
 * the gradient at the post-norm's output comes from the GEMM of the layer that
 * consumes it, Z = C @ op(W): dC = G @ op(W)^T with G = dL/dZ [M, J].
 *   [TFN] ("fusion regrouping": in the backward the norm is fused with a
 *   different linear layer than in the forward, so that the backward also
 *   gets an epilogue fusion).  dC is the accumulator of one fused GEMM and is
 *   never written: its epilogue rebuilds h_hat = (C - beta) / gamma from the
 *   forward output, takes the norm backward's two row sums (exchanged between
 *   the CTAs of a cluster for rows of 257 to 1024 columns, grid-wide through
 *   the workspace for wider rows, as fnorm_gemm_postnorm_ws does with the
 *   forward's statistics), writes dH, and
 *   writes per-32-row column partials of dC * h_hat and dC, which a
 *   fixed-order column sum turns into dgamma and dbeta (deterministic).  Then
 *   dA = dH @ B^T and dB = A^T @ dH as in fnorm_gemm_postnorm_backward.
 *   G: [M, J] bf16, 16-byte aligned.
 *   W: the consumer's bf16 weight, read in place as stored:
 *     trans_w = 0: W is [N, J] and the consumer computes Z = C @ W (this
 *                  library's B layout); dC = G @ W^T.
 *     trans_w = 1: W is [J, N] (a linear layer's [out, in] weight) and the
 *                  consumer computes Z = C @ W^T; dC = G @ W.
 *   J: the consumer's output width, a multiple of 8.
 *   A, B, C, norm, gamma, beta, rstd, dA, dB, dgamma, dbeta, M, N, K: as
 *   fnorm_gemm_postnorm_backward.
 *   dH: [M,N] bf16 output (always needed): receives dH.
 *   part: fp32 workspace of 2 * N * ceil(M / 32) values, needed with dgamma or
 *   dbeta.
 *   workspace, workspace_bytes: the grid exchange's workspace for rows of more
 *   than 1024 columns, exactly as fnorm_gemm_postnorm_ws's (sized by
 *   fnorm_postnorm_workspace_size(M, N), zero-filled before its first use,
 *   left zeroed by every call, calls sharing it ordered); without one such
 *   rows are FNORM_ERR_UNSUPPORTED.  Ignored (may be NULL) for narrower rows.
 *   A row of more 256-column tiles than the device has SMs, or more than 2^21
 *   rows with N > 1024, is FNORM_ERR_UNSUPPORTED.  A cluster size forced
 *   through fnorm_set_postnorm_cluster must be 1, 2 or 4 and leave at most 256
 *   columns per CTA.
 */
fnorm_status_t fnorm_gemm_postnorm_backward_regrouped(const fnorm_bf16* G, const fnorm_bf16* W, int64_t J,
                                                     int trans_w, const fnorm_bf16* A, const fnorm_bf16* B,
                                                     const fnorm_bf16* C, fnorm_norm_t norm,
                                                     const fnorm_bf16* gamma, const fnorm_bf16* beta,
                                                     const float* rstd, fnorm_bf16* dA, fnorm_bf16* dB,
                                                     float* dgamma, float* dbeta, fnorm_bf16* dH, float* part,
                                                     void* workspace, size_t workspace_bytes, int64_t M, int64_t N,
                                                     int64_t K, void* stream);

/*
 * fnorm_gemm_add_postnorm — C = norm(A @ B + R) * gamma + beta: a residual
 * added to the fp32 accumulator in the epilogue, before the post-norm's row
 * statistics.
 *   [FNF-ru] "FlashNormAttention" (a residual connection followed by a
 *   post-RMSNorm, with the tensor-core accumulator used for the addition);
 *   [ATB] 1.1 and 1.2 for the norms.  The row split over a cluster and the
 *   spill layout for wide rows are those of fnorm_gemm_postnorm; in the spill
 *   layout the bf16 values written before normalisation are A @ B + R.
 *   R:           [M,N] bf16 residual, 16-byte aligned; must not overlap C.
 *   Other arguments as fnorm_gemm_postnorm (this form has no pre-norm).
 */
fnorm_status_t fnorm_gemm_add_postnorm(const fnorm_bf16* A, const fnorm_bf16* B, const fnorm_bf16* R,
                                       fnorm_bf16* C, int64_t M, int64_t N, int64_t K, fnorm_norm_t norm,
                                       const fnorm_bf16* gamma, const fnorm_bf16* beta, float eps,
                                       float* mean_out, float* rstd_out, void* stream);

/*
 * fnorm_fold_prenorm_affine — fold the fixed elementwise affine of a pre-norm
 * into the weight of the GEMM that the normalised rows feed:
 *   B_folded[k,n] = bf16(gamma[k] * B[k,n])   (round to nearest even)
 *   colsum[n]     = sum_k B_folded[k,n]       (fp32, over the rounded values)
 *   bias[n]       = sum_k beta[k] * B[k,n]    (fp32)
 *   [ATB] 6.4 (with gamma fixed, as at inference, it can be folded into the
 *   weights of the following matmul; a training step, whose gamma changes,
 *   folds again); [FNF-ru] "Lazy Pre-Norm" limits (the per-column affine does
 *   not commute with the GEMM, so it cannot stay in the prologue).
 *   B:        [K,N] bf16.
 *   gamma:    [K] bf16, or NULL (B_folded is then a copy of B).
 *   beta:     [K] bf16, or NULL; bias must be non-NULL exactly when beta is.
 *   B_folded: [K,N] bf16 output; may be B itself (in place), no other overlap.
 *   colsum:   [N] fp32 output (16-byte aligned), or NULL.  Needed by
 *             fnorm_prenorm_gemm for LayerNorm.
 *   bias:     [N] fp32 output (16-byte aligned), or NULL.
 *   Reductions run in a fixed order: the outputs are deterministic.
 *   (M is absent: there is no A; K and N follow the shared size rules.)
 */
fnorm_status_t fnorm_fold_prenorm_affine(const fnorm_bf16* B, int64_t K, int64_t N, const fnorm_bf16* gamma,
                                         const fnorm_bf16* beta, fnorm_bf16* B_folded, float* colsum,
                                         float* bias, void* stream);

/*
 * fnorm_prenorm_gemm — C = (norm(A) * gamma + beta) @ B, a pre-norm with
 * elementwise affine feeding a GEMM, in one lazy kernel on the weight folded
 * by fnorm_fold_prenorm_affine:
 *   RMSNorm:   C = rstd * (A @ B_folded) + bias
 *   LayerNorm: C = rstd * (A @ B_folded - mean * colsum) + bias
 *   mean and rstd are the row statistics of A (rstd = 1/sqrt(var + eps) with
 *   the biased variance for LayerNorm, 1/sqrt(mean(a^2) + eps) for RMSNorm),
 *   summed in fp32 from the A tiles in shared memory by a dedicated norm warp
 *   group while the tensor cores run (LayerNorm: sums shifted by the row's
 *   first element), and applied to the fp32 accumulator before the bf16
 *   rounding of C.
 *   [FNF-ru] "Lazy Pre-Norm" (the row scale applied after the k-loop) and
 *   "FlashNormAttention" (a pre-LayerNorm computed by its own warp group);
 *   [ATB] 1.1, 1.2.  Removing the mean after the GEMM is exact in real
 *   arithmetic: sum_k (a_k - mean) * B'[k,n] = (A @ B')[m,n] - mean * colsum[n];
 *   colsum sums the same rounded B' the tensor cores multiply.
 *   B_folded: [K,N] bf16 (fnorm_fold_prenorm_affine; with gamma = NULL it is B).
 *   colsum:   [N] fp32, 16-byte aligned; required for LayerNorm, unused (may
 *             be NULL) for RMSNorm.
 *   bias:     [N] fp32, 16-byte aligned, or NULL (beta = 0).
 *   eps:      epsilon of the pre-norm, inside the square root.
 *   mean_out: [M] fp32 (LayerNorm only, else must be NULL), or NULL.
 *   rstd_out: [M] fp32, or NULL.
 *   With RMSNorm and bias == NULL this is fnorm_lazy_prenorm_gemm on B_folded.
 */
fnorm_status_t fnorm_prenorm_gemm(const fnorm_bf16* A, const fnorm_bf16* B_folded, fnorm_bf16* C,
                                  int64_t M, int64_t N, int64_t K, fnorm_norm_t norm, const float* colsum,
                                  const float* bias, float eps, float* mean_out, float* rstd_out,
                                  void* stream);

/*
 * fnorm_rmsnorm — standalone row RMSNorm, Y = X / sqrt(mean(X^2) + eps) * gamma.
 *   [ATB] 1.2.  The unfused comparison kernel ([FNF-ru] FAQ: a standalone norm
 *   stays memory-bound however well it is written).  gamma: [N] or NULL.
 *   rstd_out: [M] fp32 or NULL.
 */
fnorm_status_t fnorm_rmsnorm(const fnorm_bf16* X, fnorm_bf16* Y, int64_t M, int64_t N,
                             const fnorm_bf16* gamma, float eps, float* rstd_out, void* stream);

/*
 * fnorm_layernorm — standalone row LayerNorm,
 *   Y = (X - mean) / sqrt(var + eps) * gamma + beta, biased variance ([ATB] 1.1).
 *   gamma, beta: [N] or NULL.  mean_out, rstd_out: [M] fp32 or NULL.
 */
fnorm_status_t fnorm_layernorm(const fnorm_bf16* X, fnorm_bf16* Y, int64_t M, int64_t N,
                               const fnorm_bf16* gamma, const fnorm_bf16* beta, float eps,
                               float* mean_out, float* rstd_out, void* stream);

/*
 * fnorm_add_rownorm — standalone residual-add row norm,
 *   Y = norm(X + R) * gamma + beta, the sum X + R taken in fp32 per element.
 *   The unfused comparison of fnorm_gemm_add_postnorm (its norm half after a
 *   plain fnorm_gemm); [FNF-ru] "FlashNormAttention" (residual connection and
 *   post-RMSNorm); [ATB] 1.1, 1.2.
 *   X, R, Y: [M,N] bf16; R must not overlap Y.  norm: FNORM_LAYERNORM or
 *   FNORM_RMSNORM.  gamma, beta: [N] or NULL.  mean_out (LayerNorm only),
 *   rstd_out: [M] fp32 or NULL.  N <= 32768.
 */
fnorm_status_t fnorm_add_rownorm(const fnorm_bf16* X, const fnorm_bf16* R, fnorm_bf16* Y, int64_t M, int64_t N,
                                 fnorm_norm_t norm, const fnorm_bf16* gamma, const fnorm_bf16* beta, float eps,
                                 float* mean_out, float* rstd_out, void* stream);

/*
 * fnorm_rmsnorm_backward — standalone RMSNorm backward without affine: for
 * Y = X * rstd (rstd = 1/sqrt(mean(X^2) + eps) per row, given),
 *   dX = rstd * dY - rstd^3 * X * sum_n(dY * X) / N.
 *   [ATB] 1.2 (the RMSNorm it differentiates); the unfused comparison of
 *   fnorm_lazy_prenorm_gemm_backward's dA.  dY, X, dX: [M,N] bf16; rstd: [M]
 *   fp32.  N <= 16384.
 */
fnorm_status_t fnorm_rmsnorm_backward(const fnorm_bf16* dY, const fnorm_bf16* X, const float* rstd, fnorm_bf16* dX,
                                      int64_t M, int64_t N, void* stream);

/*
 * fnorm_check_status — synchronise `stream`, then read and clear the device
 * status word of the current device.  Returns FNORM_ERR_TIMEOUT if a kernel
 * gave up on a bounded wait since the last check; FNORM_ERR_CUDA if the
 * stream reported an error, or if a clustered kernel ran in a cluster of
 * another size than it was launched with (it then returns at once and
 * writes nothing: profilers that replay a cooperative launch drop its
 * clusters); else FNORM_OK.
 */
fnorm_status_t fnorm_check_status(void* stream);

/*
 * fnorm_last_error — message describing the last failing call on this host
 * thread ("" if none).  The pointer stays valid until the next call on the
 * same thread.
 */
const char* fnorm_last_error(void);

/*
 * fnorm_set_wait_limit_ns — upper bound, in nanoseconds of GPU global time,
 * on every wait inside the kernels launched after this call (process-wide;
 * default 2e9 = 2 s).  0 restores the default.
 */
fnorm_status_t fnorm_set_wait_limit_ns(uint64_t ns);

/*
 * fnorm_postnorm_plan — how fnorm_gemm_postnorm (no workspace) splits a row
 * of width N: *cluster receives the CTAs per cluster along N and
 * *cols_per_cta the columns each CTA owns (a multiple of 64; more than 256
 * means the spill layout).  With a workspace, rows of more than 1024 columns
 * are instead 256-column tiles over the whole grid
 * (fnorm_postnorm_workspace_size > 0).  Host only; launches nothing.
 */
fnorm_status_t fnorm_postnorm_plan(int64_t N, int* cluster, int* cols_per_cta);

/*
 * fnorm_set_postnorm_cluster — force the cluster size used by
 * fnorm_gemm_postnorm (1, 2, 4 or 8; 0 = automatic, the default).  A testing
 * and tuning knob: statistics agree across cluster sizes up to fp32
 * summation order.  Process-wide.  A forced size that cannot hold the row
 * (8 CTAs hold at most 128 columns each) makes later calls return
 * FNORM_ERR_UNSUPPORTED.
 */
fnorm_status_t fnorm_set_postnorm_cluster(int cluster_size);

/*
 * fnorm_set_pair_mma — choose when fnorm_gemm, fnorm_lazy_prenorm_gemm and
 * fnorm_prenorm_gemm run their 256-column tiles as two-CTA MMAs (a cluster of
 * two CTAs computes a [256 x 256] tile with tcgen05 cta_group::2; each CTA
 * stages its 128 rows of A and half of the tile's B columns, and the second
 * CTA's copies complete on the first CTA's barriers).  mode: 1 = whenever the
 * tile is 256 columns wide and B is not resident; 0 = never; -1 = automatic,
 * the default, which keeps the one-CTA tiles (on GB300 they measured as fast
 * or faster on every shape tried).  It changes the schedule, not the
 * arithmetic: every output is the same sum over K in the same order, and the
 * two forms agree bit for bit.  Process-wide.  Any other mode returns
 * FNORM_ERR_INVALID_ARG.
 */
fnorm_status_t fnorm_set_pair_mma(int mode);

/*
 * fnorm_set_b_multicast — choose when fnorm_gemm, fnorm_gemm_ex,
 * fnorm_lazy_prenorm_gemm, fnorm_prenorm_gemm, the plain GEMMs of the
 * backward entry points (dA, dB) and the grid exchange of
 * fnorm_gemm_postnorm_ws share B between the two CTAs of a 2-CTA cluster
 * along M: the CTAs compute the
 * tiles of two neighbouring 128-row blocks at the same 256 columns, each
 * with its own one-CTA MMAs, and each loads half of every k-block's B tile
 * into both CTAs' shared memory with one TMA multicast (a third less read
 * from L2 per SM).  mode: 1 = whenever the tile is 256 columns wide and B is
 * not resident; 0 = never; -1 = automatic, the default (the same, for more
 * than one row block).  It changes the schedule, not the arithmetic: every
 * output is the same sum in the same order as with one-CTA tiles.
 * Process-wide.  Any other mode returns FNORM_ERR_INVALID_ARG.
 */
fnorm_status_t fnorm_set_b_multicast(int mode);

/*
 * fnorm_debug_wait_timeout — failure-detection self test.  Launches one small
 * kernel that waits, with a bound of limit_ns, on a barrier that nothing
 * arrives on; the wait runs out, the kernel records a timeout in the device
 * status word and returns.  fnorm_check_status(stream) then returns
 * FNORM_ERR_TIMEOUT and the CUDA context stays usable.  limit_ns is clamped
 * to [1e3, 1e10].
 */
fnorm_status_t fnorm_debug_wait_timeout(uint64_t limit_ns, void* stream);

/*
 * fnorm_debug_cluster_shape — self test of the check every clustered kernel
 * makes at entry.  Launches a small kernel that expects clusters of two CTAs
 * in clusters of `cluster` CTAs (1 or 2; anything else is
 * FNORM_ERR_INVALID_ARG).  With 2 the check passes; with 1 it records the
 * mismatch in the device status word, which fnorm_check_status(stream) then
 * reports as FNORM_ERR_CUDA.  The kernel performs no cluster operation
 * either way.
 */
fnorm_status_t fnorm_debug_cluster_shape(int cluster, void* stream);

/* Library version, major * 10000 + minor * 100 + patch. */
int fnorm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FNORM_H */
