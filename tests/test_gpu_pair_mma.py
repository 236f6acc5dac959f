"""GPU parity of the two-CTA MMA (tcgen05 cta_group::2) kernels against the fp64 oracle.

The pair path is forced on (fnorm_set_pair_mma(1)) for the plain GEMM, the
Lazy Pre-RMSNorm GEMM and the lazy pre-norms with the affine folded into B:
256-row tiles whose second CTA holds ragged or no rows, ragged N and K,
several tiles per CTA pair (both accumulator buffers cycling, the paired tile
order of the lazy pre-norm), and agreement with the one-CTA kernels.
"""
import numpy as np
import pytest
import torch

import normalization_gemm_tcgen05_gb300 as fn
import oracle
from gpu_util import assert_mean_close, assert_out_close, assert_rstd_close
from workloads import WORKLOADS, make_inputs, to_f64

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


def _dev(t):
    return None if t is None else t.to(DEV)


@pytest.fixture
def pair_on():
    fn.set_pair_mma(1)
    try:
        yield
    finally:
        fn.set_pair_mma(-1)


# (M, N, K): one pair tile with all rows; second CTA with no rows (M < 256) or
# a ragged share; N tails inside a half of B; K tails; several column groups;
# several tiles per pair
GEMM_SHAPES = [(256, 256, 512), (200, 256, 72), (300, 264, 1000), (1, 264, 8), (513, 520, 264),
               (1000, 1024, 128), (8192, 2048, 128)]


@pytest.mark.parametrize("M,N,K", GEMM_SHAPES, ids=lambda v: str(v))
def test_pair_gemm(pair_on, M, N, K):
    w = WORKLOADS["cfg3"].scaled(M=M, N=N, K=K, b_std=1.0 / np.sqrt(K), a_row_scale=False)
    d = make_inputs(w, M * 5 + N + K)
    C = fn.gemm(_dev(d["A"]), _dev(d["B"]))
    assert_out_close(C, oracle.gemm(to_f64(d["A"]), to_f64(d["B"])), f"pair gemm {M}x{N}x{K}")
    fn.check_status(DEV)


PRE_SHAPES = [(256, 256, 512), (333, 256, 1024), (129, 520, 256), (640, 4096, 256), (8192, 2048, 128)]


@pytest.mark.parametrize("M,N,K", PRE_SHAPES, ids=lambda v: str(v))
def test_pair_lazy_prenorm(pair_on, M, N, K):
    w = WORKLOADS["cfg3"].scaled(M=M, N=N, K=K, b_std=1.0 / np.sqrt(K))
    d = make_inputs(w, 7 * M + K)
    C, rstd = fn.lazy_prenorm_gemm(_dev(d["A"]), _dev(d["B"]), w.eps, return_rstd=True)
    Cr, rr = oracle.lazy_prenorm_gemm(to_f64(d["A"]), to_f64(d["B"]), w.eps)
    assert_out_close(C, Cr, f"pair prenorm {M}x{N}x{K}")
    assert_rstd_close(rstd, rr, f"pair prenorm rstd {M}x{N}x{K}")
    fn.check_status(DEV)


PRE_AFF_SHAPES = [(300, 256, 512), (513, 520, 200), (2048, 1024, 256)]


@pytest.mark.parametrize("M,N,K", PRE_AFF_SHAPES, ids=lambda v: str(v))
@pytest.mark.parametrize("norm", ["layernorm", "rmsnorm"])
def test_pair_prenorm_affine(pair_on, norm, M, N, K):
    base = "preln_affine" if norm == "layernorm" else "prerms_gamma"
    w = WORKLOADS[base].scaled(M=M, N=N, K=K, b_std=1.0 / np.sqrt(K), gamma=True, beta=True,
                               a_row_offset=1.0 if norm == "layernorm" else 0.0)
    d = make_inputs(w, M + 3 * N + K)
    Bf, colsum, bias = fn.fold_prenorm_affine(_dev(d["B"]), _dev(d["gamma"]), _dev(d["beta"]))
    C, st = fn.prenorm_gemm(_dev(d["A"]), Bf, w.norm, colsum, bias, w.eps, return_stats=True)
    Cr, mr, rr = oracle.prenorm_affine_gemm(to_f64(d["A"]), to_f64(d["B"]), w.norm, to_f64(d["gamma"]),
                                            to_f64(d["beta"]), w.eps)
    what = f"pair pre-{norm}+affine {M}x{N}x{K}"
    assert_out_close(C, Cr, what)
    assert_rstd_close(st["rstd"], rr, what + " rstd")
    if norm == "layernorm":
        assert_mean_close(st["mean"], mr, rr, what + " mean")
    fn.check_status(DEV)


def test_pair_identity_B(pair_on):
    # B = I: every product is exact in fp32, so C reproduces A bit for bit,
    # whichever CTA of the pair holds a row or a column half
    w = WORKLOADS["cfg3"].scaled(M=600, N=512, K=512, a_row_scale=False)
    A = make_inputs(w, 11)["A"]
    C = fn.gemm(_dev(A), torch.eye(512, dtype=torch.bfloat16, device=DEV))
    assert torch.equal(C.cpu(), A), "A @ I != A on the two-CTA path"
    fn.check_status(DEV)


@pytest.mark.parametrize("kind", ["gemm", "prenorm"])
def test_pair_matches_one_cta(kind):
    # the same sums over K in the same k-block order: the two schedules agree
    # element for element
    M, N, K = 1000, 768, 640
    w = WORKLOADS["cfg3"].scaled(M=M, N=N, K=K, b_std=1.0 / np.sqrt(K))
    d = make_inputs(w, 5)
    A, B = _dev(d["A"]), _dev(d["B"])
    outs = []
    try:
        for mode in (0, 1):
            fn.set_pair_mma(mode)
            outs.append(fn.gemm(A, B) if kind == "gemm" else fn.lazy_prenorm_gemm(A, B, w.eps, return_rstd=True))
    finally:
        fn.set_pair_mma(-1)
    fn.check_status(DEV)
    if kind == "gemm":
        assert torch.equal(outs[0], outs[1]), "one-CTA and two-CTA GEMMs differ"
    else:
        assert torch.equal(outs[0][0], outs[1][0]), "one-CTA and two-CTA lazy pre-norms differ"
        assert torch.equal(outs[0][1], outs[1][1]), "one-CTA and two-CTA rstd differ"


def test_pair_mode_argument_checked():
    with pytest.raises(fn.FnormError):
        fn.set_pair_mma(2)
    fn.set_pair_mma(-1)
