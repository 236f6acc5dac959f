"""GPU parity of the residual-add post-norm, the affine fold and the pre-norm
with affine (LayerNorm or RMSNorm) feeding a GEMM, against the fp64 oracle.

Small cases spanning several tiles, ragged tails in M, N and K, every
post-norm layout (one CTA, resident cluster, spill), the resident-B variant,
and the degenerate rows of each form.
"""
import numpy as np
import pytest
import torch

import normalization_gemm_tcgen05_gb300 as fn
import oracle
from gpu_util import assert_mean_close, assert_out_close, assert_rstd_close, np64
from workloads import WORKLOADS, make_inputs, to_f64

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


def _dev(t):
    return None if t is None else t.to(DEV)


# ----------------------------------------------------------------------------
# residual-add post-norm: C = norm(A @ B + R) * gamma + beta
# ----------------------------------------------------------------------------
RES_CASES = [  # (norm, M, N, K): one CTA, resident cluster, spill layout
    ("layernorm", 256, 64, 256), ("rmsnorm", 200, 128, 72), ("layernorm", 333, 200, 1000),
    ("layernorm", 256, 256, 512), ("rmsnorm", 129, 8, 64),
    # first-tile residual by TMA: a half's box partly past N (128- and 64-column tiles)
    ("layernorm", 200, 72, 128), ("rmsnorm", 131, 40, 64),
    ("layernorm", 256, 320, 256), ("rmsnorm", 300, 512, 512), ("layernorm", 256, 1024, 256),
    ("layernorm", 256, 1032, 256), ("rmsnorm", 256, 2048, 128), ("layernorm", 130, 4096, 256),
]


def _res_case(norm, M, N, K, seed, affine=True):
    base = "res_ln_n128" if norm == "layernorm" else "res_rms_n1024"
    w = WORKLOADS[base].scaled(M=M, N=N, K=K, b_std=1.0 / np.sqrt(K))
    d = make_inputs(w, seed)
    g = d["gamma"] if affine else None
    b = d["beta"] if affine else None
    return w, d, g, b


def _check_res(w, d, g, b, what):
    C, st = fn.gemm_add_postnorm(_dev(d["A"]), _dev(d["B"]), _dev(d["R"]), w.norm, _dev(g), _dev(b), w.eps,
                                 return_stats=True)
    ref = oracle.gemm_add_postnorm(to_f64(d["A"]), to_f64(d["B"]), to_f64(d["R"]), w.norm, to_f64(g), to_f64(b),
                                   w.eps)
    assert_out_close(C, ref["C"], what)
    assert_rstd_close(st["rstd"], ref["rstd"], what + " rstd")
    if w.norm == "layernorm":
        assert_mean_close(st["mean"], ref["mean"], ref["rstd"], what + " mean")
    fn.check_status(DEV)
    return C


@pytest.mark.parametrize("norm,M,N,K", RES_CASES, ids=lambda v: str(v))
def test_add_postnorm(norm, M, N, K):
    w, d, g, b = _res_case(norm, M, N, K, seed=M + N + K)
    _check_res(w, d, g, b, f"add+{norm} {M}x{N}x{K}")


def test_add_postnorm_no_affine():
    w, d, _, _ = _res_case("layernorm", 256, 512, 128, seed=3)
    _check_res(w, d, None, None, "add+LN without affine")


def test_add_postnorm_resident_b():
    # more row blocks than SMs with N <= 128 and short K: B resident in shared memory
    w, d, g, b = _res_case("layernorm", 160 * 128 + 77, 64, 256, seed=4)
    _check_res(w, d, g, b, "add+LN resident B")


@pytest.mark.parametrize("N", [128, 1024, 2048])
def test_add_postnorm_zero_residual_is_postnorm(N):
    # R = 0: v = u * 1 + 0 = u exactly, so the output must equal the plain
    # post-norm's bit for bit (same arithmetic, same summation order)
    # (the same layout for both: wide rows of the plain post-norm would
    # otherwise take the grid-wide exchange, which sums in another order)
    w, d, g, b = _res_case("layernorm", 256, N, 256, seed=N)
    A, B = _dev(d["A"]), _dev(d["B"])
    Z = torch.zeros(256, N, dtype=torch.bfloat16, device=DEV)
    try:
        fn.set_postnorm_cluster(0 if N <= 1024 else 4)
        C1 = fn.gemm_add_postnorm(A, B, Z, "layernorm", _dev(g), _dev(b), w.eps)
        C0 = fn.gemm_postnorm(A, B, "layernorm", _dev(g), _dev(b), w.eps)
    finally:
        fn.set_postnorm_cluster(0)
    assert torch.equal(C1, C0)


@pytest.mark.parametrize("N", [256, 1024, 4096])
def test_add_postnorm_zero_gemm_is_norm_of_residual(N):
    # A = 0: C = norm(R) * gamma + beta, the standalone norm of R
    w, d, g, b = _res_case("layernorm", 200, N, 128, seed=N + 1)
    A = torch.zeros(200, 128, dtype=torch.bfloat16, device=DEV)
    C = fn.gemm_add_postnorm(A, _dev(d["B"]), _dev(d["R"]), "layernorm", _dev(g), _dev(b), w.eps)
    Y = fn.layernorm(_dev(d["R"]), _dev(g), _dev(b), w.eps)
    ref, _, _ = oracle.layernorm(to_f64(d["R"]), to_f64(g), to_f64(b), w.eps)
    assert_out_close(C, ref, "norm of R through the fused kernel")
    assert_out_close(Y, ref, "standalone norm of R")


def test_add_postnorm_forced_clusters_agree():
    w, d, g, b = _res_case("rmsnorm", 256, 1024, 256, seed=9)
    outs = {}
    try:
        for c in (1, 2, 4, 8):
            fn.set_postnorm_cluster(c)
            outs[c] = _check_res(w, d, g, b, f"add+RMS cluster {c}")
    finally:
        fn.set_postnorm_cluster(0)
    for c in (1, 2, 8):
        assert_out_close(outs[c], np64(outs[4]), f"cluster {c} vs 4")


def test_add_postnorm_empty():
    w, d, g, b = _res_case("layernorm", 0, 128, 64, seed=1)
    C = fn.gemm_add_postnorm(torch.empty(0, 64, dtype=torch.bfloat16, device=DEV),
                             _dev(d["B"]), torch.empty(0, 128, dtype=torch.bfloat16, device=DEV), "layernorm")
    assert C.shape == (0, 128)


# ----------------------------------------------------------------------------
# affine fold: B' = bf16(gamma_k B[k, n]), colsum = sum_k B', bias = beta @ B
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("K,N", [(64, 64), (72, 200), (4096, 8), (1000, 4104)], ids=lambda v: str(v))
def test_fold(K, N):
    w = WORKLOADS["preln_affine"].scaled(M=8, K=K, N=N)
    d = make_inputs(w, K + N)
    Bf, colsum, bias = fn.fold_prenorm_affine(_dev(d["B"]), _dev(d["gamma"]), _dev(d["beta"]))
    # B' is defined bit for bit: an exact fp32 product rounded once to bf16
    want = (d["gamma"].float()[:, None] * d["B"].float()).to(torch.bfloat16)
    assert torch.equal(Bf.cpu(), want)
    Bf64 = to_f64(want)
    cs_ref = Bf64.sum(axis=0)
    b_ref = to_f64(d["beta"]) @ to_f64(d["B"])
    tol_cs = 1e-5 * np.abs(Bf64).sum(axis=0) + 1e-6
    tol_b = 1e-5 * (np.abs(to_f64(d["beta"]))[:, None] * np.abs(to_f64(d["B"]))).sum(axis=0) + 1e-6
    assert np.all(np.abs(np64(colsum) - cs_ref) <= tol_cs)
    assert np.all(np.abs(np64(bias) - b_ref) <= tol_b)


def test_fold_without_gamma_copies_and_in_place():
    w = WORKLOADS["preln_affine"].scaled(M=8, K=256, N=128)
    d = make_inputs(w, 5)
    B = _dev(d["B"])
    Bf, colsum, bias = fn.fold_prenorm_affine(B, None, None)
    assert torch.equal(Bf, B) and bias is None
    Bc = B.clone()
    Bf2, colsum2, _ = fn.fold_prenorm_affine(Bc, _dev(d["gamma"]), None, out=Bc)  # in place
    want = (d["gamma"].float()[:, None] * d["B"].float()).to(torch.bfloat16)
    assert Bf2.data_ptr() == Bc.data_ptr() and torch.equal(Bc.cpu(), want)
    Bf3, colsum3, _ = fn.fold_prenorm_affine(B, _dev(d["gamma"]), None)
    assert torch.equal(Bf3, Bc) and torch.equal(colsum3, colsum2)  # deterministic


# ----------------------------------------------------------------------------
# pre-norm with affine feeding a GEMM: C = (norm(A) * gamma + beta) @ B
# ----------------------------------------------------------------------------
PRE_AFF_SHAPES = [(256, 128, 512), (200, 64, 72), (333, 256, 1000), (128, 520, 256), (1, 8, 8),
                  (300, 4096, 128)]


def _pre_aff(norm, M, N, K, seed, gamma=True, beta=True, offset=1.0):
    base = "preln_affine" if norm == "layernorm" else "prerms_gamma"
    w = WORKLOADS[base].scaled(M=M, N=N, K=K, b_std=1.0 / np.sqrt(K), gamma=gamma, beta=beta,
                               a_row_offset=offset if norm == "layernorm" else 0.0)
    return w, make_inputs(w, seed)


def _check_pre_aff(w, d, what, A=None):
    A = d["A"] if A is None else A
    Bf, colsum, bias = fn.fold_prenorm_affine(_dev(d["B"]), _dev(d["gamma"]), _dev(d["beta"]))
    C, st = fn.prenorm_gemm(_dev(A), Bf, w.norm, colsum, bias, w.eps, return_stats=True)
    Cr, mr, rr = oracle.prenorm_affine_gemm(to_f64(A), to_f64(d["B"]), w.norm, to_f64(d["gamma"]),
                                            to_f64(d["beta"]), w.eps)
    assert_out_close(C, Cr, what)
    assert_rstd_close(st["rstd"], rr, what + " rstd")
    if w.norm == "layernorm":
        assert_mean_close(st["mean"], mr, rr, what + " mean")
    fn.check_status(DEV)
    return C, Cr, st


@pytest.mark.parametrize("M,N,K", PRE_AFF_SHAPES, ids=lambda v: str(v))
@pytest.mark.parametrize("norm", ["layernorm", "rmsnorm"])
def test_prenorm_affine(norm, M, N, K):
    w, d = _pre_aff(norm, M, N, K, seed=M + 3 * N + K, beta=True)
    _check_pre_aff(w, d, f"pre-{norm}+affine {M}x{N}x{K}")


@pytest.mark.parametrize("gamma,beta", [(True, False), (False, True), (False, False)])
@pytest.mark.parametrize("norm", ["layernorm", "rmsnorm"])
def test_prenorm_affine_variants(norm, gamma, beta):
    # RMSNorm with gamma only (or nothing) runs the plain lazy kernel on B'
    w, d = _pre_aff(norm, 256, 192, 320, seed=11, gamma=gamma, beta=beta)
    _check_pre_aff(w, d, f"pre-{norm} gamma={gamma} beta={beta}")


def test_preln_large_row_offsets():
    # row means 20x the row spread: the mean is removed after the GEMM by the
    # column-sum correction, which must survive the cancellation
    w, d = _pre_aff("layernorm", 256, 256, 1024, seed=12, offset=20.0)
    _check_pre_aff(w, d, "pre-LN offset 20 sigma")


def test_prenorm_affine_special_rows():
    # zero row and constant row: LayerNorm gives x - mean = 0, so C = beta @ B;
    # RMSNorm of a zero row gives C = beta @ B too
    for norm in ("layernorm", "rmsnorm"):
        w, d = _pre_aff(norm, 300, 128, 512, seed=13)
        A = d["A"].clone()
        A[5] = 0
        A[6] = 2.5
        A[299] = -1.0
        C, Cr, st = _check_pre_aff(w, d, f"pre-{norm} special rows", A=A)
        bias = to_f64(d["beta"]) @ to_f64(d["B"])
        assert np.max(np.abs(np64(C)[5] - bias)) <= 2e-2 * np.max(np.abs(bias)) + 1e-3
        if norm == "layernorm":
            for r in (6, 299):
                assert np.max(np.abs(np64(C)[r] - bias)) <= 2e-2 * np.max(np.abs(bias)) + 1e-3
            assert abs(float(st["rstd"][6]) - 1 / np.sqrt(w.eps)) <= 1e-4 / np.sqrt(w.eps)


def test_preln_identity_B_is_layernorm():
    # B = I: C = LN(A) * gamma + beta, the standalone LayerNorm (both kernels)
    w, d = _pre_aff("layernorm", 256, 256, 256, seed=14)
    eye = torch.eye(256, dtype=torch.bfloat16)
    Bf, colsum, bias = fn.fold_prenorm_affine(_dev(eye), _dev(d["gamma"]), _dev(d["beta"]))
    C = fn.prenorm_gemm(_dev(d["A"]), Bf, "layernorm", colsum, bias, w.eps)
    Y = fn.layernorm(_dev(d["A"]), _dev(d["gamma"]), _dev(d["beta"]), w.eps)
    ref, _, _ = oracle.layernorm(to_f64(d["A"]), to_f64(d["gamma"]), to_f64(d["beta"]), w.eps)
    assert_out_close(C, ref, "pre-LN with B = I")
    assert_out_close(Y, ref, "standalone layernorm")


def test_prenorm_affine_resident_b():
    w, d = _pre_aff("layernorm", 160 * 128 + 5, 64, 256, seed=15)
    _check_pre_aff(w, d, "pre-LN resident B")


def test_prenorm_gemm_empty():
    C = fn.prenorm_gemm(torch.empty(0, 64, dtype=torch.bfloat16, device=DEV),
                        torch.zeros(64, 128, dtype=torch.bfloat16, device=DEV), "layernorm",
                        torch.zeros(128, dtype=torch.float32, device=DEV))
    assert C.shape == (0, 128)


@pytest.mark.parametrize("norm,N", [("layernorm", 128), ("rmsnorm", 1024), ("layernorm", 4104)])
def test_add_rownorm_standalone(norm, N):
    # the unfused residual-add norm kernel: norm(X + R) * gamma + beta
    w, d, g, b = _res_case(norm, 300, N, 64, seed=N + 5)
    X = torch.randn(300, N, generator=torch.Generator().manual_seed(N)).to(torch.bfloat16)
    Y, st = fn.add_rownorm(_dev(X), _dev(d["R"]), norm, _dev(g), _dev(b), w.eps, return_stats=True)
    H = to_f64(X) + to_f64(d["R"])
    if norm == "layernorm":
        ref, mr, rr = oracle.layernorm(H, to_f64(g), to_f64(b), w.eps)
        assert_mean_close(st["mean"], mr, rr)
    else:
        ref, rr = oracle.rmsnorm(H, to_f64(g), to_f64(b), w.eps)
    assert_out_close(Y, ref, f"add_rownorm {norm} N={N}")
    assert_rstd_close(st["rstd"], rr)
