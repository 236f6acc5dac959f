"""GPU parity of the backward of the Lazy Pre-RMSNorm GEMM and of the GEMM
post-norm against the fp64 oracle.

The forward runs on the GPU (its bf16 output C and fp32 rstd are what a
training step saves); the backward's dA and dB are compared with the oracle's
chain rule on the same bf16 inputs.  Small cases span several tiles and ragged
tails in M, N and K; the degenerate rows are a zero row and a constant row.
"""
import numpy as np
import pytest
import torch

import normalization_gemm_tcgen05_gb300 as fn
import oracle
from gpu_util import assert_out_close, np64
from workloads import WORKLOADS, make_inputs, to_f64

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


def _case(M, N, K, seed):
    w = WORKLOADS["prenorm_bwd"].scaled(M=M, N=N, K=K, b_std=1.0 / np.sqrt(K))
    return w, make_inputs(w, seed)


def _run(w, d, A=None):
    A = d["A"] if A is None else A
    Ad, Bd, dCd = A.to(DEV), d["B"].to(DEV), d["dC"].to(DEV)
    C, rstd = fn.lazy_prenorm_gemm(Ad, Bd, w.eps, return_rstd=True)
    dA, dB = fn.lazy_prenorm_gemm_backward(Ad, Bd, C, dCd, rstd)
    fn.check_status(DEV)
    rA, rB, _ = oracle.lazy_prenorm_gemm_backward(to_f64(A), to_f64(d["B"]), to_f64(d["dC"]), w.eps)
    return dA, dB, rA, rB


SHAPES = [(256, 128, 512), (200, 64, 72), (336, 256, 1000), (128, 520, 256), (8, 8, 8), (304, 192, 4096),
          (1000, 1024, 128), (136, 4096, 64)]


@pytest.mark.parametrize("M,N,K", SHAPES, ids=lambda v: str(v))
def test_prenorm_backward(M, N, K):
    w, d = _case(M, N, K, seed=M + 5 * N + K)
    dA, dB, rA, rB = _run(w, d)
    assert_out_close(dA, rA, f"dA {M}x{N}x{K}")
    assert_out_close(dB, rB, f"dB {M}x{N}x{K}")


def test_prenorm_backward_special_rows():
    # a zero row has no gradient through the norm (dA row = rstd * dA_hat with
    # rstd = 1/sqrt(eps)); a constant row and an outlier row stress the
    # cancellation in the RMSNorm backward
    w, d = _case(304, 128, 512, seed=3)
    A = d["A"].clone()
    A[4] = 0
    A[5] = 1.5
    A[6] *= 100
    dA, dB, rA, rB = _run(w, d, A)
    assert_out_close(dA, rA, "dA special rows")
    assert_out_close(dB, rB, "dB special rows")
    assert np.all(np64(dB).shape == (512, 128))


def test_prenorm_backward_one_side():
    w, d = _case(256, 256, 256, seed=4)
    Ad, Bd, dCd = d["A"].to(DEV), d["B"].to(DEV), d["dC"].to(DEV)
    C, rstd = fn.lazy_prenorm_gemm(Ad, Bd, w.eps, return_rstd=True)
    dA, dB = fn.lazy_prenorm_gemm_backward(Ad, Bd, C, dCd, rstd, need_dB=False)
    assert dB is None
    dA2, dB2 = fn.lazy_prenorm_gemm_backward(Ad, Bd, C, dCd, rstd, need_dA=False)
    assert dA2 is None
    dA3, dB3 = fn.lazy_prenorm_gemm_backward(Ad, Bd, C, dCd, rstd)
    assert torch.equal(dA, dA3) and torch.equal(dB2, dB3)


def test_prenorm_backward_dA_any_M():
    # dA alone has no M % 8 rule (only dB reads A^T); M = 333 and M = 1
    for M in (333, 1):
        w, d = _case(M, 128, 256, seed=M)
        Ad, Bd, dCd = d["A"].to(DEV), d["B"].to(DEV), d["dC"].to(DEV)
        C, rstd = fn.lazy_prenorm_gemm(Ad, Bd, w.eps, return_rstd=True)
        dA, _ = fn.lazy_prenorm_gemm_backward(Ad, Bd, C, dCd, rstd, need_dB=False)
        rA, _, _ = oracle.lazy_prenorm_gemm_backward(to_f64(d["A"]), to_f64(d["B"]), to_f64(d["dC"]), w.eps)
        assert_out_close(dA, rA, f"dA M={M}")


def test_prenorm_backward_scale_invariance():
    # rmsnorm(c a) = rmsnorm(a) up to eps: sum_k dA[m,k] A[m,k] = eps r^3 (dA_hat . a),
    # tiny next to |dA| |a|, so each dA row is nearly orthogonal to its A row
    w, d = _case(256, 256, 512, seed=5)
    dA, _, _, _ = _run(w, d)
    a = to_f64(d["A"])
    g = np64(dA)
    cos = np.abs(np.sum(g * a, axis=1)) / (np.linalg.norm(g, axis=1) * np.linalg.norm(a, axis=1) + 1e-30)
    assert np.max(cos) < 2e-2, f"dA rows not orthogonal to A rows: max |cos| {np.max(cos):.3e}"


def test_prenorm_backward_empty():
    B = torch.randn(64, 128, device=DEV).to(torch.bfloat16)
    E = torch.empty(0, 64, dtype=torch.bfloat16, device=DEV)
    E2 = torch.empty(0, 128, dtype=torch.bfloat16, device=DEV)
    dA, dB = fn.lazy_prenorm_gemm_backward(E, B, E2, E2, torch.empty(0, device=DEV))
    assert dA.shape == (0, 64) and torch.all(dB == 0)


def test_prenorm_backward_full_size():
    # the bench's backward workload, in its launch configuration; sampled rows
    # of dA and columns of dB recomputed by the oracle one at a time
    w = WORKLOADS["prenorm_bwd"]
    d = make_inputs(w, 0)
    Ad, Bd, dCd = d["A"].to(DEV), d["B"].to(DEV), d["dC"].to(DEV)
    C, rstd = fn.lazy_prenorm_gemm(Ad, Bd, w.eps, return_rstd=True)
    dA, dB = fn.lazy_prenorm_gemm_backward(Ad, Bd, C, dCd, rstd)
    fn.check_status(DEV)
    rng = np.random.default_rng(7)
    rows = np.unique(np.concatenate([[0, 127, 128, w.M - 1], rng.choice(w.M, 24, replace=False)]))
    A64, B64, dC64 = to_f64(d["A"]), to_f64(d["B"]), to_f64(d["dC"])
    rA, _, r = oracle.lazy_prenorm_gemm_backward(A64[rows], B64, dC64[rows], w.eps)
    assert_out_close(dA[torch.from_numpy(rows).to(DEV)], rA, "dA sampled rows")
    cols = np.unique(np.concatenate([[0, 255, 256, w.K - 1], rng.choice(w.K, 12, replace=False)]))
    _, r_all = oracle.rmsnorm(A64, None, None, w.eps)
    ref = (A64[:, cols] * r_all[:, None]).T @ dC64
    assert_out_close(dB[torch.from_numpy(cols).to(DEV)], ref, "dB sampled rows")


# ----------------------------------------------------------------------------
# the unfused comparison's pieces: transposed-operand GEMM, standalone RMSNorm backward
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("ta,tb", [(0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("M,N,K", [(256, 128, 512), (200, 72, 136), (128, 520, 64), (1000, 256, 1000),
                                   # A^T with more than 8 column groups (12, 17)
                                   (1160, 2824, 136), (640, 4104, 64),
                                   # A^T with more tiles than SMs (160): second tiles walk the
                                   # reduction backwards, starting on the ragged last k-block
                                   (2048, 2560, 200)],
                         ids=lambda v: str(v))
def test_gemm_transposed(M, N, K, ta, tb):
    rng = np.random.default_rng(M + N + K + 2 * ta + tb)
    A = torch.from_numpy(rng.standard_normal((K, M) if ta else (M, K), dtype=np.float32)).to(torch.bfloat16)
    B = torch.from_numpy((rng.standard_normal((N, K) if tb else (K, N), dtype=np.float32)
                          / np.float32(np.sqrt(K)))).to(torch.bfloat16)
    C = fn.gemm_ex(A.to(DEV), B.to(DEV), trans_a=bool(ta), trans_b=bool(tb))
    a64, b64 = to_f64(A), to_f64(B)
    ref = oracle.gemm(a64.T if ta else a64, b64.T if tb else b64)
    assert_out_close(C, ref, f"gemm_ex ta={ta} tb={tb} {M}x{N}x{K}")


def test_gemm_transposed_identity_exact():
    # op(A) @ I reproduces op(A) exactly (each product is exact in fp32)
    A = torch.randn(192, 256, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    eye = torch.eye(192, dtype=torch.bfloat16)
    C = fn.gemm_ex(A.to(DEV), eye.to(DEV), trans_a=True)
    assert torch.equal(C.cpu(), A.t().contiguous())
    # A @ (I given as its own transpose) = A
    C2 = fn.gemm_ex(A.to(DEV), torch.eye(256, dtype=torch.bfloat16, device=DEV), trans_b=True)
    assert torch.equal(C2.cpu(), A)


@pytest.mark.parametrize("M,N", [(300, 64), (257, 1000), (64, 4096), (17, 8192)])
def test_rmsnorm_backward_standalone(M, N):
    rng = np.random.default_rng(M * N)
    X = torch.from_numpy(rng.standard_normal((M, N), dtype=np.float32) * 3).to(torch.bfloat16)
    dY = torch.from_numpy(rng.standard_normal((M, N), dtype=np.float32)).to(torch.bfloat16)
    eps = 1e-6
    _, r = oracle.rmsnorm(to_f64(X), None, None, eps)
    rstd = torch.from_numpy(r.astype(np.float32)).to(DEV)
    dX = fn.rmsnorm_backward(dY.to(DEV), X.to(DEV), rstd)
    # the oracle's backward with B = I: dA_hat = dC, the RMSNorm backward itself
    ref, _, _ = oracle.lazy_prenorm_gemm_backward(to_f64(X), np.eye(N), to_f64(dY), eps)
    assert_out_close(dX, ref, f"rmsnorm_backward {M}x{N}")


# ----------------------------------------------------------------------------
# post-norm backward: dA, dB, dgamma, dbeta of norm(A @ B) * gamma + beta
# ----------------------------------------------------------------------------
POSTB = [("layernorm", 256, 64, 256), ("rmsnorm", 200, 128, 72), ("layernorm", 256, 1024, 256),
         ("rmsnorm", 1000, 200, 128), ("layernorm", 128, 4096, 64), ("layernorm", 8, 8, 8),
         # 41 groups of 64 rows (the column sum's thread rows wrap), N not a
         # multiple of 32 (a ragged last block of columns)
         ("layernorm", 2568, 200, 64),
         # a [2048 x 1024] weight gradient: 64 tiles of 128 x 256 would not
         # fill the GPU, so it runs as 128 tiles of 128 x 128
         ("rmsnorm", 512, 1024, 2048)]


def _postb(norm, M, N, K, seed, affine=True):
    base = "cfg2_n128" if norm == "layernorm" else "cfg4_n1024_rms"
    w = WORKLOADS[base].scaled(M=M, N=N, K=K, b_std=1.0 / np.sqrt(K))
    d = make_inputs(w, seed)
    g = d["gamma"] if affine else None
    b = d["beta"] if affine else None
    dC = torch.from_numpy(np.random.default_rng(seed + 1).standard_normal((M, N), dtype=np.float32)).to(torch.bfloat16)
    Ad, Bd = d["A"].to(DEV), d["B"].to(DEV)
    gd = None if g is None else g.to(DEV)
    bd = None if b is None else b.to(DEV)
    C, st = fn.gemm_postnorm(Ad, Bd, norm, gd, bd, w.eps, return_stats=True)
    need = ("dA", "dB", "dgamma", "dbeta") if M % 8 == 0 else ("dA", "dgamma", "dbeta")
    got = fn.gemm_postnorm_backward(Ad, Bd, C, dC.to(DEV), st["rstd"], norm, gd, bd, need=need)
    fn.check_status(DEV)
    ref = oracle.gemm_postnorm_backward(to_f64(d["A"]), to_f64(d["B"]), to_f64(dC), norm, to_f64(g), to_f64(b), w.eps)
    return got, ref


@pytest.mark.parametrize("norm,M,N,K", POSTB, ids=lambda v: str(v))
def test_postnorm_backward(norm, M, N, K):
    got, ref = _postb(norm, M, N, K, seed=M + N + K)
    assert_out_close(got["dH"], ref["dH"], "dH")
    assert_out_close(got["dA"], ref["dA"], "dA")
    if got["dB"] is not None:
        assert_out_close(got["dB"], ref["dB"], "dB")
    assert_out_close(got["dgamma"], ref["dgamma"], "dgamma")
    assert_out_close(got["dbeta"], ref["dbeta"], "dbeta")


def test_postnorm_backward_no_affine_and_ragged_M():
    got, ref = _postb("layernorm", 333, 256, 128, seed=9, affine=False)
    assert got["dB"] is None
    assert_out_close(got["dA"], ref["dA"], "dA without affine")
    assert_out_close(got["dbeta"], ref["dbeta"], "dbeta without affine")


def test_postnorm_backward_layernorm_rows_sum_to_zero():
    # LayerNorm ignores a constant added to a row: each row of dH sums to ~0
    got, _ = _postb("layernorm", 256, 512, 128, seed=10)
    h = np64(got["dH"])
    scale = np.abs(h).sum(axis=1)
    assert np.all(np.abs(h.sum(axis=1)) <= 2e-2 * scale + 1e-3)


# ----------------------------------------------------------------------------
# the post-norm backward regrouped onto the consuming layer's data-gradient
# GEMM: dC = G @ op(W)^T lives only in the fused kernel's accumulator
# ----------------------------------------------------------------------------
def _rg(norm, M, N, K, J, trans_w, seed, affine=True, need=("dA", "dB", "dgamma", "dbeta")):
    base = "cfg2_n128" if norm == "layernorm" else "cfg4_n1024_rms"
    w = WORKLOADS[base].scaled(M=M, N=N, K=K, b_std=1.0 / np.sqrt(K))
    d = make_inputs(w, seed)
    rng = np.random.default_rng(seed + 2)
    G = torch.from_numpy(rng.standard_normal((M, J), dtype=np.float32)).to(torch.bfloat16)
    W = torch.from_numpy(rng.standard_normal((J, N) if trans_w else (N, J), dtype=np.float32)
                         / np.float32(np.sqrt(J))).to(torch.bfloat16)
    g = d["gamma"] if affine else None
    b = d["beta"] if affine and norm == "layernorm" else None
    Ad, Bd = d["A"].to(DEV), d["B"].to(DEV)
    gd = None if g is None else g.to(DEV)
    bd = None if b is None else b.to(DEV)
    C, st = fn.gemm_postnorm(Ad, Bd, norm, gd, bd, w.eps, return_stats=True)
    if M % 8 != 0:
        need = tuple(x for x in need if x != "dB")
    got = fn.gemm_postnorm_backward_regrouped(G.to(DEV), W.to(DEV), Ad, Bd, C, st["rstd"], norm, gd, bd,
                                              trans_w=trans_w, need=need)
    fn.check_status(DEV)
    ref = oracle.gemm_postnorm_backward_regrouped(to_f64(G), to_f64(W), to_f64(d["A"]), to_f64(d["B"]), norm,
                                                  to_f64(g), to_f64(b), w.eps, trans_w=trans_w)
    return got, ref, (G, W, C, st, Ad, Bd, gd, bd)


RG = [("layernorm", 256, 64, 256, 128, False),   # one CTA, 128-column tile, half past N
      ("rmsnorm", 200, 128, 72, 96, True),       # ragged M
      ("layernorm", 333, 200, 128, 256, False),  # a partial 32-row group; a ragged 256-column tile
      ("layernorm", 256, 256, 128, 520, True),
      ("rmsnorm", 384, 512, 256, 264, False),    # a cluster of 2
      ("layernorm", 1000, 1024, 128, 256, True),  # a cluster of 4, ragged M
      ("rmsnorm", 136, 1000, 64, 64, False),     # a cluster of 4, ragged N
      ("layernorm", 8, 8, 8, 8, False),
      # wider rows: the row sums exchanged grid-wide through the workspace
      ("layernorm", 264, 2048, 64, 128, False),
      ("rmsnorm", 300, 4096, 128, 256, True),
      ("layernorm", 128 * 20 + 5, 8192, 64, 64, False),  # 21 row blocks x 32 tiles: several waves
      ("rmsnorm", 520, 1032, 64, 72, True)]      # one tile past a cluster's reach, a ragged last tile


@pytest.mark.parametrize("norm,M,N,K,J,trans_w", RG, ids=lambda v: str(v))
def test_postnorm_backward_regrouped(norm, M, N, K, J, trans_w):
    got, ref, _ = _rg(norm, M, N, K, J, trans_w, seed=M + N + K + J)
    assert_out_close(got["dH"], ref["dH"], "dH")
    assert_out_close(got["dA"], ref["dA"], "dA")
    if got["dB"] is not None:
        assert_out_close(got["dB"], ref["dB"], "dB")
    assert_out_close(got["dgamma"], ref["dgamma"], "dgamma")
    assert_out_close(got["dbeta"], ref["dbeta"], "dbeta")


def test_postnorm_backward_regrouped_no_affine_and_partial_need():
    got, ref, _ = _rg("layernorm", 520, 384, 64, 128, True, seed=31, affine=False, need=("dgamma", "dbeta"))
    assert got["dA"] is None and got["dB"] is None
    assert_out_close(got["dH"], ref["dH"], "dH without affine")
    assert_out_close(got["dgamma"], ref["dgamma"], "dgamma without affine")
    assert_out_close(got["dbeta"], ref["dbeta"], "dbeta without affine")


def test_postnorm_backward_regrouped_matches_unfused_pipeline():
    # the consumer's GEMM to a bf16 dC, then the unfused post-norm backward:
    # the same gradients up to dC's rounding to bf16
    got, ref, (G, W, C, st, Ad, Bd, gd, bd) = _rg("layernorm", 512, 1024, 256, 512, False, seed=33)
    dC = fn.gemm_ex(G.to(DEV), W.to(DEV), trans_b=True)
    un = fn.gemm_postnorm_backward(Ad, Bd, C, dC, st["rstd"], "layernorm", gd, bd)
    fn.check_status(DEV)
    for k in ("dH", "dA", "dB", "dgamma", "dbeta"):
        assert_out_close(got[k], np64(un[k]), f"regrouped vs unfused {k}")
        assert_out_close(un[k], ref[k], f"unfused {k} vs oracle")


@pytest.mark.parametrize("cluster", [1, 2, 4])
def test_postnorm_backward_regrouped_cluster_sizes(cluster):
    try:
        fn.set_postnorm_cluster(cluster)
        got, ref, _ = _rg("layernorm", 264, 256, 64, 128, True, seed=35)
    finally:
        fn.set_postnorm_cluster(0)
    for k in ("dH", "dA", "dB", "dgamma", "dbeta"):
        assert_out_close(got[k], ref[k], f"cluster {cluster}: {k}")


def test_postnorm_backward_regrouped_deterministic():
    a, _, _ = _rg("rmsnorm", 1000, 1024, 64, 128, False, seed=37)
    b, _, _ = _rg("rmsnorm", 1000, 1024, 64, 128, False, seed=37)
    for k in ("dH", "dA", "dgamma", "dbeta"):
        assert torch.equal(a[k], b[k]), f"{k} differs between two runs"


def test_postnorm_backward_regrouped_wide_rows_need_a_workspace():
    w = WORKLOADS["cfg2_n128"].scaled(M=128, N=2048, K=64)
    d = make_inputs(w, 39)
    A, B = d["A"].to(DEV), d["B"].to(DEV)
    C, st = fn.gemm_postnorm(A, B, "layernorm", return_stats=True)
    G = torch.randn(128, 64, device=DEV).to(torch.bfloat16)
    W = torch.randn(2048, 64, device=DEV).to(torch.bfloat16)
    with pytest.raises(fn.FnormError) as e:
        fn.gemm_postnorm_backward_regrouped(G, W, A, B, C, st["rstd"], "layernorm", workspace=False)
    assert e.value.status == fn.UNSUPPORTED and "workspace" in str(e.value)


@pytest.mark.parametrize("name", ["postnorm_bwd", "postnorm_bwd_rg", "postnorm_bwd_rg_n4096"])
def test_postnorm_backward_full_size(name):
    # the bench's post-norm backward workloads in their launch configuration,
    # every gradient element against the oracle at full size
    w = WORKLOADS[name]
    d = make_inputs(w, 0)
    Ad, Bd, gd, bd = d["A"].to(DEV), d["B"].to(DEV), d["gamma"].to(DEV), d["beta"].to(DEV)
    C, st = fn.gemm_postnorm(Ad, Bd, w.norm, gd, bd, w.eps, return_stats=True)
    g64, b64 = to_f64(d["gamma"]), to_f64(d["beta"])
    if w.kind == "postnorm_backward":
        got = fn.gemm_postnorm_backward(Ad, Bd, C, d["dC"].to(DEV), st["rstd"], w.norm, gd, bd)
        fn.check_status(DEV)
        ref = oracle.gemm_postnorm_backward(to_f64(d["A"]), to_f64(d["B"]), to_f64(d["dC"]), w.norm, g64, b64, w.eps)
    else:
        got = fn.gemm_postnorm_backward_regrouped(d["G"].to(DEV), d["W"].to(DEV), Ad, Bd, C, st["rstd"], w.norm, gd,
                                                  bd)
        fn.check_status(DEV)
        ref = oracle.gemm_postnorm_backward_regrouped(to_f64(d["G"]), to_f64(d["W"]), to_f64(d["A"]),
                                                      to_f64(d["B"]), w.norm, g64, b64, w.eps)
    for k in ("dH", "dA", "dB", "dgamma", "dbeta"):
        assert_out_close(got[k], ref[k], f"{name} {k} (every element)")


def test_postnorm_backward_regrouped_empty_batch():
    # M = 0: dB, dgamma and dbeta are zero, nothing else is touched
    A = torch.empty(0, 64, dtype=torch.bfloat16, device=DEV)
    B = torch.randn(64, 256, device=DEV).to(torch.bfloat16)
    C = torch.empty(0, 256, dtype=torch.bfloat16, device=DEV)
    G = torch.empty(0, 128, dtype=torch.bfloat16, device=DEV)
    W = torch.randn(256, 128, device=DEV).to(torch.bfloat16)
    got = fn.gemm_postnorm_backward_regrouped(G, W, A, B, C, torch.empty(0, device=DEV), "layernorm")
    fn.check_status(DEV)
    assert got["dA"].shape == (0, 64) and torch.all(got["dB"] == 0)
    assert torch.all(got["dgamma"] == 0) and torch.all(got["dbeta"] == 0)
