"""B shared by a 2-CTA cluster along M (TMA multicast): the same arithmetic as
the one-CTA tiles, so every output and statistic must agree bit for bit, on
row-block counts that pair up and on odd ones (the second CTA of the last
cluster then has no rows), and match the fp64 oracle.  The forward GEMMs, the
grid exchange, the transposed-operand GEMMs (B^T loaded as two half boxes,
one per CTA) and the backward entry points.
"""
import numpy as np
import pytest
import torch

import normalization_gemm_tcgen05_gb300 as fn
import oracle
from gpu_util import assert_out_close, assert_rstd_close
from workloads import WORKLOADS, make_inputs, to_f64

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


def _both(call):
    """call() with B multicast forced off, then on; returns both results."""
    out = []
    try:
        for mode in (0, 1):
            fn.set_b_multicast(mode)
            out.append(call())
            fn.check_status(DEV)
    finally:
        fn.set_b_multicast(-1)
    return out


def _equal(a, b, what):
    if isinstance(a, torch.Tensor):
        assert torch.equal(a, b), f"{what}: B multicast differs from one-CTA tiles"
    elif isinstance(a, dict):
        for k in a:
            if a[k] is not None:
                _equal(a[k], b[k], f"{what} {k}")
    else:
        for i, (x, y) in enumerate(zip(a, b)):
            _equal(x, y, f"{what}[{i}]")


@pytest.mark.parametrize("M,N,K", [(256, 256, 128), (384, 512, 320), (1000, 768, 256), (129, 1024, 64),
                                   (2048, 4096, 512), (1, 256, 64)], ids=lambda v: str(v))
def test_gemm_multicast(M, N, K):
    w = WORKLOADS["cfg3"].scaled(M=M, N=N, K=K, b_std=1.0 / np.sqrt(K), a_row_scale=False)
    d = make_inputs(w, M + N + K)
    A, B = d["A"].to(DEV), d["B"].to(DEV)
    c0, c1 = _both(lambda: fn.gemm(A, B))
    _equal(c0, c1, "gemm")
    assert_out_close(c1, oracle.gemm(to_f64(d["A"]), to_f64(d["B"])), f"gemm {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(512, 1024, 512), (640, 4096, 256), (333, 512, 1024), (8192, 2048, 128)],
                         ids=lambda v: str(v))
def test_lazy_prenorm_multicast(M, N, K):
    w = WORKLOADS["cfg1"].scaled(M=M, N=N, K=K, b_std=1.0 / np.sqrt(K))
    d = make_inputs(w, M * 3 + K)
    A, B = d["A"].to(DEV), d["B"].to(DEV)
    r0, r1 = _both(lambda: fn.lazy_prenorm_gemm(A, B, w.eps, return_rstd=True))
    _equal(r0, r1, "lazy prenorm")
    Cr, rr = oracle.lazy_prenorm_gemm(to_f64(d["A"]), to_f64(d["B"]), w.eps)
    assert_out_close(r1[0], Cr, "lazy prenorm C")
    assert_rstd_close(r1[1], rr, "lazy prenorm rstd")


@pytest.mark.parametrize("norm", ["layernorm", "rmsnorm"])
def test_prenorm_affine_multicast(norm):
    w = WORKLOADS["preln_affine" if norm == "layernorm" else "prerms_gamma"].scaled(M=520, K=512, N=768)
    d = make_inputs(w, 61)
    A, B = d["A"].to(DEV), d["B"].to(DEV)
    g = d["gamma"].to(DEV)
    b = None if d["beta"] is None else d["beta"].to(DEV)
    Bf, colsum, bias = fn.fold_prenorm_affine(B, g, b)
    r0, r1 = _both(lambda: fn.prenorm_gemm(A, Bf, norm, colsum if norm == "layernorm" else None, bias, w.eps,
                                           return_stats=True))
    _equal(r0, r1, "prenorm affine")
    Cr, _, rr = oracle.prenorm_affine_gemm(to_f64(d["A"]), to_f64(d["B"]), norm, to_f64(d["gamma"]),
                                           to_f64(d["beta"]), w.eps)
    assert_out_close(r1[0], Cr, "prenorm affine C")
    assert_rstd_close(r1[1]["rstd"], rr, "prenorm affine rstd")


@pytest.mark.parametrize("M,N", [(520, 4096), (128 * 33, 2048), (300, 8192), (128 * 160 + 37, 3072)],
                         ids=lambda v: str(v))
@pytest.mark.parametrize("norm", ["layernorm", "rmsnorm"])
def test_grid_exchange_multicast(norm, M, N):
    w = WORKLOADS["cfg4_n4096_ln"].scaled(M=M, N=N, K=128)
    d = make_inputs(w, M + N + (norm == "rmsnorm"))
    A, B = d["A"].to(DEV), d["B"].to(DEV)
    g = d["gamma"].to(DEV)
    b = d["beta"].to(DEV) if norm == "layernorm" else None
    r0, r1 = _both(lambda: fn.gemm_postnorm(A, B, norm, g, b, w.eps, return_stats=True))
    _equal(r0, r1, "grid exchange")
    ref = oracle.gemm_postnorm(to_f64(d["A"]), to_f64(d["B"]), norm, to_f64(d["gamma"]),
                               to_f64(d["beta"]) if norm == "layernorm" else None, w.eps)
    assert_out_close(r1[0], ref["C"], f"grid exchange {norm} C")
    assert_rstd_close(r1[1]["rstd"], ref["rstd"], f"grid exchange {norm} rstd")


def test_grid_exchange_multicast_with_pre():
    w = WORKLOADS["cfg5"].scaled(M=700, N=4096, K=256)
    d = make_inputs(w, 71)
    A, B = d["A"].to(DEV), d["B"].to(DEV)
    g, b = d["gamma"].to(DEV), d["beta"].to(DEV)
    r0, r1 = _both(lambda: fn.gemm_postnorm(A, B, "layernorm", g, b, w.eps, pre_rmsnorm=True, pre_eps=w.pre_eps,
                                            return_stats=True))
    _equal(r0, r1, "grid exchange with pre-norm")
    ref = oracle.gemm_postnorm(to_f64(d["A"]), to_f64(d["B"]), "layernorm", to_f64(d["gamma"]),
                               to_f64(d["beta"]), w.eps, pre_rmsnorm=True, pre_eps=w.pre_eps)
    assert_out_close(r1[0], ref["C"], "grid exchange with pre-norm C")
    assert_rstd_close(r1[1]["pre_rstd"], ref["pre_rstd"], "pre rstd")


# The transposed-operand GEMMs, from their row-major sources: (M, N, K,
# trans_a, trans_b), 256-column tiles, even and odd row-block counts, ragged K
TRANSPOSED = [(2048, 4096, 320, True, False), (1288, 2560, 200, False, True), (1288, 2560, 136, True, True),
              (1032, 3072, 64, True, False)]


@pytest.mark.parametrize("M,N,K,ta,tb", TRANSPOSED, ids=lambda v: str(v))
def test_transposed_gemm_multicast(M, N, K, ta, tb):
    w = WORKLOADS["cfg3"].scaled(M=M, N=N, K=K, b_std=1.0 / np.sqrt(K), a_row_scale=False)
    d = make_inputs(w, M + N + K + ta + 2 * tb)
    A = (d["A"].t().contiguous() if ta else d["A"]).to(DEV)
    B = (d["B"].t().contiguous() if tb else d["B"]).to(DEV)
    c0, c1 = _both(lambda: fn.gemm_ex(A, B, trans_a=ta, trans_b=tb))
    _equal(c0, c1, "transposed gemm")
    assert_out_close(c1, oracle.gemm(to_f64(d["A"]), to_f64(d["B"])), f"gemm_ex {M}x{N}x{K} {ta} {tb}")


def test_lazy_prenorm_backward_multicast():
    # dgrad [1288 x 2560] and wgrad [2560 x 1024]: both on 256-column tiles
    M, N, K = 1288, 1024, 2560
    w = WORKLOADS["prenorm_bwd"].scaled(M=M, N=N, K=K, b_std=1.0 / np.sqrt(K))
    d = make_inputs(w, 83)
    Ad, Bd, dCd = d["A"].to(DEV), d["B"].to(DEV), d["dC"].to(DEV)
    C, rstd = fn.lazy_prenorm_gemm(Ad, Bd, w.eps, return_rstd=True)
    r0, r1 = _both(lambda: fn.lazy_prenorm_gemm_backward(Ad, Bd, C, dCd, rstd))
    _equal(r0, r1, "lazy prenorm backward")
    rA, rB, _ = oracle.lazy_prenorm_gemm_backward(to_f64(d["A"]), to_f64(d["B"]), to_f64(d["dC"]), w.eps)
    assert_out_close(r1[0], rA, "lazy prenorm backward dA")
    assert_out_close(r1[1], rB, "lazy prenorm backward dB")


_PLAIN_GX_CHILD = """
import sys, torch
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import normalization_gemm_tcgen05_gb300 as fn
from workloads import WORKLOADS, make_inputs
w = WORKLOADS["cfg4_n4096_ln"].scaled(M=1300, N=2048, K=192)
d = make_inputs(w, 97)
dev = torch.device("cuda", 0)
C, st = fn.gemm_postnorm(d["A"].to(dev), d["B"].to(dev), "layernorm", d["gamma"].to(dev), d["beta"].to(dev), w.eps,
                         return_stats=True)
fn.check_status(dev)
torch.save({{"C": C.cpu(), "rstd": st["rstd"].cpu(), "mean": st["mean"].cpu()}}, {out!r})
"""


def test_plain_cluster_grid_exchange_launch_matches(tmp_path):
    # FNORM_PLAIN_GX_LAUNCH=1 (read once per process, so in a child process)
    # launches the clustered grid exchange as a plain cluster launch, for
    # profilers; the kernel is the same, so the results are bit for bit the
    # default cooperative launch's
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = str(tmp_path / "plain.pt")
    code = _PLAIN_GX_CHILD.format(root=root, tests=os.path.join(root, "tests"), out=out)
    env = dict(os.environ, FNORM_PLAIN_GX_LAUNCH="1")
    subprocess.run([sys.executable, "-c", code], env=env, check=True, timeout=600)
    plain = torch.load(out)
    w = WORKLOADS["cfg4_n4096_ln"].scaled(M=1300, N=2048, K=192)
    d = make_inputs(w, 97)
    C, st = fn.gemm_postnorm(d["A"].to(DEV), d["B"].to(DEV), "layernorm", d["gamma"].to(DEV), d["beta"].to(DEV),
                             w.eps, return_stats=True)
    fn.check_status(DEV)
    assert torch.equal(C.cpu(), plain["C"]), "plain cluster launch differs from the cooperative launch"
    assert torch.equal(st["rstd"].cpu(), plain["rstd"]) and torch.equal(st["mean"].cpu(), plain["mean"])


def test_multicast_setter_rejects_bad_modes():
    for bad in (2, -2):
        with pytest.raises(fn.FnormError):
            fn.set_b_multicast(bad)
    fn.set_b_multicast(-1)
