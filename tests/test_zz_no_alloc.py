"""The allocation-free post-norm entry point (collected last on purpose: it
must agree with the workspace entry point whether it runs alone or after
every other test, i.e. whatever state the library's fixed workspace was left
in; each test also runs a differently shaped call first, so the fixed
workspace's counters are never fresh when the compared calls start).

fnorm_gemm_postnorm_noalloc keeps the wide-row grid exchange's statistics in
a fixed device array instead of a caller's workspace; results must equal
fnorm_gemm_postnorm_ws's bit for bit (same kernels, same plan), on two calls
in a row, and shapes past the array must be refused with a clear error.
"""
import numpy as np
import pytest
import torch

import normalization_gemm_tcgen05_gb300 as fn
import oracle
from gpu_util import assert_out_close
from workloads import WORKLOADS, make_inputs, to_f64

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)

CASES = [("layernorm", 1024, 4096, 256),   # wide rows: the grid exchange, fixed workspace
         ("rmsnorm", 640, 8192, 128),
         ("layernorm", 300, 512, 128),     # resident cluster: no workspace at all
         ("layernorm", 200, 128, 64)]      # one CTA per row block


@pytest.mark.parametrize("norm,M,N,K", CASES, ids=lambda v: str(v))
def test_noalloc_matches_postnorm_twice(norm, M, N, K):
    w = WORKLOADS["cfg4_n4096_ln"].scaled(M=M, N=N, K=K, b_std=1.0 / np.sqrt(K))
    d = make_inputs(w, M + N)
    A, B = d["A"].to(DEV), d["B"].to(DEV)
    g = d["gamma"].to(DEV)
    b = d["beta"].to(DEV) if norm == "layernorm" else None
    C0, st0 = fn.gemm_postnorm(A, B, norm, g, b, w.eps, return_stats=True)
    # a wide RMSNorm call of another shape through the fixed workspace first
    Mw, Nw = 384, 8192
    Aw = torch.randn(Mw, 64, device=DEV).to(torch.bfloat16)
    Bw = torch.randn(64, Nw, device=DEV).to(torch.bfloat16)
    fn.gemm_postnorm_noalloc(Aw, Bw, torch.empty(Mw, Nw, dtype=torch.bfloat16, device=DEV), "rmsnorm")
    for _ in range(2):  # two calls in a row: the second reuses the counters
        C = torch.empty_like(C0)
        rstd = torch.empty(M, dtype=torch.float32, device=DEV)
        mean = torch.empty(M, dtype=torch.float32, device=DEV) if norm == "layernorm" else None
        fn.gemm_postnorm_noalloc(A, B, C, norm, g, b, w.eps, mean_out=mean, rstd_out=rstd)
        fn.check_status(DEV)
        assert torch.equal(C, C0)
        assert torch.equal(rstd, st0["rstd"])
        if mean is not None:
            assert torch.equal(mean, st0["mean"])
    ref = oracle.gemm_postnorm(to_f64(d["A"]), to_f64(d["B"]), norm, to_f64(d["gamma"]),
                               to_f64(d["beta"]) if norm == "layernorm" else None, w.eps)
    assert_out_close(C0, ref["C"], f"{norm} {M}x{N}x{K} vs oracle")


def test_noalloc_refuses_a_shape_past_its_workspace():
    # 2049 row blocks of one 1032-column chunk: 2049 units > 2048
    M, N, K = 128 * 2049, 1032, 64
    A = torch.zeros(M, K, dtype=torch.bfloat16, device=DEV)
    B = torch.zeros(K, N, dtype=torch.bfloat16, device=DEV)
    C = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(fn.FnormError) as e:
        fn.gemm_postnorm_noalloc(A, B, C, "layernorm")
    assert e.value.status == fn.UNSUPPORTED and "workspace" in str(e.value)
    fn.gemm_postnorm(A, B, "layernorm", out=C)  # the allocating entry point takes it
    fn.check_status(DEV)
    assert torch.all(C == 0)
