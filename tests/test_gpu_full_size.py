"""GPU parity at the full workload sizes, in the launch configuration bench.py times.

The fused kernel runs over the whole workload; the fp64 oracle recomputes a
sample of rows one by one (first and last rows, tile boundaries, seeded random
rows and, for the outlier workload, outlier rows), all N columns each, since
rows of the path are independent.  (The backward's full-size case is in
test_gpu_backward.py.)  The pre-norm statistics (rstd, and the
mean of a pre-LayerNorm) are compared on every row (they depend on A alone).
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


def _rows(w, outliers, seed):
    rng = np.random.default_rng(seed)
    picks = list(range(min(16, w.M))) + list(range(max(0, w.M - 16), w.M))
    for b in (127, 128, 255, 256):
        if b < w.M:
            picks.append(b)
    picks += list(rng.choice(w.M, size=min(32, w.M), replace=False))
    picks += list(outliers[:16])
    return np.unique(np.asarray(picks, dtype=np.int64))


@pytest.mark.parametrize("name", sorted(n for n, w in WORKLOADS.items() if not w.kind.endswith("_backward")))
def test_full_size(name):
    w = WORKLOADS[name]
    d = make_inputs(w, 0)
    A, B = d["A"].to(DEV), d["B"].to(DEV)
    rows = _rows(w, d["outliers"], seed=len(name))
    A64 = to_f64(d["A"])
    if w.kind == "prenorm":
        C, rstd = fn.lazy_prenorm_gemm(A, B, w.eps, return_rstd=True)
        Cr, rr = oracle.lazy_prenorm_gemm(A64[rows], to_f64(d["B"]), w.eps)
        assert_out_close(C[torch.from_numpy(rows).to(DEV)], Cr, f"{name} sampled rows")
        _, r_all = oracle.rmsnorm(A64, None, None, w.eps)
        assert_rstd_close(rstd, r_all, f"{name} rstd (all rows)")
    elif w.kind == "prenorm_affine":
        g = None if d["gamma"] is None else d["gamma"].to(DEV)
        be = None if d["beta"] is None else d["beta"].to(DEV)
        Bf, colsum, bias = fn.fold_prenorm_affine(B, g, be)
        C, st = fn.prenorm_gemm(A, Bf, w.norm, colsum, bias, w.eps, return_stats=True)
        Cr, _, _ = oracle.prenorm_affine_gemm(A64[rows], to_f64(d["B"]), w.norm, to_f64(d["gamma"]),
                                              to_f64(d["beta"]), w.eps)
        assert_out_close(C[torch.from_numpy(rows).to(DEV)], Cr, f"{name} sampled rows")
        if w.norm == "layernorm":
            _, m_all, r_all = oracle.layernorm(A64, None, None, w.eps)
            assert_mean_close(st["mean"], m_all, r_all, f"{name} mean (all rows)")
        else:
            _, r_all = oracle.rmsnorm(A64, None, None, w.eps)
        assert_rstd_close(st["rstd"], r_all, f"{name} rstd (all rows)")
    elif w.residual:
        g = None if d["gamma"] is None else d["gamma"].to(DEV)
        b = None if d["beta"] is None else d["beta"].to(DEV)
        C, st = fn.gemm_add_postnorm(A, B, d["R"].to(DEV), w.norm, g, b, w.eps, return_stats=True)
        ref = oracle.gemm_add_postnorm(A64[rows], to_f64(d["B"]), to_f64(d["R"])[rows], w.norm,
                                       to_f64(d["gamma"]), to_f64(d["beta"]), w.eps)
        idx = torch.from_numpy(rows).to(DEV)
        assert_out_close(C[idx], ref["C"], f"{name} sampled rows")
        assert_rstd_close(st["rstd"][idx], ref["rstd"], f"{name} rstd")
        if w.norm == "layernorm":
            assert_mean_close(st["mean"][idx], ref["mean"], ref["rstd"], f"{name} mean")
    else:
        g = None if d["gamma"] is None else d["gamma"].to(DEV)
        b = None if d["beta"] is None else d["beta"].to(DEV)
        C, st = fn.gemm_postnorm(A, B, w.norm, g, b, w.eps, pre_rmsnorm=w.pre_rmsnorm, pre_eps=w.pre_eps,
                                 return_stats=True)
        ref = oracle.gemm_postnorm(A64[rows], to_f64(d["B"]), w.norm, to_f64(d["gamma"]), to_f64(d["beta"]),
                                   w.eps, pre_rmsnorm=w.pre_rmsnorm, pre_eps=w.pre_eps)
        idx = torch.from_numpy(rows).to(DEV)
        assert_out_close(C[idx], ref["C"], f"{name} sampled rows")
        assert_rstd_close(st["rstd"][idx], ref["rstd"], f"{name} rstd")
        if w.norm == "layernorm":
            assert_mean_close(st["mean"][idx], ref["mean"], ref["rstd"], f"{name} mean")
        if w.pre_rmsnorm:
            _, pr_all = oracle.rmsnorm(A64, None, None, w.pre_eps)
            assert_rstd_close(st["pre_rstd"], pr_all, f"{name} pre rstd (all rows)")
    fn.check_status(DEV)
    assert torch.isfinite(C.float()).all()
