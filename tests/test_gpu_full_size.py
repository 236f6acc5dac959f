"""GPU parity at the full workload sizes, in the launch configuration bench.py times.

The fused kernel runs over the whole workload and every output element is
compared with the fp64 oracle, together with the row statistics of every row
(post-norm mean and rstd, pre-norm rstd and mean).  Rows of the path are
independent, so the oracle is evaluated on consecutive blocks of rows (its
own definition applied to fewer rows at a time, which bounds the host memory
of the largest workloads); the tolerance is applied over all of them at once.
(The backward's full-size case is in test_gpu_backward.py.)
"""
import numpy as np
import pytest
import torch

import normalization_gemm_tcgen05_gb300 as fn
import oracle
from gpu_util import OUT_ABS, OUT_REL, assert_mean_close, assert_rstd_close, np64
from workloads import WORKLOADS, make_inputs, to_f64

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
ROWS_PER_BLOCK = 2048


class FullCompare:
    """Running max |C_gpu - C_ref| and max |C_ref| over blocks of rows, so the
    output bound max|err| <= 2e-2 * max|C_ref| + 1e-3 holds over the whole
    output; statistics are gathered for a check over every row."""

    def __init__(self, M):
        self.err = 0.0
        self.ref_max = 0.0
        self.stats = {}
        self.M = M

    def add(self, got, ref, r0):
        g = np64(got)
        assert np.all(np.isfinite(g)), f"non-finite output in rows {r0}.."
        self.err = max(self.err, float(np.max(np.abs(g - ref))))
        self.ref_max = max(self.ref_max, float(np.max(np.abs(ref))))

    def add_stat(self, key, r0, vals):
        if key not in self.stats:
            self.stats[key] = np.zeros(self.M)
        self.stats[key][r0:r0 + len(vals)] = vals

    def check(self, what):
        bound = OUT_REL * self.ref_max + OUT_ABS
        assert self.err <= bound, f"{what}: max |err| {self.err:.4e} > bound {bound:.4e} over every element"


@pytest.mark.parametrize("name", sorted(n for n, w in WORKLOADS.items() if not w.kind.endswith("_backward")))
def test_full_size(name):
    w = WORKLOADS[name]
    d = make_inputs(w, 0)
    A, B = d["A"].to(DEV), d["B"].to(DEV)
    A64, B64 = to_f64(d["A"]), to_f64(d["B"])
    g64, b64 = to_f64(d["gamma"]), to_f64(d["beta"])
    g = None if d["gamma"] is None else d["gamma"].to(DEV)
    b = None if d["beta"] is None else d["beta"].to(DEV)
    st = {}
    if w.kind == "prenorm":
        C, st["rstd"] = fn.lazy_prenorm_gemm(A, B, w.eps, return_rstd=True)
    elif w.kind == "prenorm_affine":
        Bf, colsum, bias = fn.fold_prenorm_affine(B, g, b)
        C, st = fn.prenorm_gemm(A, Bf, w.norm, colsum, bias, w.eps, return_stats=True)
    elif w.residual:
        C, st = fn.gemm_add_postnorm(A, B, d["R"].to(DEV), w.norm, g, b, w.eps, return_stats=True)
    else:
        C, st = fn.gemm_postnorm(A, B, w.norm, g, b, w.eps, pre_rmsnorm=w.pre_rmsnorm, pre_eps=w.pre_eps,
                                 return_stats=True)
    fn.check_status(DEV)
    Ch = C.cpu()
    st = {k: np64(v) for k, v in st.items() if v is not None}
    cmp = FullCompare(w.M)
    R64 = to_f64(d["R"]) if w.residual else None
    for r0 in range(0, w.M, ROWS_PER_BLOCK):
        rows = slice(r0, min(w.M, r0 + ROWS_PER_BLOCK))
        if w.kind == "prenorm":
            Cr, rr = oracle.lazy_prenorm_gemm(A64[rows], B64, w.eps)
            cmp.add_stat("rstd", r0, rr)
        elif w.kind == "prenorm_affine":
            Cr, mr, rr = oracle.prenorm_affine_gemm(A64[rows], B64, w.norm, g64, b64, w.eps)
            cmp.add_stat("rstd", r0, rr)
            if mr is not None:
                cmp.add_stat("mean", r0, mr)
        else:
            if w.residual:
                ref = oracle.gemm_add_postnorm(A64[rows], B64, R64[rows], w.norm, g64, b64, w.eps)
            else:
                ref = oracle.gemm_postnorm(A64[rows], B64, w.norm, g64, b64, w.eps, pre_rmsnorm=w.pre_rmsnorm,
                                           pre_eps=w.pre_eps)
            Cr = ref["C"]
            cmp.add_stat("rstd", r0, ref["rstd"])
            if ref["mean"] is not None:
                cmp.add_stat("mean", r0, ref["mean"])
            if ref.get("pre_rstd") is not None:
                cmp.add_stat("pre_rstd", r0, ref["pre_rstd"])
        cmp.add(Ch[rows], Cr, r0)
    cmp.check(f"{name} (every element)")
    assert_rstd_close(torch.from_numpy(st["rstd"]), cmp.stats["rstd"], f"{name} rstd (every row)")
    if "mean" in cmp.stats:
        assert_mean_close(torch.from_numpy(st["mean"]), cmp.stats["mean"], cmp.stats["rstd"],
                          f"{name} mean (every row)")
    if "pre_rstd" in cmp.stats:
        assert_rstd_close(torch.from_numpy(st["pre_rstd"]), cmp.stats["pre_rstd"], f"{name} pre rstd (every row)")
