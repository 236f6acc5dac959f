"""Seeded random sweep of every fused form against the fp64 oracle.

Shapes are drawn at random (ragged M from 1 row up, N and K any multiple of 8)
so that they land in every layout class: one CTA per row, resident clusters,
the grid-wide exchange, resident B, B multicast over 2-CTA clusters, the
transposed operands, ragged tails of every tile dimension.  Every entry point
of the path is drawn: the fused forward forms, the backward entry points, the
allocation-free post-norm and the standalone comparison norms.
Every output element and every row statistic is compared; the draws are
fixed by the seeds, so a failure reproduces.
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


def _shapes(seed, n):
    rng = np.random.default_rng(seed)
    return [(int(rng.integers(1, 1500)), int(8 * rng.integers(1, 700)), int(8 * rng.integers(1, 160)))
            for _ in range(n)]


FORMS = ["gemm", "prenorm", "post_ln", "post_rms", "pre_post_ln", "res_rms", "preaff_ln", "regrouped_ln", "gemm_ex",
         "prenorm_bwd", "postnorm_bwd", "rownorm", "add_rownorm", "noalloc_ln"]
CASES = [(form, M, N, K) for i, form in enumerate(FORMS) for (M, N, K) in _shapes(100 + i, 12)]

# the opt-in paths: two-CTA MMA, B multicast off and forced on, forced cluster sizes
KNOBS = [("pair", 1), ("mcb", 0), ("mcb", 1), ("cluster", 2), ("cluster", 4)]
KNOB_CASES = [(knob, v, form, M, N, K) for j, (knob, v) in enumerate(KNOBS)
              for i, form in enumerate(("gemm", "prenorm", "post_ln", "post_rms", "gemm_ex"))
              for (M, N, K) in _shapes(200 + 10 * j + i, 2)
              if not (knob == "cluster" and form in ("gemm", "prenorm", "gemm_ex"))]


def _dev(t):
    return None if t is None else t.to(DEV)


@pytest.mark.parametrize("form,M,N,K", CASES, ids=lambda v: str(v))
def test_random_shape(form, M, N, K):
    _run(form, M, N, K)


@pytest.mark.parametrize("knob,value,form,M,N,K", KNOB_CASES, ids=lambda v: str(v))
def test_random_shape_opt_in_paths(knob, value, form, M, N, K):
    # (a forced cluster too narrow for the row takes the spill layout)
    setter = {"pair": fn.set_pair_mma, "mcb": fn.set_b_multicast, "cluster": fn.set_postnorm_cluster}[knob]
    try:
        setter(value)
        _run(form, M, N, K)
    finally:
        setter(0 if knob == "cluster" else -1)


def _run(form, M, N, K):
    seed = M * 7 + N * 3 + K
    what = f"{form} {M}x{N}x{K}"
    if form == "gemm":
        w = WORKLOADS["cfg3"].scaled(M=M, N=N, K=K, b_std=1.0 / np.sqrt(K), a_row_scale=False)
        d = make_inputs(w, seed)
        C = fn.gemm(_dev(d["A"]), _dev(d["B"]))
        fn.check_status(DEV)
        assert_out_close(C, oracle.gemm(to_f64(d["A"]), to_f64(d["B"])), what)
    elif form == "prenorm":
        w = WORKLOADS["cfg1"].scaled(M=M, N=N, K=K, b_std=1.0 / np.sqrt(K))
        d = make_inputs(w, seed)
        C, rstd = fn.lazy_prenorm_gemm(_dev(d["A"]), _dev(d["B"]), w.eps, return_rstd=True)
        fn.check_status(DEV)
        Cr, rr = oracle.lazy_prenorm_gemm(to_f64(d["A"]), to_f64(d["B"]), w.eps)
        assert_out_close(C, Cr, what)
        assert_rstd_close(rstd, rr, what + " rstd")
    elif form in ("post_ln", "post_rms", "pre_post_ln"):
        base = {"post_ln": "cfg4_n4096_ln", "post_rms": "cfg4_n4096_rms", "pre_post_ln": "cfg5"}[form]
        w = WORKLOADS[base].scaled(M=M, N=N, K=K, b_std=1.0 / np.sqrt(K))
        d = make_inputs(w, seed)
        C, st = fn.gemm_postnorm(_dev(d["A"]), _dev(d["B"]), w.norm, _dev(d["gamma"]), _dev(d["beta"]), w.eps,
                                 pre_rmsnorm=w.pre_rmsnorm, pre_eps=w.pre_eps, return_stats=True)
        fn.check_status(DEV)
        ref = oracle.gemm_postnorm(to_f64(d["A"]), to_f64(d["B"]), w.norm, to_f64(d["gamma"]), to_f64(d["beta"]),
                                   w.eps, pre_rmsnorm=w.pre_rmsnorm, pre_eps=w.pre_eps)
        assert_out_close(C, ref["C"], what)
        assert_rstd_close(st["rstd"], ref["rstd"], what + " rstd")
        if w.pre_rmsnorm:
            assert_rstd_close(st["pre_rstd"], ref["pre_rstd"], what + " pre rstd")
    elif form == "res_rms":
        w = WORKLOADS["res_rms_n1024"].scaled(M=M, N=N, K=K, b_std=1.0 / np.sqrt(K))
        d = make_inputs(w, seed)
        C, st = fn.gemm_add_postnorm(_dev(d["A"]), _dev(d["B"]), _dev(d["R"]), w.norm, _dev(d["gamma"]), None, w.eps,
                                     return_stats=True)
        fn.check_status(DEV)
        ref = oracle.gemm_add_postnorm(to_f64(d["A"]), to_f64(d["B"]), to_f64(d["R"]), w.norm, to_f64(d["gamma"]),
                                       None, w.eps)
        assert_out_close(C, ref["C"], what)
        assert_rstd_close(st["rstd"], ref["rstd"], what + " rstd")
    elif form == "preaff_ln":
        w = WORKLOADS["preln_affine"].scaled(M=M, N=N, K=K, b_std=1.0 / np.sqrt(K))
        d = make_inputs(w, seed)
        Bf, colsum, bias = fn.fold_prenorm_affine(_dev(d["B"]), _dev(d["gamma"]), _dev(d["beta"]))
        C = fn.prenorm_gemm(_dev(d["A"]), Bf, "layernorm", colsum, bias, w.eps)
        fn.check_status(DEV)
        Cr, _, _ = oracle.prenorm_affine_gemm(to_f64(d["A"]), to_f64(d["B"]), "layernorm", to_f64(d["gamma"]),
                                              to_f64(d["beta"]), w.eps)
        assert_out_close(C, Cr, what)
    elif form == "gemm_ex":
        # op(A) from an A^T source ([K, M]; M a multiple of 8) and/or op(B) from a B^T source ([N, K])
        ta, tb = bool((seed >> 1) & 1) and M % 8 == 0, bool((seed >> 2) & 1)
        w = WORKLOADS["cfg3"].scaled(M=M, N=N, K=K, b_std=1.0 / np.sqrt(K), a_row_scale=False)
        d = make_inputs(w, seed)
        A = d["A"].t().contiguous() if ta else d["A"]
        B = d["B"].t().contiguous() if tb else d["B"]
        C = fn.gemm_ex(_dev(A), _dev(B), trans_a=ta, trans_b=tb)
        fn.check_status(DEV)
        assert_out_close(C, oracle.gemm(to_f64(d["A"]), to_f64(d["B"])), f"{what} trans_a={ta} trans_b={tb}")
    elif form == "prenorm_bwd":
        w = WORKLOADS["prenorm_bwd"].scaled(M=M, N=N, K=K, b_std=1.0 / np.sqrt(K))
        d = make_inputs(w, seed)
        Ad, Bd = _dev(d["A"]), _dev(d["B"])
        C, rstd = fn.lazy_prenorm_gemm(Ad, Bd, w.eps, return_rstd=True)
        dA, dB = fn.lazy_prenorm_gemm_backward(Ad, Bd, C, _dev(d["dC"]), rstd, need_dB=M % 8 == 0)
        fn.check_status(DEV)
        rA, rB, _ = oracle.lazy_prenorm_gemm_backward(to_f64(d["A"]), to_f64(d["B"]), to_f64(d["dC"]), w.eps)
        assert_out_close(dA, rA, what + " dA")
        if dB is not None:
            assert_out_close(dB, rB, what + " dB")
    elif form == "postnorm_bwd":
        # the post-norm backward from a given dC (the unfused comparison path)
        norm = "layernorm" if seed & 1 else "rmsnorm"
        w = WORKLOADS["cfg4_n1024_ln" if norm == "layernorm" else "cfg4_n1024_rms"].scaled(M=M, N=N, K=K,
                                                                                          b_std=1.0 / np.sqrt(K))
        d = make_inputs(w, seed)
        Ad, Bd, gd, bd = _dev(d["A"]), _dev(d["B"]), _dev(d["gamma"]), _dev(d["beta"])
        dC = torch.from_numpy(np.random.default_rng(seed + 1).standard_normal((M, N), dtype=np.float32)).to(torch.bfloat16)
        C, st = fn.gemm_postnorm(Ad, Bd, norm, gd, bd, w.eps, return_stats=True)
        need = ("dA", "dB", "dgamma", "dbeta") if M % 8 == 0 else ("dA", "dgamma", "dbeta")
        got = fn.gemm_postnorm_backward(Ad, Bd, C, _dev(dC), st["rstd"], norm, gd, bd, need=need)
        fn.check_status(DEV)
        ref = oracle.gemm_postnorm_backward(to_f64(d["A"]), to_f64(d["B"]), to_f64(dC), norm, to_f64(d["gamma"]),
                                            to_f64(d["beta"]), w.eps)
        for k in need + ("dH",):
            assert_out_close(got[k], ref[k], f"{what} {norm} {k}")
    elif form in ("rownorm", "add_rownorm"):
        # the standalone norms (the unfused comparison kernels): M rows of N columns
        norm = "layernorm" if seed & 1 else "rmsnorm"
        rng = np.random.default_rng(seed)
        X = torch.from_numpy(rng.standard_normal((M, N), dtype=np.float32) * 3 + 0.5).to(torch.bfloat16)
        R = torch.from_numpy(rng.standard_normal((M, N), dtype=np.float32)).to(torch.bfloat16)
        g = torch.from_numpy(1 + 0.1 * rng.standard_normal(N, dtype=np.float32)).to(torch.bfloat16)
        b = torch.from_numpy(0.1 * rng.standard_normal(N, dtype=np.float32)).to(torch.bfloat16)
        eps = 1e-5
        if form == "rownorm":
            if norm == "layernorm":
                Y, st = fn.layernorm(_dev(X), _dev(g), _dev(b), eps, return_stats=True)
                ref, mr, rr = oracle.layernorm(to_f64(X), to_f64(g), to_f64(b), eps)
            else:
                Y, rstd = fn.rmsnorm(_dev(X), _dev(g), eps, return_rstd=True)
                st = {"rstd": rstd}
                ref, rr = oracle.rmsnorm(to_f64(X), to_f64(g), None, eps)
        else:
            Y, st = fn.add_rownorm(_dev(X), _dev(R), norm, _dev(g), _dev(b) if norm == "layernorm" else None, eps,
                                   return_stats=True)
            S = to_f64(X) + to_f64(R)
            if norm == "layernorm":
                ref, mr, rr = oracle.layernorm(S, to_f64(g), to_f64(b), eps)
            else:
                ref, rr = oracle.rmsnorm(S, to_f64(g), None, eps)
        fn.check_status(DEV)
        assert_out_close(Y, ref, f"{what} {norm}")
        assert_rstd_close(st["rstd"], rr, f"{what} {norm} rstd")
    elif form == "noalloc_ln":
        # the allocation-free entry point (its fixed grid-exchange workspace for rows past 1024 columns)
        w = WORKLOADS["cfg4_n4096_ln"].scaled(M=M, N=N, K=K, b_std=1.0 / np.sqrt(K))
        d = make_inputs(w, seed)
        out = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
        rstd = torch.empty(M, dtype=torch.float32, device=DEV)
        fn.gemm_postnorm_noalloc(_dev(d["A"]), _dev(d["B"]), out, "layernorm", _dev(d["gamma"]), _dev(d["beta"]), w.eps,
                                 rstd_out=rstd)
        fn.check_status(DEV)
        ref = oracle.gemm_postnorm(to_f64(d["A"]), to_f64(d["B"]), "layernorm", to_f64(d["gamma"]), to_f64(d["beta"]),
                                   w.eps)
        assert_out_close(out, ref["C"], what)
        assert_rstd_close(rstd, ref["rstd"], what + " rstd")
    else:
        J = 8 * (1 + (seed % 97))
        trans_w = bool(seed & 1)
        w = WORKLOADS["postnorm_bwd_rg"].scaled(M=M, N=N, K=K, J=J, b_std=1.0 / np.sqrt(K))
        d = make_inputs(w, seed)
        W = d["W"] if not trans_w else d["W"].t().contiguous()
        Ad, Bd, gd, bd = _dev(d["A"]), _dev(d["B"]), _dev(d["gamma"]), _dev(d["beta"])
        C, st = fn.gemm_postnorm(Ad, Bd, w.norm, gd, bd, w.eps, return_stats=True)
        need = ("dA", "dB", "dgamma", "dbeta") if M % 8 == 0 else ("dA", "dgamma", "dbeta")
        got = fn.gemm_postnorm_backward_regrouped(_dev(d["G"]), _dev(W), Ad, Bd, C, st["rstd"], w.norm, gd, bd,
                                                  trans_w=trans_w, need=need)
        fn.check_status(DEV)
        ref = oracle.gemm_postnorm_backward_regrouped(to_f64(d["G"]), to_f64(W), to_f64(d["A"]), to_f64(d["B"]),
                                                      w.norm, to_f64(d["gamma"]), to_f64(d["beta"]), w.eps,
                                                      trans_w=trans_w)
        for k in need + ("dH",):
            assert_out_close(got[k], ref[k], f"{what} J={J} trans_w={trans_w} {k}")
