"""Plant plausible mistakes in the oracle (on the CPU) and show a pin catches each.

Every mutant replaces one function of the oracle module for the duration of a
test; the pins in ``oracle_pins`` must then fail at least once.
"""
import numpy as np
import pytest

import oracle.fnorm_oracle as O
from oracle_pins import ALL_CHECKS

_real = {name: getattr(O, name) for name in ("gemm", "rmsnorm", "layernorm", "lazy_prenorm_gemm",
                                             "gemm_postnorm", "prenorm_affine_gemm", "gemm_add_postnorm",
                                             "lazy_prenorm_gemm_backward", "gemm_postnorm_backward",
                                             "gemm_postnorm_backward_regrouped")}


def _gemm_transposed(A, B):          # transposed operand
    A = np.asarray(A, np.float64)
    B = np.asarray(B, np.float64)
    return A @ B.T


def _gemm_dropped_k(A, B):           # off-by-one k range
    A = np.asarray(A, np.float64)
    B = np.asarray(B, np.float64)
    return A[:, :-1] @ B[:-1, :]


def _rms(X, gamma=None, beta=None, eps=1e-6, *, outside=False, use_sum=False, drop_gamma=False,
         axis=1):
    X = np.asarray(X, np.float64)
    ms = np.sum(X * X, axis=axis) / (1 if use_sum else X.shape[axis])
    r = 1 / (np.sqrt(ms) + eps) if outside else 1 / np.sqrt(ms + eps)
    Y = X * (r[:, None] if axis == 1 else r[None, :])
    if gamma is not None and not drop_gamma:
        Y = Y * np.asarray(gamma, np.float64)[None, :]
    if beta is not None:
        Y = Y + np.asarray(beta, np.float64)[None, :]
    return Y, r


def _ln(X, gamma=None, beta=None, eps=1e-5, *, unbiased=False, no_center=False, drop_beta=False):
    X = np.asarray(X, np.float64)
    H = X.shape[1]
    mu = X.mean(axis=1)
    D = X - mu[:, None]
    var = (D * D).sum(axis=1) / (H - 1 if unbiased else H)
    r = 1 / np.sqrt(var + eps)
    Y = (X if no_center else D) * r[:, None]
    if gamma is not None:
        Y = Y * np.asarray(gamma, np.float64)[None, :]
    if beta is not None and not drop_beta:
        Y = Y + np.asarray(beta, np.float64)[None, :]
    return Y, mu, r


def _prenorm_cols(A, B, eps=1e-6):   # normalise A over the wrong axis
    A = np.asarray(A, np.float64)
    X = A * (1 / np.sqrt(np.mean(A * A, axis=0) + eps))[None, :]
    return _real["gemm"](X, B), 1 / np.sqrt(np.mean(A * A, axis=1) + eps)


def _postnorm_before_gemm(A, B, norm, gamma=None, beta=None, eps=1e-5, pre_rmsnorm=False,
                          pre_eps=1e-6):  # normalise A instead of A @ B
    if norm == "layernorm":
        Y, mu, r = _real["layernorm"](A, None, None, eps)
    else:
        Y, r = _real["rmsnorm"](A, None, None, eps)
        mu = None
    C = _real["gemm"](Y, B)
    if gamma is not None:
        C = C * np.asarray(gamma)[None, :]
    if beta is not None:
        C = C + np.asarray(beta)[None, :]
    return {"C": C, "mean": mu, "rstd": r, "pre_rstd": None}


def _postnorm_rms_centred(A, B, norm, gamma=None, beta=None, eps=1e-5, pre_rmsnorm=False,
                          pre_eps=1e-6):  # RMSNorm implemented as LayerNorm
    d = _real["gemm_postnorm"](A, B, "layernorm", gamma, beta, eps, pre_rmsnorm, pre_eps)
    return d


def _postnorm_skip_pre(A, B, norm, gamma=None, beta=None, eps=1e-5, pre_rmsnorm=False,
                       pre_eps=1e-6):    # forget the pre-RMSNorm stage
    d = _real["gemm_postnorm"](A, B, norm, gamma, beta, eps, False, pre_eps)
    if pre_rmsnorm:
        d["pre_rstd"] = np.ones(np.asarray(A).shape[0])
    return d


def _prenorm_affine_after_gemm(A, B, norm, gamma=None, beta=None, eps=1e-6):
    # the affine applied to the GEMM output instead of to the normalised A
    if norm == "layernorm":
        Y, mu, r = _real["layernorm"](A, None, None, eps)
    else:
        (Y, r), mu = _real["rmsnorm"](A, None, None, eps), None
    C = _real["gemm"](Y, B)
    if gamma is not None:
        C = C * np.mean(gamma)
    if beta is not None:
        C = C + np.mean(beta)
    return C, mu, r


def _add_postnorm_residual_dropped(A, B, R, norm, gamma=None, beta=None, eps=1e-5):
    d = _real["gemm_postnorm"](A, B, norm, gamma, beta, eps)
    d["H"] = _real["gemm"](A, B)
    return d


def _prenorm_bwd_no_norm_term(A, B, dC, eps=1e-6):   # dA = r * dA_hat only
    dA, dB, r = _real["lazy_prenorm_gemm_backward"](A, B, dC, eps)
    return r[:, None] * (np.asarray(dC, np.float64) @ np.asarray(B, np.float64).T), dB, r


def _prenorm_bwd_dB_unscaled(A, B, dC, eps=1e-6):    # dB from A instead of the rebuilt A_hat
    dA, dB, r = _real["lazy_prenorm_gemm_backward"](A, B, dC, eps)
    return dA, np.asarray(A, np.float64).T @ np.asarray(dC, np.float64), r


def _postnorm_bwd_no_mean_term(A, B, dC, norm, gamma=None, beta=None, eps=1e-5):
    d = _real["gemm_postnorm_backward"](A, B, dC, "rmsnorm" if norm == "layernorm" else norm, gamma, beta, eps)
    if norm == "layernorm":  # LayerNorm backward without the mean removal
        d["dbeta"] = np.sum(np.asarray(dC, np.float64), axis=0)
    return d


def _postnorm_bwd_gamma_ignored(A, B, dC, norm, gamma=None, beta=None, eps=1e-5):
    return _real["gemm_postnorm_backward"](A, B, dC, norm, None, beta, eps)


def _regrouped_w_flipped(G, W, A, B, norm, gamma=None, beta=None, eps=1e-5, trans_w=False):
    # the consumer's weight taken the wrong way round
    return _real["gemm_postnorm_backward_regrouped"](G, W, A, B, norm, gamma, beta, eps, not trans_w)


def _regrouped_consumer_skipped(G, W, A, B, norm, gamma=None, beta=None, eps=1e-5, trans_w=False):
    # G used as the post-norm's output gradient, without the consumer's GEMM
    d = _real["gemm_postnorm_backward"](A, B, G, norm, gamma, beta, eps)
    d["dC"] = np.asarray(G, np.float64)
    return d


MUTANTS = {
    "gemm_transposed_B": ("gemm", _gemm_transposed),
    "gemm_dropped_k_term": ("gemm", _gemm_dropped_k),
    "rmsnorm_eps_outside_root": ("rmsnorm", lambda *a, **k: _rms(*a, **k, outside=True)),
    "rmsnorm_sum_not_mean": ("rmsnorm", lambda *a, **k: _rms(*a, **k, use_sum=True)),
    "rmsnorm_gamma_dropped": ("rmsnorm", lambda *a, **k: _rms(*a, **k, drop_gamma=True)),
    "layernorm_unbiased_var": ("layernorm", lambda *a, **k: _ln(*a, **k, unbiased=True)),
    "layernorm_not_centred": ("layernorm", lambda *a, **k: _ln(*a, **k, no_center=True)),
    "layernorm_beta_dropped": ("layernorm", lambda *a, **k: _ln(*a, **k, drop_beta=True)),
    "prenorm_wrong_axis": ("lazy_prenorm_gemm", _prenorm_cols),
    "postnorm_norm_before_gemm": ("gemm_postnorm", _postnorm_before_gemm),
    "postnorm_rms_as_layernorm": ("gemm_postnorm", _postnorm_rms_centred),
    "postnorm_pre_stage_skipped": ("gemm_postnorm", _postnorm_skip_pre),
    "prenorm_affine_after_gemm": ("prenorm_affine_gemm", _prenorm_affine_after_gemm),
    "add_postnorm_residual_dropped": ("gemm_add_postnorm", _add_postnorm_residual_dropped),
    "prenorm_backward_norm_term_dropped": ("lazy_prenorm_gemm_backward", _prenorm_bwd_no_norm_term),
    "prenorm_backward_dB_not_rebuilt": ("lazy_prenorm_gemm_backward", _prenorm_bwd_dB_unscaled),
    "postnorm_backward_mean_term_dropped": ("gemm_postnorm_backward", _postnorm_bwd_no_mean_term),
    "postnorm_backward_gamma_ignored": ("gemm_postnorm_backward", _postnorm_bwd_gamma_ignored),
    "regrouped_backward_w_flipped": ("gemm_postnorm_backward_regrouped", _regrouped_w_flipped),
    "regrouped_backward_consumer_skipped": ("gemm_postnorm_backward_regrouped", _regrouped_consumer_skipped),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, monkeypatch):
    fn_name, mutant = MUTANTS[name]
    monkeypatch.setattr(O, fn_name, mutant)
    failures = []
    for check in ALL_CHECKS:
        try:
            check(O)
        except Exception as e:  # any failure (assertion, shape error) counts
            failures.append(f"{check.__name__}: {e}")
    assert failures, f"no pin caught the planted mistake {name}"
