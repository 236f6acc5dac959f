"""Plain float64 definitions of the fused normalization + GEMM path.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``): used by the tests, the
smoke check and the bench's CPU-baseline leg, never by the product path.

Readings taken where the pages are silent or garbled:

* epsilon sits inside the square root, 1/sqrt(var + eps) and
  1/sqrt(mean(x^2) + eps) ([ATB] sections 1.1 and 1.2 lost the '+' in
  extraction; this is the only reading that stays finite at var = 0);
* LayerNorm variance is the biased one, (1/H) * sum (x - mu)^2, computed in two
  passes ([ATB] section 1.1);
* post-RMSNorm applies gamma (and beta only when one is given) ([ATB] 1.2);
* Lazy Pre-Norm is RMSNorm without affine ([FNF-ru] "Lazy Pre-Norm" limits);
  the oracle materialises the normalised A and multiplies it, which is the
  plain definition; the fused kernel reaches the same value through the
  identity (A * rstd) @ B = (A @ B) * rstd.
"""
from __future__ import annotations

from typing import Optional

import numpy as np

__all__ = ["gemm", "rmsnorm", "layernorm", "lazy_prenorm_gemm", "gemm_postnorm", "prenorm_affine_gemm",
           "gemm_add_postnorm"]


def _f64(x) -> np.ndarray:
    a = np.asarray(x, dtype=np.float64)
    if a.ndim != 2:
        raise ValueError("expected a 2-D array")
    return a


def gemm(A, B) -> np.ndarray:
    """C = A @ B in float64.

    The plain GEMM that every fused form builds on ([FNF-ru] "Why normalization
    is a performance problem": the GEMM tiles its input over both dimensions).
    A is [M, K], B is [K, N]; a library matmul serves as the step.
    """
    A = _f64(A)
    B = _f64(B)
    if A.shape[1] != B.shape[0]:
        raise ValueError(f"inner dimensions differ: {A.shape} @ {B.shape}")
    return A @ B


def rmsnorm(X, gamma=None, beta=None, eps: float = 1e-6):
    """Row RMSNorm: y = x / sqrt(mean(x^2) + eps) * gamma (+ beta).

    [ATB] section 1.2 (RMSNorm definition: one reduction, the sum of squares,
    then a divide and the gamma scale).  Returns (Y, rstd) with
    rstd[m] = 1 / sqrt((1/H) * sum_n x[m,n]^2 + eps) and H the row length.
    """
    X = _f64(X)
    H = X.shape[1]
    ms = np.sum(X * X, axis=1) / H
    rstd = 1.0 / np.sqrt(ms + eps)
    Y = X * rstd[:, None]
    if gamma is not None:
        Y = Y * np.asarray(gamma, dtype=np.float64)[None, :]
    if beta is not None:
        Y = Y + np.asarray(beta, dtype=np.float64)[None, :]
    return Y, rstd


def layernorm(X, gamma=None, beta=None, eps: float = 1e-5):
    """Row LayerNorm: y = (x - mu) / sqrt(var + eps) * gamma + beta.

    [ATB] section 1.1 (LayerNorm: mean mu = (1/H) sum x, variance
    (1/H) sum (x - mu)^2, normalise, then the gamma/beta affine).  The variance
    is computed in a second pass over (x - mu).  Returns (Y, mean, rstd).
    """
    X = _f64(X)
    H = X.shape[1]
    mean = np.sum(X, axis=1) / H
    D = X - mean[:, None]
    var = np.sum(D * D, axis=1) / H
    rstd = 1.0 / np.sqrt(var + eps)
    Y = D * rstd[:, None]
    if gamma is not None:
        Y = Y * np.asarray(gamma, dtype=np.float64)[None, :]
    if beta is not None:
        Y = Y + np.asarray(beta, dtype=np.float64)[None, :]
    return Y, mean, rstd


def lazy_prenorm_gemm(A, B, eps: float = 1e-6):
    """C = rmsnorm(A) @ B with RMSNorm without affine.

    [FNF-ru] "Lazy Pre-Norm" (the problem statement C = rmsnorm(A) @ B with
    rmsnorm(A) = A * rstd(A), rstd the inverse root-mean-square of the row);
    [FNF-es] "Lazy Pre-Norm: el truco matemático".  The oracle takes the plain
    route: it materialises A_hat = A * rstd (float64, unrounded) and multiplies
    it by B.  Returns (C, rstd).
    """
    A_hat, rstd = rmsnorm(A, None, None, eps)
    return gemm(A_hat, B), rstd


def gemm_postnorm(A, B, norm: str, gamma=None, beta=None, eps: float = 1e-5,
                  pre_rmsnorm: bool = False, pre_eps: float = 1e-6) -> dict:
    """C = norm(A @ B), optionally norm(rmsnorm(A) @ B).

    [FNF-ru] "Multi-CTA Norm Fusion" (the norm of the GEMM result, for
    LayerNorm and RMSNorm, with or without the elementwise affine, at any N);
    [FNF-es] "El problema del tiling" (epilogue fusion of the norm after the
    GEMM).  The oracle materialises C0 = A @ B (or rmsnorm(A) @ B when
    ``pre_rmsnorm``) in float64 and applies the row norm to C0.

    Returns a dict with "C", "rstd", "mean" (LayerNorm only, else None) and
    "pre_rstd" (``pre_rmsnorm`` only, else None).
    """
    if pre_rmsnorm:
        C0, pre_rstd = lazy_prenorm_gemm(A, B, pre_eps)
    else:
        C0, pre_rstd = gemm(A, B), None
    if norm == "layernorm":
        C, mean, rstd = layernorm(C0, gamma, beta, eps)
    elif norm == "rmsnorm":
        C, rstd = rmsnorm(C0, gamma, beta, eps)
        mean = None
    else:
        raise ValueError(f"unknown norm {norm!r}")
    return {"C": C, "mean": mean, "rstd": rstd, "pre_rstd": pre_rstd}


def prenorm_affine_gemm(A, B, norm: str, gamma=None, beta=None, eps: float = 1e-6):
    """C = (norm(A) * gamma + beta) @ B, the pre-norm with its elementwise affine.

    [FNF-ru] "Lazy Pre-Norm" (the pre-norm feeding a GEMM) and its limits
    section (the affine and the LayerNorm mean do not commute with the row
    scale); [ATB] 1.1 / 1.2 for the norms.  The oracle materialises the
    normalised, affine-transformed A in float64 and multiplies it by B.
    Returns (C, mean or None, rstd) of the rows of A.
    """
    if norm == "layernorm":
        Y, mean, rstd = layernorm(A, gamma, beta, eps)
    elif norm == "rmsnorm":
        Y, rstd = rmsnorm(A, gamma, beta, eps)
        mean = None
    else:
        raise ValueError(f"unknown norm {norm!r}")
    return gemm(Y, B), mean, rstd


def gemm_add_postnorm(A, B, R, norm: str, gamma=None, beta=None, eps: float = 1e-5) -> dict:
    """C = norm(A @ B + R) * gamma + beta: a residual added before the post-norm.

    [FNF-ru] "FlashNormAttention" (a residual connection followed by a
    post-RMSNorm, the residual added through the accumulator); [ATB] 1.1 / 1.2.
    The oracle materialises H = A @ B + R in float64 and normalises its rows.
    Returns a dict with "C", "H", "rstd" and "mean" (LayerNorm only).
    """
    H = gemm(A, B) + _f64(R)
    if norm == "layernorm":
        C, mean, rstd = layernorm(H, gamma, beta, eps)
    elif norm == "rmsnorm":
        C, rstd = rmsnorm(H, gamma, beta, eps)
        mean = None
    else:
        raise ValueError(f"unknown norm {norm!r}")
    return {"C": C, "H": H, "mean": mean, "rstd": rstd}
