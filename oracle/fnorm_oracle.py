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
           "gemm_add_postnorm", "lazy_prenorm_gemm_backward", "gemm_postnorm_backward",
           "gemm_postnorm_backward_regrouped"]


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


def lazy_prenorm_gemm_backward(A, B, dC, eps: float = 1e-6):
    """Gradients of C = rmsnorm(A) @ B (RMSNorm without affine) w.r.t. A and B.

    [FNF-ru] "Lazy Pre-Norm" limits (the forward never materialises the
    normalised A, so its backward has to rebuild it) and [TFN] (the backward's
    norm work rides on a GEMM too).  The oracle materialises the forward and
    applies the chain rule step by step:

        A_hat  = A * r,  r = 1 / sqrt(mean_k(A^2) + eps)   (per row)
        dA_hat = dC @ B^T
        dB     = A_hat^T @ dC
        dA     = r * dA_hat - r^3 * A * (sum_k dA_hat * A) / K   (RMSNorm backward)

    Returns (dA, dB, r).
    """
    A = _f64(A)
    B = _f64(B)
    dC = _f64(dC)
    K = A.shape[1]
    A_hat, r = rmsnorm(A, None, None, eps)
    dA_hat = gemm(dC, B.T)
    dB = gemm(A_hat.T, dC)
    dot = np.sum(dA_hat * A, axis=1)
    dA = r[:, None] * dA_hat - (r ** 3 * dot / K)[:, None] * A
    return dA, dB, r


def gemm_postnorm_backward(A, B, dC, norm: str, gamma=None, beta=None, eps: float = 1e-5) -> dict:
    """Gradients of C = norm(A @ B) * gamma + beta w.r.t. A, B, gamma, beta.

    [TFN] ("fusion regrouping": the post-norm's backward is fused with a GEMM
    other than its forward's); the norm derivatives are those of [ATB] 1.1 /
    1.2's definitions.  The oracle materialises H = A @ B and its normalised
    rows h_hat, then:

        dgamma = sum_m dC * h_hat,   dbeta = sum_m dC,   dh = dC * gamma
        LayerNorm: dH = rstd * (dh - mean_n(dh) - h_hat * mean_n(dh * h_hat))
        RMSNorm:   dH = rstd * (dh - h_hat * mean_n(dh * h_hat))
        dA = dH @ B^T,   dB = A^T @ dH

    Returns a dict with "dA", "dB", "dH", "dgamma", "dbeta", "mean" (LayerNorm,
    else None) and "rstd".
    """
    A = _f64(A)
    B = _f64(B)
    dC = _f64(dC)
    H = gemm(A, B)
    N = H.shape[1]
    g = np.ones(N) if gamma is None else np.asarray(gamma, dtype=np.float64)
    if norm == "layernorm":
        h_hat, mean, rstd = layernorm(H, None, None, eps)
    elif norm == "rmsnorm":
        h_hat, rstd = rmsnorm(H, None, None, eps)
        mean = None
    else:
        raise ValueError(f"unknown norm {norm!r}")
    dgamma = np.sum(dC * h_hat, axis=0)
    dbeta = np.sum(dC, axis=0)
    dh = dC * g[None, :]
    proj = np.sum(dh * h_hat, axis=1) / N
    if norm == "layernorm":
        dH = rstd[:, None] * (dh - (np.sum(dh, axis=1) / N)[:, None] - h_hat * proj[:, None])
    else:
        dH = rstd[:, None] * (dh - h_hat * proj[:, None])
    return {"dA": gemm(dH, B.T), "dB": gemm(A.T, dH), "dH": dH, "dgamma": dgamma, "dbeta": dbeta,
            "mean": mean, "rstd": rstd}


def gemm_postnorm_backward_regrouped(G, W, A, B, norm: str, gamma=None, beta=None, eps: float = 1e-5,
                                     trans_w: bool = False) -> dict:
    """The post-norm's backward when the gradient reaching its output comes
    from the GEMM of the layer that consumes it.

    [TFN] ("fusion regrouping": in the backward a norm is fused with a
    different linear layer than in the forward, so that the backward also
    gets an epilogue fusion).  The forward is two layers,

        Y = norm(A @ B) * gamma + beta,    Z = Y @ op(W),

    with op(W) = W ([N, J]) or, with trans_w, W^T (W stored as [J, N]); G is
    dL/dZ [M, J].  The gradient at the post-norm's output is the consumer's
    data-gradient GEMM, dY = G @ op(W)^T, and from there the chain rule of
    gemm_postnorm_backward.  The oracle materialises dY in float64.

    Returns gemm_postnorm_backward's dict plus "dC" (= dY).
    """
    G = _f64(G)
    W = _f64(W)
    dY = gemm(G, W if trans_w else W.T)
    d = gemm_postnorm_backward(A, B, dY, norm, gamma, beta, eps)
    d["dC"] = dY
    return d
