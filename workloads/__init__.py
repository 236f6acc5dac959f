"""Seeded synthetic inputs for the fused normalization + GEMM path.

This module is data plumbing shared by the tests, the bench and the oracle
checks.  It holds the workload table (shapes, epsilons, distributions) and the
seeded generators, and none of the method's arithmetic: no norm, no matmul.

Workloads (all bf16, row-major; "N(0, s)" means standard deviation s):

* ``cfg1``  Lazy Pre-RMSNorm GEMM, no affine: A[256,512] rows N(0,1) times a
  per-row scale log-uniform in [0.1, 10]; B[512,128] N(0, 1/sqrt(512));
  eps 1e-6.
* ``cfg2_n64`` / ``cfg2_n128``  GEMM + post-LayerNorm with affine:
  A[16384,1024] N(0,1); B[1024,N] N(0,1/32); gamma 1+N(0,0.1); beta N(0,0.1);
  eps 1e-5.
* ``cfg3``  Lazy Pre-RMSNorm GEMM, LLM-shaped: A[8192,4096] N(0,1) times a
  log-uniform row scale; B[4096,4096] N(0,1/64); eps 1e-6.
* ``cfg4_n{1024,4096,8192}_{ln,rms}``  GEMM + post-norm over a cluster of CTAs
  along N: A[16384,2048] N(0,1); B[2048,N] N(0,1/45); LayerNorm with gamma and
  beta, or RMSNorm with gamma only; eps 1e-5.
* ``cfg5``  pre-RMSNorm (eps 1e-6, no affine) and post-LayerNorm (gamma, beta,
  eps 1e-5) in one kernel: A[65536,256] N(0,1) with 1% of rows (655 rows,
  drawn without replacement) scaled by 100; B[256,256] N(0,1/16).

Forms beyond the five configurations (same distributions where they apply):

* ``res_ln_n128``  residual-add post-LayerNorm: cfg2_n128 plus R[16384,128]
  N(0,1).
* ``res_rms_n1024``  residual-add post-RMSNorm (gamma only) over a cluster:
  cfg4_n1024_rms plus R[16384,1024] N(0,1).
* ``preln_affine``  pre-LayerNorm with affine feeding a GEMM:
  A[8192,4096] = (N(0,1) + o_m) * s_m with a per-row offset o_m ~ N(0,1) (a
  row mean of the order of the row's spread) and the log-uniform row scale
  s_m; gamma[4096] 1+N(0,0.1), beta[4096] N(0,0.1); B[4096,4096] N(0,1/64);
  eps 1e-5.
* ``prerms_gamma``  Lazy Pre-RMSNorm with gamma folded into B: cfg3's A and B,
  gamma[4096] 1+N(0,0.1), no beta, eps 1e-6.
* ``prenorm_bwd``  backward of the Lazy Pre-RMSNorm GEMM at cfg3's shape: cfg3's
  A and B and an upstream gradient dC[8192,4096] N(0,1).
* ``postnorm_bwd``  backward of the GEMM + post-LayerNorm at cfg4_n1024_ln's
  shape: its A, B, gamma, beta and dC[16384,1024] N(0,1).
* ``postnorm_bwd_rg``  the same backward regrouped onto the consuming layer's
  data-gradient GEMM: cfg4_n1024_ln's A, B, gamma, beta; the consumer
  Z = C @ W with W[1024,2048] N(0,1/sqrt(2048)) and the gradient reaching it,
  G = dL/dZ [16384,2048] N(0,1).
* ``postnorm_bwd_rg_n4096``  the same at cfg4_n4096_ln's shape: W[4096,2048].

Random numbers come from ``numpy.random.default_rng(seed)`` (PCG64), drawn in
float32 in the order A, row scale, outlier rows, row offset, B, gamma, beta, R
(each only where the workload has it), then rounded once to bf16 (round to
nearest even) by ``torch.Tensor.to(torch.bfloat16)``.  gamma and beta have
length N for a post-norm and K for a pre-norm with affine.  The backward's
dC is drawn last (the regrouped backward draws G, then W, instead).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace
from typing import Optional

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str                 # "prenorm" | "postnorm" | "prenorm_affine" | "prenorm_backward" |
                              # "postnorm_backward" | "postnorm_regrouped_backward" | "gemm"
    M: int
    K: int
    N: int
    b_std: float
    eps: float = 1e-5
    norm: Optional[str] = None        # "layernorm" | "rmsnorm" (postnorm, prenorm_affine)
    gamma: bool = False
    beta: bool = False
    pre_rmsnorm: bool = False         # cfg5: pre-RMSNorm scale before the post-norm
    pre_eps: float = 1e-6
    a_row_scale: bool = False         # log-uniform [0.1, 10] per-row scale on A
    a_outlier_frac: float = 0.0       # fraction of rows of A multiplied by 100
    a_row_offset: float = 0.0         # std of a per-row offset added to A before the row scale
    residual: bool = False            # residual R[M,N] N(0,1) added before the post-norm
    J: int = 0                        # regrouped backward: the consuming layer's output width
    description: str = ""

    def scaled(self, **kw) -> "Workload":
        """Same distributions at other sizes (used by the small parity cases)."""
        return replace(self, **kw)

    @property
    def flops(self) -> float:
        """2MNK per GEMM (the backward runs two: dA over N, dB over M; the
        regrouped backward also the consumer's data-gradient GEMM, 2MNJ)."""
        f = (4.0 if self.kind.endswith("_backward") else 2.0) * self.M * self.N * self.K
        if self.kind == "postnorm_regrouped_backward":
            f += 2.0 * self.M * self.N * self.J
        return f

    @property
    def affine_len(self) -> int:
        """Length of gamma/beta: K for a pre-norm with affine, else N."""
        return self.K if self.kind == "prenorm_affine" else self.N

    @property
    def algorithmic_bytes(self) -> float:
        """Bytes one fused launch must move: A + B + C in bf16 (+ R), gamma/beta
        (post-norm) or the folded weight's fp32 column sums and bias row
        (pre-norm with affine), and the fp32 row statistics."""
        if self.kind == "postnorm_regrouped_backward":
            # the fused GEMM reads G, W, C (and rstd) and writes dH and the
            # 32-row column partials (read back by the column sum); the
            # GEMMs read dH, B and A, dH and write dA, dB
            M, N, K, J = self.M, self.N, self.K, self.J
            return (2.0 * (M * J + N * J + 4 * M * N + 2 * K * N + 2 * M * K) + 4.0 * M
                    + 2 * 8.0 * N * ((M + 31) // 32))
        if self.kind == "postnorm_backward":
            # row pass reads dC, C and writes dH; column pass reads dC, C; the
            # GEMMs read dH, B and A, dH and write dA, dB
            return 2.0 * (7 * self.M * self.N + 3 * self.M * self.K + 2 * self.K * self.N) + 4.0 * self.M
        if self.kind == "prenorm_backward":
            # dgrad reads dC, B, C, A, rstd and writes dA; wgrad reads A, dC,
            # rstd and writes dB
            return 2.0 * (3 * self.M * self.N + 3 * self.M * self.K + 2 * self.K * self.N) + 8.0 * self.M
        b = 2.0 * (self.M * self.K + self.K * self.N + self.M * self.N)
        if self.residual:
            b += 2.0 * self.M * self.N
        if self.kind == "prenorm_affine":
            if self.norm == "layernorm":
                b += 4.0 * self.N
            if self.beta:
                b += 4.0 * self.N
        else:
            if self.gamma:
                b += 2.0 * self.N
            if self.beta:
                b += 2.0 * self.N
        nstats = 0
        if self.kind == "prenorm":
            nstats = 1
        elif self.kind == "prenorm_affine":
            nstats = 2 if self.norm == "layernorm" else 1
        elif self.kind == "postnorm":
            nstats = 2 if self.norm == "layernorm" else 1
            if self.pre_rmsnorm:
                nstats += 1
        return b + 4.0 * self.M * nstats


def _cfg4(n: int, norm: str) -> Workload:
    return Workload(
        name=f"cfg4_n{n}_{'ln' if norm == 'layernorm' else 'rms'}",
        kind="postnorm", M=16384, K=2048, N=n, b_std=1.0 / 45.0, eps=1e-5,
        norm=norm, gamma=True, beta=(norm == "layernorm"),
        description=f"GEMM + post-{norm} over a CTA cluster along N, "
                    f"A[16384,2048] @ B[2048,{n}]")


WORKLOADS: dict[str, Workload] = {w.name: w for w in [
    Workload("cfg1", "prenorm", M=256, K=512, N=128, b_std=1.0 / math.sqrt(512.0),
             eps=1e-6, a_row_scale=True,
             description="Lazy Pre-RMSNorm GEMM, A[256,512] @ B[512,128]"),
    Workload("cfg2_n64", "postnorm", M=16384, K=1024, N=64, b_std=1.0 / 32.0, eps=1e-5,
             norm="layernorm", gamma=True, beta=True,
             description="GEMM + post-LayerNorm(affine), A[16384,1024] @ B[1024,64]"),
    Workload("cfg2_n128", "postnorm", M=16384, K=1024, N=128, b_std=1.0 / 32.0, eps=1e-5,
             norm="layernorm", gamma=True, beta=True,
             description="GEMM + post-LayerNorm(affine), A[16384,1024] @ B[1024,128]"),
    Workload("cfg3", "prenorm", M=8192, K=4096, N=4096, b_std=1.0 / 64.0, eps=1e-6,
             a_row_scale=True,
             description="Lazy Pre-RMSNorm GEMM, A[8192,4096] @ B[4096,4096]"),
    _cfg4(1024, "layernorm"), _cfg4(1024, "rmsnorm"),
    _cfg4(4096, "layernorm"), _cfg4(4096, "rmsnorm"),
    _cfg4(8192, "layernorm"), _cfg4(8192, "rmsnorm"),
    Workload("cfg5", "postnorm", M=65536, K=256, N=256, b_std=1.0 / 16.0, eps=1e-5,
             norm="layernorm", gamma=True, beta=True, pre_rmsnorm=True, pre_eps=1e-6,
             a_outlier_frac=0.01,
             description="pre-RMSNorm + GEMM + post-LayerNorm(affine) in one kernel, "
                         "A[65536,256] @ B[256,256]"),
    Workload("res_ln_n128", "postnorm", M=16384, K=1024, N=128, b_std=1.0 / 32.0, eps=1e-5,
             norm="layernorm", gamma=True, beta=True, residual=True,
             description="GEMM + residual + post-LayerNorm(affine), A[16384,1024] @ B[1024,128] + R"),
    Workload("res_rms_n1024", "postnorm", M=16384, K=2048, N=1024, b_std=1.0 / 45.0, eps=1e-5,
             norm="rmsnorm", gamma=True, beta=False, residual=True,
             description="GEMM + residual + post-RMSNorm(gamma) over a CTA cluster, "
                         "A[16384,2048] @ B[2048,1024] + R"),
    Workload("preln_affine", "prenorm_affine", M=8192, K=4096, N=4096, b_std=1.0 / 64.0, eps=1e-5,
             norm="layernorm", gamma=True, beta=True, a_row_scale=True, a_row_offset=1.0,
             description="pre-LayerNorm(affine, folded into B) + GEMM, A[8192,4096] @ B[4096,4096]"),
    Workload("prerms_gamma", "prenorm_affine", M=8192, K=4096, N=4096, b_std=1.0 / 64.0, eps=1e-6,
             norm="rmsnorm", gamma=True, beta=False, a_row_scale=True,
             description="Lazy Pre-RMSNorm with gamma folded into B, A[8192,4096] @ B[4096,4096]"),
    Workload("prenorm_bwd", "prenorm_backward", M=8192, K=4096, N=4096, b_std=1.0 / 64.0, eps=1e-6,
             a_row_scale=True,
             description="backward (dA, dB) of the Lazy Pre-RMSNorm GEMM, A[8192,4096] @ B[4096,4096]"),
    Workload("postnorm_bwd", "postnorm_backward", M=16384, K=2048, N=1024, b_std=1.0 / 45.0, eps=1e-5,
             norm="layernorm", gamma=True, beta=True,
             description="backward (dA, dB, dgamma, dbeta) of GEMM + post-LayerNorm, A[16384,2048] @ B[2048,1024]"),
    Workload("postnorm_bwd_rg", "postnorm_regrouped_backward", M=16384, K=2048, N=1024, b_std=1.0 / 45.0,
             eps=1e-5, norm="layernorm", gamma=True, beta=True, J=2048,
             description="backward (dA, dB, dgamma, dbeta) of GEMM + post-LayerNorm, A[16384,2048] @ B[2048,1024], "
                         "regrouped onto the consumer's data-gradient GEMM G[16384,2048] @ W[1024,2048]^T"),
    Workload("postnorm_bwd_rg_n4096", "postnorm_regrouped_backward", M=16384, K=2048, N=4096, b_std=1.0 / 45.0,
             eps=1e-5, norm="layernorm", gamma=True, beta=True, J=2048,
             description="backward (dA, dB, dgamma, dbeta) of GEMM + post-LayerNorm, A[16384,2048] @ B[2048,4096], "
                         "regrouped onto the consumer's data-gradient GEMM G[16384,2048] @ W[4096,2048]^T "
                         "(row sums exchanged grid-wide)"),
]}


def outlier_rows(M: int, frac: float, rng: np.random.Generator) -> np.ndarray:
    """floor(frac*M) distinct row indices, sorted."""
    n = int(math.floor(frac * M))
    if n == 0:
        return np.zeros(0, dtype=np.int64)
    return np.sort(rng.choice(M, size=n, replace=False)).astype(np.int64)


def make_inputs(w: Workload, seed: int = 0) -> dict:
    """CPU bf16 tensors A[M,K], B[K,N] and optional gamma[N], beta[N].

    Also returns the drawn ``row_scale`` (float32, or None) and ``outliers``
    (row indices) so tests can reason about the structure of A.
    """
    rng = np.random.default_rng(seed)
    a = rng.standard_normal((w.M, w.K), dtype=np.float32)
    row_scale = None
    if w.a_row_scale:
        lo, hi = math.log(0.1), math.log(10.0)
        row_scale = np.exp(rng.uniform(lo, hi, size=w.M)).astype(np.float32)
    outl = outlier_rows(w.M, w.a_outlier_frac, rng)
    row_offset = None
    if w.a_row_offset > 0.0:
        row_offset = rng.standard_normal(w.M, dtype=np.float32) * np.float32(w.a_row_offset)
        a += row_offset[:, None]
    if row_scale is not None:
        a *= row_scale[:, None]
    if outl.size:
        a[outl] *= np.float32(100.0)
    b = rng.standard_normal((w.K, w.N), dtype=np.float32) * np.float32(w.b_std)
    gamma = beta = r = None
    n_aff = w.affine_len
    if w.gamma:
        gamma = np.float32(1.0) + np.float32(0.1) * rng.standard_normal(n_aff, dtype=np.float32)
    if w.beta:
        beta = np.float32(0.1) * rng.standard_normal(n_aff, dtype=np.float32)
    if w.residual:
        r = rng.standard_normal((w.M, w.N), dtype=np.float32)
    dc = g_up = w_up = None
    if w.kind == "postnorm_regrouped_backward":
        g_up = rng.standard_normal((w.M, w.J), dtype=np.float32)
        w_up = rng.standard_normal((w.N, w.J), dtype=np.float32) * np.float32(1.0 / math.sqrt(w.J))
    elif w.kind.endswith("_backward"):
        dc = rng.standard_normal((w.M, w.N), dtype=np.float32)

    def bf16(x):
        return None if x is None else torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16)

    return {"A": bf16(a), "B": bf16(b), "gamma": bf16(gamma), "beta": bf16(beta), "R": bf16(r), "dC": bf16(dc),
            "G": bf16(g_up), "W": bf16(w_up), "row_scale": row_scale, "outliers": outl, "row_offset": row_offset}


def make_rows_inputs(w: Workload, rows: np.ndarray, seed: int = 0) -> dict:
    """The full-size inputs restricted to ``rows`` of A (for sampled checks)."""
    d = make_inputs(w, seed)
    idx = torch.from_numpy(np.asarray(rows, dtype=np.int64))
    d["A"] = d["A"][idx].contiguous()
    if d["R"] is not None:
        d["R"] = d["R"][idx].contiguous()
    return d


def to_f64(t: Optional[torch.Tensor]) -> Optional[np.ndarray]:
    """Exact widening of a bf16/fp32 CPU tensor to a float64 numpy array."""
    if t is None:
        return None
    return t.detach().to("cpu").to(torch.float64).numpy()
