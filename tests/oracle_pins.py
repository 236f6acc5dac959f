"""Checks that pin the fp64 oracle to something other than itself.

Each check takes the oracle module (so the mutation tests can swap a function
in it for a planted mistake) and raises on failure.  The pins are:

* hand-derived golden vectors in ``tests/golden`` (exact rationals);
* brute force (a pure-Python triple loop in another loop order);
* float64 library routines: ``torch.matmul``, ``torch.nn.functional.layer_norm``
  and ``torch.nn.functional.rms_norm``;
* identities and invariants the pages fix: (A * rstd) @ B == (A @ B) * rstd,
  unit row RMS, zero row mean and the variance ratio var/(var + eps), the
  split of a row reduction into partial reductions, B = I reducing the fused
  forms to the plain norms;
* closed forms for constant and zero rows.
"""
from __future__ import annotations

import os
from fractions import Fraction

import numpy as np
import torch
import torch.nn.functional as F

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# golden fixtures
# --------------------------------------------------------------------------
def load_golden(name: str) -> dict:
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rhs = line.partition("=")
            rows = [[float(Fraction(v)) for v in r.split()] for r in rhs.split(";")]
            arr = np.array(rows, dtype=np.float64)
            if arr.shape[0] == 1:
                arr = arr[0]
                if arr.size == 1:
                    arr = float(arr[0])
            out[key.strip()] = arr
    return out


def _close(a, b, rtol=1e-12, atol=1e-12, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    if a.shape != b.shape:
        raise AssertionError(f"{what}: shape {a.shape} != {b.shape}")
    if not np.allclose(a, b, rtol=rtol, atol=atol):
        err = np.max(np.abs(a - b))
        raise AssertionError(f"{what}: max abs err {err:.3e}")


def _t(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float64))


def _rng(seed=1234):
    return np.random.default_rng(seed)


# --------------------------------------------------------------------------
# gemm
# --------------------------------------------------------------------------
def check_gemm_bruteforce(o):
    rng = _rng(1)
    A = rng.integers(-5, 6, size=(5, 7)).astype(np.float64)
    B = rng.integers(-5, 6, size=(7, 3)).astype(np.float64)
    ref = [[0.0] * 3 for _ in range(5)]
    for k in range(7):                       # k outermost: another loop order
        for n in range(3):
            for m in range(5):
                ref[m][n] += A[m, k] * B[k, n]
    got = o.gemm(A, B)
    if not np.array_equal(got, np.array(ref)):
        raise AssertionError("gemm != brute-force triple loop on integers")


def check_gemm_torch(o):
    rng = _rng(2)
    A = rng.standard_normal((9, 16))
    B = rng.standard_normal((16, 11))
    _close(o.gemm(A, B), (_t(A) @ _t(B)).numpy(), 1e-13, 1e-13, "gemm vs torch fp64")


# --------------------------------------------------------------------------
# rmsnorm
# --------------------------------------------------------------------------
def check_rmsnorm_golden(o):
    g = load_golden("rmsnorm_rows.txt")
    y, r = o.rmsnorm(g["x"], None, None, g["eps"])
    _close(y, g["y_plain"], what="rmsnorm golden y")
    _close(r * r, g["rstd_sq"], what="rmsnorm golden rstd^2")
    y, _ = o.rmsnorm(g["x"], g["gamma"], None, g["eps"])
    _close(y, g["y_affine"], what="rmsnorm golden y*gamma")


def check_rmsnorm_torch(o):
    rng = _rng(3)
    X = rng.standard_normal((6, 40)) * rng.uniform(0.1, 10, size=(6, 1))
    gam = 1 + 0.1 * rng.standard_normal(40)
    y, _ = o.rmsnorm(X, gam, None, 1e-6)
    ref = F.rms_norm(_t(X), (40,), _t(gam), 1e-6).numpy()
    _close(y, ref, 1e-12, 1e-12, "rmsnorm vs torch fp64")


def check_rmsnorm_unit_rms(o):
    rng = _rng(4)
    X = rng.standard_normal((5, 33)) * 3.0
    eps = 0.25
    y, _ = o.rmsnorm(X, None, None, eps)
    ms = np.mean(X * X, axis=1)
    # without affine the output row's mean square is ms / (ms + eps): 1 as eps -> 0
    _close(np.mean(y * y, axis=1), ms / (ms + eps), what="rmsnorm unit RMS")


def check_rmsnorm_const_and_zero_rows(o):
    X = np.array([[2.0] * 8, [-3.0] * 8, [0.0] * 8])
    eps = 0.5
    beta = np.linspace(-1, 1, 8)
    y, r = o.rmsnorm(X, None, beta, eps)
    _close(r, [1 / np.sqrt(4 + eps), 1 / np.sqrt(9 + eps), 1 / np.sqrt(eps)],
           what="rmsnorm constant-row rstd")
    _close(y[2], beta, what="rmsnorm zero row gives beta")


# --------------------------------------------------------------------------
# layernorm
# --------------------------------------------------------------------------
def check_layernorm_golden(o):
    g = load_golden("layernorm_rows.txt")
    y, mu, r = o.layernorm(g["x"], None, None, g["eps"])
    _close(y, g["y_plain"], what="layernorm golden y")
    _close(mu, g["mean"], what="layernorm golden mean")
    _close(r, g["rstd"], what="layernorm golden rstd")
    y, _, _ = o.layernorm(g["x"], g["gamma"], g["beta"], g["eps"])
    _close(y, g["y_affine"], what="layernorm golden affine")


def check_layernorm_torch(o):
    rng = _rng(5)
    X = rng.standard_normal((7, 48)) + 0.5
    gam = 1 + 0.1 * rng.standard_normal(48)
    bet = 0.1 * rng.standard_normal(48)
    y, _, _ = o.layernorm(X, gam, bet, 1e-5)
    ref = F.layer_norm(_t(X), (48,), _t(gam), _t(bet), 1e-5).numpy()
    _close(y, ref, 1e-12, 1e-12, "layernorm vs torch fp64")


def check_layernorm_moments(o):
    rng = _rng(6)
    X = rng.standard_normal((4, 64)) * 2 + 3
    gam = 1 + 0.1 * rng.standard_normal(64)
    bet = 0.1 * rng.standard_normal(64)
    eps = 0.3
    y, _, _ = o.layernorm(X, gam, bet, eps)
    z = (y - bet) / gam
    v = np.var(X, axis=1)
    _close(np.mean(z, axis=1), np.zeros(4), 0, 1e-12, "layernorm zero row mean")
    _close(np.mean(z * z, axis=1), v / (v + eps), what="layernorm unit variance")


def check_layernorm_const_row(o):
    X = np.full((2, 16), 7.0)
    X[1] = -2.5
    bet = np.arange(16) / 16.0
    eps = 0.01
    y, mu, r = o.layernorm(X, np.full(16, 3.0), bet, eps)
    _close(y, np.stack([bet, bet]), what="layernorm constant row gives beta")
    _close(mu, [7.0, -2.5], what="layernorm constant-row mean")
    _close(r, [1 / np.sqrt(eps)] * 2, what="layernorm constant-row rstd")


# --------------------------------------------------------------------------
# lazy prenorm gemm
# --------------------------------------------------------------------------
def check_prenorm_golden(o):
    g = load_golden("lazy_prenorm_gemm.txt")
    C, r = o.lazy_prenorm_gemm(g["A"], g["B"], g["eps"])
    _close(C, g["C"], what="prenorm golden C")
    _close(r, g["rstd"], what="prenorm golden rstd")


def check_prenorm_identity(o):
    # (A * rstd) @ B == (A @ B) * rstd: the commuting identity of Lazy Pre-Norm
    rng = _rng(7)
    A = rng.standard_normal((12, 24)) * rng.uniform(0.1, 10, size=(12, 1))
    B = rng.standard_normal((24, 10)) / np.sqrt(24)
    C, r = o.lazy_prenorm_gemm(A, B, 1e-6)
    lazy = (_t(A) @ _t(B)).numpy() * r[:, None]
    _close(C, lazy, 1e-12, 1e-14, "prenorm commuting identity")


def check_prenorm_identity_B(o):
    # B = I reduces the fused form to the standalone RMSNorm
    rng = _rng(8)
    A = rng.standard_normal((6, 16)) * 4
    C, _ = o.lazy_prenorm_gemm(A, np.eye(16), 1e-6)
    ref = F.rms_norm(_t(A), (16,), None, 1e-6).numpy()
    _close(C, ref, 1e-12, 1e-12, "prenorm with B = I")


def check_prenorm_const_row(o):
    A = np.array([[3.0] * 8, [0.0] * 8, [-1.0] * 8])
    B = np.arange(24, dtype=np.float64).reshape(8, 3)
    eps = 0.75
    C, r = o.lazy_prenorm_gemm(A, B, eps)
    _close(r, [1 / np.sqrt(9 + eps), 1 / np.sqrt(eps), 1 / np.sqrt(1 + eps)],
           what="prenorm constant-row rstd")
    _close(C[1], np.zeros(3), what="prenorm zero row")


# --------------------------------------------------------------------------
# gemm + post-norm
# --------------------------------------------------------------------------
def check_postnorm_golden(o):
    g = load_golden("gemm_postnorm_layernorm.txt")
    d = o.gemm_postnorm(g["A"], g["B"], "layernorm", g["gamma"], g["beta"], g["eps"])
    _close(d["C"], g["C"], what="post-LN golden C")
    _close(d["mean"], g["mean"], what="post-LN golden mean")
    _close(d["rstd"], g["rstd"], what="post-LN golden rstd")
    g = load_golden("gemm_postnorm_rmsnorm.txt")
    d = o.gemm_postnorm(g["A"], g["B"], "rmsnorm", g["gamma"], None, g["eps"])
    _close(d["C"], g["C"], what="post-RMS golden C")
    _close(d["rstd"], g["rstd"], what="post-RMS golden rstd")


def check_postnorm_torch(o):
    rng = _rng(9)
    A = rng.standard_normal((10, 32))
    B = rng.standard_normal((32, 24)) / np.sqrt(32)
    gam = 1 + 0.1 * rng.standard_normal(24)
    bet = 0.1 * rng.standard_normal(24)
    C0 = _t(A) @ _t(B)
    d = o.gemm_postnorm(A, B, "layernorm", gam, bet, 1e-5)
    _close(d["C"], F.layer_norm(C0, (24,), _t(gam), _t(bet), 1e-5).numpy(),
           1e-12, 1e-12, "post-LN vs torch")
    d = o.gemm_postnorm(A, B, "rmsnorm", gam, None, 1e-5)
    _close(d["C"], F.rms_norm(C0, (24,), _t(gam), 1e-5).numpy(),
           1e-12, 1e-12, "post-RMS vs torch")


def check_postnorm_identity_B(o):
    rng = _rng(10)
    A = rng.standard_normal((5, 16)) * 2 + 1
    d = o.gemm_postnorm(A, np.eye(16), "layernorm", None, None, 1e-5)
    _close(d["C"], F.layer_norm(_t(A), (16,), None, None, 1e-5).numpy(),
           1e-12, 1e-12, "post-LN with B = I")


def check_postnorm_split_stats(o):
    # the row reduction splits into per-slice partials (count, mean, M2) that
    # combine to the whole-row statistics, for any number of slices
    rng = _rng(11)
    A = rng.standard_normal((8, 20))
    B = rng.standard_normal((20, 96))
    C0 = (_t(A) @ _t(B)).numpy()
    d = o.gemm_postnorm(A, B, "layernorm", None, None, 1e-5)
    dr = o.gemm_postnorm(A, B, "rmsnorm", None, None, 1e-5)
    for parts in (1, 2, 4, 8):
        n_tot = np.zeros(8)
        mean = np.zeros(8)
        m2 = np.zeros(8)
        ss = np.zeros(8)
        for sl in np.array_split(np.arange(96), parts):
            x = C0[:, sl]
            n_i = len(sl)
            m_i = x.mean(axis=1)
            m2_i = ((x - m_i[:, None]) ** 2).sum(axis=1)
            delta = m_i - mean
            n_new = n_tot + n_i
            mean = mean + delta * n_i / n_new
            m2 = m2 + m2_i + delta * delta * n_tot * n_i / n_new
            n_tot = n_new
            ss += (x * x).sum(axis=1)
        _close(d["mean"], mean, 1e-12, 1e-12, f"split mean ({parts})")
        _close(d["rstd"], 1 / np.sqrt(m2 / 96 + 1e-5), 1e-12, 0, f"split LN rstd ({parts})")
        _close(dr["rstd"], 1 / np.sqrt(ss / 96 + 1e-5), 1e-12, 0, f"split RMS rstd ({parts})")


def check_pre_and_post(o):
    # pre-RMSNorm then GEMM then post-LayerNorm, against torch fp64 routines
    rng = _rng(12)
    A = rng.standard_normal((9, 32))
    A[3] *= 100.0
    B = rng.standard_normal((32, 16)) / 4
    gam = 1 + 0.1 * rng.standard_normal(16)
    bet = 0.1 * rng.standard_normal(16)
    d = o.gemm_postnorm(A, B, "layernorm", gam, bet, 1e-5, pre_rmsnorm=True, pre_eps=1e-6)
    Ah = F.rms_norm(_t(A), (32,), None, 1e-6)
    ref = F.layer_norm(Ah @ _t(B), (16,), _t(gam), _t(bet), 1e-5).numpy()
    _close(d["C"], ref, 1e-11, 1e-11, "pre-RMS + post-LN vs torch")
    # LayerNorm hides a positive row scale, so check the pre-norm scale itself:
    # rmsnorm(A) / A element-wise gives rstd where A != 0
    _close(d["pre_rstd"], (Ah[:, 0] / _t(A)[:, 0]).numpy(), 1e-12, 0, "pre rstd")


# --------------------------------------------------------------------------
# pre-norm with affine feeding a GEMM; residual added before the post-norm
# --------------------------------------------------------------------------
def check_prenorm_affine_golden(o):
    g = load_golden("prenorm_affine_gemm.txt")
    C, mu, r = o.prenorm_affine_gemm(g["A"][None, :], g["B"], "layernorm", g["gamma"], g["beta"], g["eps"])
    _close(C, g["C"][None, :], what="pre-LN affine golden C")
    _close(mu, [g["mean"]], what="pre-LN affine golden mean")
    _close(r, [g["rstd"]], what="pre-LN affine golden rstd")


def check_prenorm_affine_torch(o):
    rng = _rng(13)
    A = rng.standard_normal((7, 40)) * 2 + 0.7
    B = rng.standard_normal((40, 12)) / np.sqrt(40)
    gam = 1 + 0.1 * rng.standard_normal(40)
    bet = 0.1 * rng.standard_normal(40)
    C, _, _ = o.prenorm_affine_gemm(A, B, "layernorm", gam, bet, 1e-5)
    ref = (F.layer_norm(_t(A), (40,), _t(gam), _t(bet), 1e-5) @ _t(B)).numpy()
    _close(C, ref, 1e-12, 1e-12, "pre-LN affine vs torch")
    C, _, _ = o.prenorm_affine_gemm(A, B, "rmsnorm", gam, None, 1e-6)
    ref = (F.rms_norm(_t(A), (40,), _t(gam), 1e-6) @ _t(B)).numpy()
    _close(C, ref, 1e-12, 1e-12, "pre-RMS affine vs torch")


def check_prenorm_affine_lazy_identity(o):
    # the lazy form: gamma folds into B, beta into a bias, the LayerNorm mean
    # into a rank-one correction with the column sums of the folded B
    rng = _rng(14)
    A = rng.standard_normal((9, 24)) * 3 + 1.5
    B = rng.standard_normal((24, 10))
    gam = 1 + 0.2 * rng.standard_normal(24)
    bet = 0.3 * rng.standard_normal(24)
    C, mu, r = o.prenorm_affine_gemm(A, B, "layernorm", gam, bet, 0.01)
    Bg = gam[:, None] * B
    lazy = r[:, None] * (A @ Bg - mu[:, None] * Bg.sum(axis=0)[None, :]) + (bet @ B)[None, :]
    _close(C, lazy, 1e-11, 1e-11, "lazy pre-LN identity")


def check_add_postnorm_torch(o):
    rng = _rng(15)
    A = rng.standard_normal((6, 16))
    B = rng.standard_normal((16, 20)) / 4
    R = rng.standard_normal((6, 20)) * 2
    gam = 1 + 0.1 * rng.standard_normal(20)
    bet = 0.1 * rng.standard_normal(20)
    d = o.gemm_add_postnorm(A, B, R, "layernorm", gam, bet, 1e-5)
    H = _t(A) @ _t(B) + _t(R)
    _close(d["C"], F.layer_norm(H, (20,), _t(gam), _t(bet), 1e-5).numpy(), 1e-12, 1e-12, "add post-LN vs torch")
    _close(d["H"], H.numpy(), 1e-13, 1e-13, "add post-LN H")
    d = o.gemm_add_postnorm(A, B, R, "rmsnorm", gam, None, 1e-5)
    _close(d["C"], F.rms_norm(H, (20,), _t(gam), 1e-5).numpy(), 1e-12, 1e-12, "add post-RMS vs torch")


def check_add_postnorm_cancel(o):
    # R = -A@B cancels the product: a zero row before the norm
    A = np.arange(12, dtype=np.float64).reshape(3, 4) - 5
    B = np.arange(8, dtype=np.float64).reshape(4, 2) / 3
    bet = np.array([0.25, -0.5])
    d = o.gemm_add_postnorm(A, B, -(A @ B), "layernorm", None, bet, 0.04)
    _close(d["C"], np.tile(bet, (3, 1)), what="cancelled residual gives beta")
    _close(d["rstd"], [5.0, 5.0, 5.0], what="cancelled residual rstd = 1/sqrt(eps)")


# --------------------------------------------------------------------------
# backward of the fused forms
# --------------------------------------------------------------------------
def check_prenorm_backward_autograd(o):
    rng = _rng(16)
    A = rng.standard_normal((6, 24)) * rng.uniform(0.2, 3.0, (6, 1))
    B = rng.standard_normal((24, 10)) / 5
    dC = rng.standard_normal((6, 10))
    dA, dB, r = o.lazy_prenorm_gemm_backward(A, B, dC, 1e-3)
    At = _t(A).requires_grad_(True)
    Bt = _t(B).requires_grad_(True)
    C = F.rms_norm(At, (24,), None, 1e-3) @ Bt
    C.backward(_t(dC))
    _close(dA, At.grad.numpy(), 1e-11, 1e-12, "prenorm dA vs autograd")
    _close(dB, Bt.grad.numpy(), 1e-11, 1e-12, "prenorm dB vs autograd")


def check_prenorm_backward_finite_diff(o):
    # central differences of L = sum(dC * C(A, B)) through the oracle's forward
    rng = _rng(17)
    A = rng.standard_normal((2, 5))
    B = rng.standard_normal((5, 3))
    dC = rng.standard_normal((2, 3))
    eps, h = 0.05, 1e-5
    dA, dB, _ = o.lazy_prenorm_gemm_backward(A, B, dC, eps)

    def loss(A_, B_):
        return float(np.sum(dC * o.lazy_prenorm_gemm(A_, B_, eps)[0]))

    for (i, j) in [(0, 0), (0, 4), (1, 2)]:
        E = np.zeros_like(A)
        E[i, j] = h
        fd = (loss(A + E, B) - loss(A - E, B)) / (2 * h)
        _close([dA[i, j]], [fd], 1e-6, 1e-8, f"prenorm dA[{i},{j}] vs finite differences")
    for (i, j) in [(0, 0), (4, 2)]:
        E = np.zeros_like(B)
        E[i, j] = h
        fd = (loss(A, B + E) - loss(A, B - E)) / (2 * h)
        _close([dB[i, j]], [fd], 1e-6, 1e-8, f"prenorm dB[{i},{j}] vs finite differences")


def check_prenorm_backward_scale_invariance(o):
    # rmsnorm(c * a) = rmsnorm(a) up to eps, so dA . A = eps r^3 (dA_hat . A) per row
    rng = _rng(18)
    A = rng.standard_normal((5, 16)) * 2
    B = rng.standard_normal((16, 7))
    dC = rng.standard_normal((5, 7))
    eps = 0.02
    dA, _, r = o.lazy_prenorm_gemm_backward(A, B, dC, eps)
    dA_hat = dC @ B.T
    _close(np.sum(dA * A, axis=1), eps * r ** 3 * np.sum(dA_hat * A, axis=1), 1e-10, 1e-12,
           "prenorm backward scale invariance")


def check_postnorm_backward_autograd(o):
    rng = _rng(19)
    A = rng.standard_normal((5, 12))
    B = rng.standard_normal((12, 20)) / 3
    dC = rng.standard_normal((5, 20))
    gam = 1 + 0.1 * rng.standard_normal(20)
    bet = 0.1 * rng.standard_normal(20)
    for norm in ("layernorm", "rmsnorm"):
        d = o.gemm_postnorm_backward(A, B, dC, norm, gam, bet if norm == "layernorm" else None, 1e-4)
        At, Bt = _t(A).requires_grad_(True), _t(B).requires_grad_(True)
        gt, bt = _t(gam).requires_grad_(True), _t(bet).requires_grad_(True)
        H = At @ Bt
        C = F.layer_norm(H, (20,), gt, bt, 1e-4) if norm == "layernorm" else F.rms_norm(H, (20,), gt, 1e-4)
        C.backward(_t(dC))
        _close(d["dA"], At.grad.numpy(), 1e-10, 1e-12, f"post-{norm} dA vs autograd")
        _close(d["dB"], Bt.grad.numpy(), 1e-10, 1e-12, f"post-{norm} dB vs autograd")
        _close(d["dgamma"], gt.grad.numpy(), 1e-10, 1e-12, f"post-{norm} dgamma vs autograd")
        if norm == "layernorm":
            _close(d["dbeta"], bt.grad.numpy(), 1e-12, 1e-12, "post-LN dbeta vs autograd")


def check_postnorm_backward_shift_invariance(o):
    # LayerNorm ignores a constant added to a row, so each row of dH sums to 0
    rng = _rng(20)
    A = rng.standard_normal((4, 8))
    B = rng.standard_normal((8, 16))
    dC = rng.standard_normal((4, 16))
    d = o.gemm_postnorm_backward(A, B, dC, "layernorm", 1 + rng.standard_normal(16) * 0.2, None, 1e-3)
    _close(np.sum(d["dH"], axis=1), np.zeros(4), 0, 1e-12, "post-LN dH rows sum to zero")


def check_postnorm_backward_regrouped_autograd(o):
    # two layers, Y = norm(A @ B) * gamma + beta and Z = Y @ op(W), differentiated
    # by autograd from dL/dZ = G: the regrouped backward starts from G and W
    rng = _rng(21)
    M, K, N = 6, 10, 12
    A = rng.standard_normal((M, K))
    B = rng.standard_normal((K, N)) / 3
    gam = 1 + 0.1 * rng.standard_normal(N)
    bet = 0.1 * rng.standard_normal(N)
    for J, trans_w in ((12, False), (12, True), (7, False), (5, True)):
        W = rng.standard_normal((J, N) if trans_w else (N, J)) / 3
        G = rng.standard_normal((M, J))
        for norm in ("layernorm", "rmsnorm"):
            b = bet if norm == "layernorm" else None
            d = o.gemm_postnorm_backward_regrouped(G, W, A, B, norm, gam, b, 1e-4, trans_w=trans_w)
            At, Bt = _t(A).requires_grad_(True), _t(B).requires_grad_(True)
            gt, bt = _t(gam).requires_grad_(True), _t(bet).requires_grad_(True)
            H = At @ Bt
            Y = F.layer_norm(H, (N,), gt, bt, 1e-4) if norm == "layernorm" else F.rms_norm(H, (N,), gt, 1e-4)
            Y.retain_grad()
            Z = Y @ (_t(W).T if trans_w else _t(W))
            Z.backward(_t(G))
            what = f"regrouped post-{norm}, J={J}, trans_w={trans_w}"
            _close(d["dC"], Y.grad.numpy(), 1e-12, 1e-12, f"{what}: dC vs autograd")
            _close(d["dA"], At.grad.numpy(), 1e-10, 1e-12, f"{what}: dA vs autograd")
            _close(d["dB"], Bt.grad.numpy(), 1e-10, 1e-12, f"{what}: dB vs autograd")
            _close(d["dgamma"], gt.grad.numpy(), 1e-10, 1e-12, f"{what}: dgamma vs autograd")
            if norm == "layernorm":
                _close(d["dbeta"], bt.grad.numpy(), 1e-12, 1e-12, f"{what}: dbeta vs autograd")


ALL_CHECKS = [
    check_gemm_bruteforce, check_gemm_torch,
    check_rmsnorm_golden, check_rmsnorm_torch, check_rmsnorm_unit_rms,
    check_rmsnorm_const_and_zero_rows,
    check_layernorm_golden, check_layernorm_torch, check_layernorm_moments,
    check_layernorm_const_row,
    check_prenorm_golden, check_prenorm_identity, check_prenorm_identity_B,
    check_prenorm_const_row,
    check_postnorm_golden, check_postnorm_torch, check_postnorm_identity_B,
    check_postnorm_split_stats, check_pre_and_post,
    check_prenorm_affine_golden, check_prenorm_affine_torch, check_prenorm_affine_lazy_identity,
    check_add_postnorm_torch, check_add_postnorm_cancel,
    check_prenorm_backward_autograd, check_prenorm_backward_finite_diff, check_prenorm_backward_scale_invariance,
    check_postnorm_backward_autograd, check_postnorm_backward_shift_invariance,
    check_postnorm_backward_regrouped_autograd,
]
