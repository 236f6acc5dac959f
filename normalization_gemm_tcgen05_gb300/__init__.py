"""Row normalization fused into a tcgen05 GEMM on GB300 (sm_103a).

Thin Python binding of ``libfnorm.so`` (C ABI: ``include/fnorm.h``).  The
functions here only marshal arguments: they check dtypes and shapes, allocate
outputs with PyTorch and pass raw device pointers and the current CUDA stream
to the library.  Every step of the computation runs in the library's CUDA
kernels; there is no fallback of any kind, and a missing or unloadable library
raises ``FnormError``.

Forms (see the header for the full contract):

* ``gemm(A, B)``                      C = A @ B
* ``gemm_ex(A, B, trans_a, trans_b)``  C = op(A) @ op(B), transposes read in place
* ``lazy_prenorm_gemm(A, B, eps)``    C = rmsnorm(A) @ B = (A @ B) * rstd(A)
* ``lazy_prenorm_gemm_backward(A, B, C, dC, rstd)``  its dA and dB
* ``gemm_postnorm(A, B, norm, ...)``  C = norm(A @ B) * gamma + beta, optionally
  norm(rmsnorm(A) @ B); rows wider than one CTA tile are split over a cluster,
  rows wider than 1024 columns over the whole grid (with a workspace this
  binding keeps per device and stream)
* ``gemm_add_postnorm(A, B, R, norm, ...)``  C = norm(A @ B + R) * gamma + beta
* ``fold_prenorm_affine(B, gamma, beta)``  B' = bf16(diag(gamma) B), colsum(B'), beta @ B
* ``prenorm_gemm(A, B', norm, colsum, bias)``  C = (norm(A) * gamma + beta) @ B,
  LayerNorm or RMSNorm, lazily on the folded weight
* ``rmsnorm(X)`` / ``layernorm(X)`` / ``add_rownorm(X, R, norm)``  standalone
  row norms (the unfused comparison)

``lib()`` returns the ctypes handle with every entry point declared, for
callers that want the raw C ABI.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

__all__ = [
    "FnormError", "lib", "LIB_PATH", "gemm", "gemm_ex", "rmsnorm_backward", "lazy_prenorm_gemm",
    "gemm_postnorm_backward", "gemm_postnorm_backward_regrouped", "gemm_postnorm_noalloc", "lazy_prenorm_gemm_backward", "gemm_postnorm",
    "postnorm_workspace_size",
    "gemm_add_postnorm",
    "fold_prenorm_affine", "prenorm_gemm", "add_rownorm", "rmsnorm",
    "layernorm", "check_status", "set_wait_limit_ns", "postnorm_plan", "set_postnorm_cluster", "set_pair_mma", "set_b_multicast",
    "debug_wait_timeout", "debug_cluster_shape", "last_error", "version", "RMSNORM", "LAYERNORM", "EXPORTED_SYMBOLS",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfnorm.so")

RMSNORM = 0
LAYERNORM = 1
_NORMS = {"rmsnorm": RMSNORM, "layernorm": LAYERNORM, RMSNORM: RMSNORM, LAYERNORM: LAYERNORM}

OK, INVALID_ARG, UNSUPPORTED, CUDA_ERROR, TIMEOUT = 0, 1, 2, 3, 4
_STATUS = {0: "FNORM_OK", 1: "FNORM_ERR_INVALID_ARG", 2: "FNORM_ERR_UNSUPPORTED", 3: "FNORM_ERR_CUDA",
           4: "FNORM_ERR_TIMEOUT"}


class FnormError(RuntimeError):
    """A libfnorm call failed; ``status`` holds the fnorm_status_t code."""

    def __init__(self, status: int, message: str):
        super().__init__(f"{_STATUS.get(status, status)}: {message}")
        self.status = status


_c_status = ctypes.c_int
_p = ctypes.c_void_p
_i64 = ctypes.c_int64
_f32 = ctypes.c_float

# name -> (restype, argtypes); the C ABI of include/fnorm.h
_SIGNATURES = {
    "fnorm_gemm": (_c_status, [_p, _p, _p, _i64, _i64, _i64, _p]),
    "fnorm_gemm_ex": (_c_status, [_p, _p, _p, _i64, _i64, _i64, ctypes.c_int, ctypes.c_int, _p]),
    "fnorm_rmsnorm_backward": (_c_status, [_p, _p, _p, _p, _i64, _i64, _p]),
    "fnorm_lazy_prenorm_gemm": (_c_status, [_p, _p, _p, _i64, _i64, _i64, _f32, _p, _p]),
    "fnorm_gemm_postnorm": (_c_status, [_p, _p, _p, _i64, _i64, _i64, ctypes.c_int, _p, _p, _f32,
                                        ctypes.c_int, _f32, _p, _p, _p, _p]),
    "fnorm_gemm_postnorm_ws": (_c_status, [_p, _p, _p, _i64, _i64, _i64, ctypes.c_int, _p, _p, _f32,
                                           ctypes.c_int, _f32, _p, _p, _p, _p, ctypes.c_size_t, _p]),
    "fnorm_postnorm_workspace_size": (_c_status, [_i64, _i64, ctypes.POINTER(ctypes.c_size_t)]),
    "fnorm_lazy_prenorm_gemm_backward": (_c_status, [_p, _p, _p, _p, _p, _p, _p, _p, _p, _i64, _i64, _i64, _p]),
    "fnorm_gemm_postnorm_noalloc": (_c_status, [_p, _p, _p, _i64, _i64, _i64, ctypes.c_int, _p, _p, _f32,
                                                ctypes.c_int, _f32, _p, _p, _p, _p]),
    "fnorm_gemm_postnorm_backward": (_c_status, [_p, _p, _p, _p, ctypes.c_int, _p, _p, _p, _p, _p, _p, _p, _p, _p,
                                                 _i64, _i64, _i64, _p]),
    "fnorm_gemm_postnorm_backward_regrouped": (_c_status, [_p, _p, _i64, ctypes.c_int, _p, _p, _p, ctypes.c_int,
                                                           _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, ctypes.c_size_t,
                                                           _i64, _i64, _i64, _p]),
    "fnorm_gemm_add_postnorm": (_c_status, [_p, _p, _p, _p, _i64, _i64, _i64, ctypes.c_int, _p, _p, _f32,
                                            _p, _p, _p]),
    "fnorm_fold_prenorm_affine": (_c_status, [_p, _i64, _i64, _p, _p, _p, _p, _p, _p]),
    "fnorm_prenorm_gemm": (_c_status, [_p, _p, _p, _i64, _i64, _i64, ctypes.c_int, _p, _p, _f32, _p, _p, _p]),
    "fnorm_rmsnorm": (_c_status, [_p, _p, _i64, _i64, _p, _f32, _p, _p]),
    "fnorm_layernorm": (_c_status, [_p, _p, _i64, _i64, _p, _p, _f32, _p, _p, _p]),
    "fnorm_add_rownorm": (_c_status, [_p, _p, _p, _i64, _i64, ctypes.c_int, _p, _p, _f32, _p, _p, _p]),
    "fnorm_check_status": (_c_status, [_p]),
    "fnorm_last_error": (ctypes.c_char_p, []),
    "fnorm_set_wait_limit_ns": (_c_status, [ctypes.c_uint64]),
    "fnorm_postnorm_plan": (_c_status, [_i64, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]),
    "fnorm_set_postnorm_cluster": (_c_status, [ctypes.c_int]),
    "fnorm_set_pair_mma": (_c_status, [ctypes.c_int]),
    "fnorm_set_b_multicast": (_c_status, [ctypes.c_int]),
    "fnorm_debug_wait_timeout": (_c_status, [ctypes.c_uint64, _p]),
    "fnorm_debug_cluster_shape": (_c_status, [ctypes.c_int, _p]),
    "fnorm_version": (ctypes.c_int, []),
}
EXPORTED_SYMBOLS = tuple(_SIGNATURES)

_lib: Optional[ctypes.CDLL] = None


def lib() -> ctypes.CDLL:
    """Load libfnorm.so (once) and declare its entry points."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise FnormError(CUDA_ERROR, f"{LIB_PATH} is not built; build it with "
                                         "`python -c 'import __graft_entry__ as g; g.build()'`")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def last_error() -> str:
    msg = lib().fnorm_last_error()
    return msg.decode() if msg else ""


def _check(status: int) -> None:
    if status != OK:
        raise FnormError(status, last_error())


def version() -> int:
    return lib().fnorm_version()


# --------------------------------------------------------------------------
# argument marshalling
# --------------------------------------------------------------------------
def _mat(t: torch.Tensor, name: str) -> torch.Tensor:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16 (got {t.dtype})")
    if t.dim() != 2:
        raise ValueError(f"{name} must be 2-D (got shape {tuple(t.shape)})")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous (row-major)")
    return t


def _vec(t: Optional[torch.Tensor], n: int, name: str, device) -> Optional[torch.Tensor]:
    if t is None:
        return None
    if t.dtype != torch.bfloat16 or t.dim() != 1 or t.numel() != n:
        raise ValueError(f"{name} must be a bfloat16 vector of length {n}")
    if not t.is_cuda or t.device != device or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor on {device}")
    return t


def _fvec(t: Optional[torch.Tensor], n: int, name: str, device) -> Optional[torch.Tensor]:
    if t is None:
        return None
    if t.dtype != torch.float32 or t.dim() != 1 or t.numel() != n:
        raise ValueError(f"{name} must be a float32 vector of length {n}")
    if not t.is_cuda or t.device != device or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor on {device}")
    return t


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _out(out: Optional[torch.Tensor], shape, device, name="out") -> torch.Tensor:
    if out is None:
        return torch.empty(shape, dtype=torch.bfloat16, device=device)
    _mat(out, name)
    if tuple(out.shape) != tuple(shape) or out.device != device:
        raise ValueError(f"{name} must have shape {tuple(shape)} on {device}")
    return out


def _stat(M: int, device) -> torch.Tensor:
    return torch.empty(M, dtype=torch.float32, device=device)


def _ab(A, B):
    _mat(A, "A")
    _mat(B, "B")
    if A.shape[1] != B.shape[0]:
        raise ValueError(f"inner dimensions differ: A {tuple(A.shape)} @ B {tuple(B.shape)}")
    if A.device != B.device:
        raise ValueError("A and B must be on the same device")
    return A.shape[0], B.shape[1], A.shape[1]


# --------------------------------------------------------------------------
# public functions
# --------------------------------------------------------------------------
def gemm(A: torch.Tensor, B: torch.Tensor, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """C = A @ B (bf16 in/out, fp32 accumulate) on the tcgen05 mainloop."""
    M, N, K = _ab(A, B)
    C = _out(out, (M, N), A.device)
    with torch.cuda.device(A.device):
        _check(lib().fnorm_gemm(_ptr(A), _ptr(B), _ptr(C), M, N, K, _stream(A.device)))
    return C


def gemm_ex(A: torch.Tensor, B: torch.Tensor, trans_a: bool = False, trans_b: bool = False,
            out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """C = op(A) @ op(B): op(A) = A.T when ``trans_a`` (A given as [K, M]),
    op(B) = B.T when ``trans_b`` (B given as [N, K]); no copy is made."""
    _mat(A, "A")
    _mat(B, "B")
    M, K = (A.shape[1], A.shape[0]) if trans_a else (A.shape[0], A.shape[1])
    Kb, N = (B.shape[1], B.shape[0]) if trans_b else (B.shape[0], B.shape[1])
    if K != Kb:
        raise ValueError(f"inner dimensions differ: op(A) is {M}x{K}, op(B) is {Kb}x{N}")
    if A.device != B.device:
        raise ValueError("A and B must be on the same device")
    C = _out(out, (M, N), A.device)
    with torch.cuda.device(A.device):
        _check(lib().fnorm_gemm_ex(_ptr(A), _ptr(B), _ptr(C), M, N, K, int(trans_a), int(trans_b),
                                   _stream(A.device)))
    return C


def rmsnorm_backward(dY: torch.Tensor, X: torch.Tensor, rstd: torch.Tensor,
                     out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Standalone RMSNorm backward (no affine): dX from dY, X and the forward rstd."""
    _mat(dY, "dY")
    _mat(X, "X")
    M, N = X.shape
    if tuple(dY.shape) != (M, N) or dY.device != X.device:
        raise ValueError(f"dY must have shape {(M, N)} on {X.device}")
    if rstd.dtype != torch.float32 or rstd.numel() != M or not rstd.is_contiguous() or rstd.device != X.device:
        raise ValueError(f"rstd must be a contiguous float32 vector of length {M} on {X.device}")
    dX = _out(out, (M, N), X.device, "out")
    with torch.cuda.device(X.device):
        _check(lib().fnorm_rmsnorm_backward(_ptr(dY), _ptr(X), _ptr(rstd), _ptr(dX), M, N, _stream(X.device)))
    return dX


def lazy_prenorm_gemm(A: torch.Tensor, B: torch.Tensor, eps: float = 1e-6, out: Optional[torch.Tensor] = None,
                      return_rstd: bool = False):
    """C = rmsnorm(A) @ B (RMSNorm without affine) computed as (A @ B) * rstd(A).

    With ``return_rstd`` also returns the fp32 rstd[M] of the rows of A.
    """
    M, N, K = _ab(A, B)
    C = _out(out, (M, N), A.device)
    rstd = _stat(M, A.device) if return_rstd else None
    with torch.cuda.device(A.device):
        _check(lib().fnorm_lazy_prenorm_gemm(_ptr(A), _ptr(B), _ptr(C), M, N, K, float(eps), _ptr(rstd),
                                             _stream(A.device)))
    return (C, rstd) if return_rstd else C


def lazy_prenorm_gemm_backward(A: torch.Tensor, B: torch.Tensor, C: torch.Tensor, dC: torch.Tensor,
                               rstd: torch.Tensor, need_dA: bool = True, need_dB: bool = True,
                               dA: Optional[torch.Tensor] = None, dB: Optional[torch.Tensor] = None,
                               work: Optional[tuple] = None):
    """Gradients (dA, dB) of C = rmsnorm(A) @ B given dC; C and rstd are the
    forward's output and row rstd (``lazy_prenorm_gemm(..., return_rstd=True)``).
    A gradient not asked for is returned as None.  ``work`` = (dCs [M, N]
    bf16, rowcoef [M] fp32) are the library's workspaces, allocated when
    absent; on return they hold rstd * dC and -rstd^2 (dC . C) / K."""
    M, N, K = _ab(A, B)
    for t, name in ((C, "C"), (dC, "dC")):
        _mat(t, name)
        if tuple(t.shape) != (M, N) or t.device != A.device:
            raise ValueError(f"{name} must have shape {(M, N)} on {A.device}")
    if rstd.dtype != torch.float32 or rstd.dim() != 1 or rstd.numel() != M or not rstd.is_contiguous() \
            or rstd.device != A.device:
        raise ValueError(f"rstd must be a contiguous float32 vector of length {M} on {A.device}")
    dA = _out(dA, (M, K), A.device, "dA") if need_dA else None
    dB = _out(dB, (K, N), A.device, "dB") if need_dB else None
    if work is None:
        work = (torch.empty((M, N), dtype=torch.bfloat16, device=A.device), _stat(M, A.device))
    dCs, coef = work
    _out(dCs, (M, N), A.device, "dCs")
    if coef.dtype != torch.float32 or coef.numel() != M or not coef.is_contiguous() or coef.device != A.device:
        raise ValueError(f"rowcoef must be a contiguous float32 vector of length {M} on {A.device}")
    with torch.cuda.device(A.device):
        _check(lib().fnorm_lazy_prenorm_gemm_backward(_ptr(A), _ptr(B), _ptr(C), _ptr(dC), _ptr(rstd), _ptr(dA),
                                                      _ptr(dB), _ptr(dCs), _ptr(coef), M, N, K, _stream(A.device)))
    return dA, dB


def postnorm_workspace_size(M: int, N: int) -> int:
    """Bytes of the grid-exchange workspace an M x N post-norm uses (0: none)."""
    n = ctypes.c_size_t(0)
    _check(lib().fnorm_postnorm_workspace_size(int(M), int(N), ctypes.byref(n)))
    return int(n.value)


# Grid-exchange workspaces, one per (device, stream handle), zero-filled on
# the stream when made and grown when a larger call needs more.  Calls on one
# stream are ordered, so they share it; different streams never do.
_workspaces = {}


def _workspace(M: int, N: int, device) -> Optional[torch.Tensor]:
    need = postnorm_workspace_size(M, N)
    if need == 0:
        return None
    key = (device.index, _stream(device))
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < need:
        ws = torch.zeros(need, dtype=torch.uint8, device=device)
        _workspaces[key] = ws
    return ws


def gemm_postnorm(A: torch.Tensor, B: torch.Tensor, norm="layernorm", gamma: Optional[torch.Tensor] = None,
                  beta: Optional[torch.Tensor] = None, eps: float = 1e-5, pre_rmsnorm: bool = False,
                  pre_eps: float = 1e-6, out: Optional[torch.Tensor] = None, return_stats: bool = False,
                  workspace: bool = True):
    """C = norm(A @ B) * gamma + beta, or norm(rmsnorm(A) @ B) * gamma + beta.

    ``norm`` is "layernorm" or "rmsnorm".  With ``return_stats`` also returns a
    dict of fp32 [M] tensors: "rstd", "mean" (LayerNorm) and "pre_rstd"
    (``pre_rmsnorm``).  Rows of more than 1024 columns use the grid-wide
    statistics exchange through ``fnorm_gemm_postnorm_ws`` with a workspace
    kept per device and stream (made, zero-filled, on the first such call on
    a stream: make it before capturing that stream into a CUDA graph);
    ``workspace=False`` calls ``fnorm_gemm_postnorm`` (no workspace: the
    cluster spill layout for wide rows).
    """
    M, N, K = _ab(A, B)
    if norm not in _NORMS:
        raise ValueError("norm must be 'layernorm' or 'rmsnorm'")
    nid = _NORMS[norm]
    gamma = _vec(gamma, N, "gamma", A.device)
    beta = _vec(beta, N, "beta", A.device)
    C = _out(out, (M, N), A.device)
    stats = {}
    if return_stats:
        stats["rstd"] = _stat(M, A.device)
        stats["mean"] = _stat(M, A.device) if nid == LAYERNORM else None
        stats["pre_rstd"] = _stat(M, A.device) if pre_rmsnorm else None
    with torch.cuda.device(A.device):
        ws = _workspace(M, N, A.device) if workspace else None
        if ws is None:
            _check(lib().fnorm_gemm_postnorm(
                _ptr(A), _ptr(B), _ptr(C), M, N, K, nid, _ptr(gamma), _ptr(beta), float(eps),
                1 if pre_rmsnorm else 0, float(pre_eps), _ptr(stats.get("mean")), _ptr(stats.get("rstd")),
                _ptr(stats.get("pre_rstd")), _stream(A.device)))
        else:
            _check(lib().fnorm_gemm_postnorm_ws(
                _ptr(A), _ptr(B), _ptr(C), M, N, K, nid, _ptr(gamma), _ptr(beta), float(eps),
                1 if pre_rmsnorm else 0, float(pre_eps), _ptr(stats.get("mean")), _ptr(stats.get("rstd")),
                _ptr(stats.get("pre_rstd")), ws.data_ptr(), ws.numel(), _stream(A.device)))
    return (C, stats) if return_stats else C


def gemm_postnorm_noalloc(A: torch.Tensor, B: torch.Tensor, out: torch.Tensor, norm="layernorm",
                          gamma: Optional[torch.Tensor] = None, beta: Optional[torch.Tensor] = None, eps: float = 1e-5,
                          pre_rmsnorm: bool = False, pre_eps: float = 1e-6, mean_out: Optional[torch.Tensor] = None,
                          rstd_out: Optional[torch.Tensor] = None, pre_rstd_out: Optional[torch.Tensor] = None):
    """``gemm_postnorm`` through the entry point that allocates nothing: every
    output (``out`` and the optional fp32 [M] statistics) is the caller's, and
    nothing is allocated here either."""
    M, N, K = _ab(A, B)
    if norm not in _NORMS:
        raise ValueError("norm must be 'layernorm' or 'rmsnorm'")
    gamma = _vec(gamma, N, "gamma", A.device)
    beta = _vec(beta, N, "beta", A.device)
    _out(out, (M, N), A.device)
    for t, name in ((mean_out, "mean_out"), (rstd_out, "rstd_out"), (pre_rstd_out, "pre_rstd_out")):
        if t is not None and (t.dtype != torch.float32 or t.numel() != M or not t.is_contiguous()
                              or t.device != A.device):
            raise ValueError(f"{name} must be a contiguous float32 vector of length {M} on {A.device}")
    with torch.cuda.device(A.device):
        _check(lib().fnorm_gemm_postnorm_noalloc(
            _ptr(A), _ptr(B), _ptr(out), M, N, K, _NORMS[norm], _ptr(gamma), _ptr(beta), float(eps),
            1 if pre_rmsnorm else 0, float(pre_eps), _ptr(mean_out), _ptr(rstd_out), _ptr(pre_rstd_out),
            _stream(A.device)))
    return out


def gemm_postnorm_backward(A: torch.Tensor, B: torch.Tensor, C: torch.Tensor, dC: torch.Tensor, rstd: torch.Tensor,
                           norm="layernorm", gamma: Optional[torch.Tensor] = None,
                           beta: Optional[torch.Tensor] = None, need=("dA", "dB", "dgamma", "dbeta")) -> dict:
    """Gradients of C = norm(A @ B) * gamma + beta given dC; C and rstd are the
    forward's output and row rstd.  Returns a dict with the gradients named in
    ``need`` (dA, dB bf16; dgamma, dbeta fp32) and "dH"."""
    M, N, K = _ab(A, B)
    for t, name in ((C, "C"), (dC, "dC")):
        _mat(t, name)
        if tuple(t.shape) != (M, N) or t.device != A.device:
            raise ValueError(f"{name} must have shape {(M, N)} on {A.device}")
    if rstd.dtype != torch.float32 or rstd.numel() != M or not rstd.is_contiguous() or rstd.device != A.device:
        raise ValueError(f"rstd must be a contiguous float32 vector of length {M} on {A.device}")
    if norm not in _NORMS:
        raise ValueError("norm must be 'layernorm' or 'rmsnorm'")
    gamma = _vec(gamma, N, "gamma", A.device)
    beta = _vec(beta, N, "beta", A.device)
    dev = A.device
    out = {"dA": torch.empty((M, K), dtype=torch.bfloat16, device=dev) if "dA" in need else None,
           "dB": torch.empty((K, N), dtype=torch.bfloat16, device=dev) if "dB" in need else None,
           "dgamma": torch.empty(N, dtype=torch.float32, device=dev) if "dgamma" in need else None,
           "dbeta": torch.empty(N, dtype=torch.float32, device=dev) if "dbeta" in need else None}
    out["dH"] = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    part = torch.empty(2 * N * ((M + 63) // 64), dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        _check(lib().fnorm_gemm_postnorm_backward(
            _ptr(A), _ptr(B), _ptr(C), _ptr(dC), _NORMS[norm], _ptr(gamma), _ptr(beta), _ptr(rstd),
            _ptr(out["dA"]), _ptr(out["dB"]), _ptr(out["dgamma"]), _ptr(out["dbeta"]), _ptr(out["dH"]), _ptr(part),
            M, N, K, _stream(dev)))
    return out


def gemm_postnorm_backward_regrouped(G: torch.Tensor, W: torch.Tensor, A: torch.Tensor, B: torch.Tensor,
                                     C: torch.Tensor, rstd: torch.Tensor, norm="layernorm",
                                     gamma: Optional[torch.Tensor] = None, beta: Optional[torch.Tensor] = None,
                                     trans_w: bool = False, need=("dA", "dB", "dgamma", "dbeta"),
                                     workspace: bool = True) -> dict:
    """gemm_postnorm_backward with the output gradient produced by the
    consuming layer's GEMM inside the same fused kernel: dC = G @ W^T for a
    consumer Z = C @ W (W [N, J]), or dC = G @ W with ``trans_w`` for a
    consumer Z = C @ W^T (W [J, N]).  G is dL/dZ [M, J].  Rows of more than
    1024 columns exchange their row sums through the stream's grid-exchange
    workspace (the one gemm_postnorm uses); ``workspace=False`` passes none
    (such rows are then refused).  Returns a dict with the gradients named in
    ``need`` and "dH"."""
    M, N, K = _ab(A, B)
    _mat(G, "G")
    _mat(W, "W")
    if G.shape[0] != M or G.device != A.device:
        raise ValueError(f"G must have {M} rows on {A.device}")
    J = G.shape[1]
    if tuple(W.shape) != ((J, N) if trans_w else (N, J)) or W.device != A.device:
        raise ValueError(f"W must have shape {(J, N) if trans_w else (N, J)} on {A.device}")
    _mat(C, "C")
    if tuple(C.shape) != (M, N) or C.device != A.device:
        raise ValueError(f"C must have shape {(M, N)} on {A.device}")
    if rstd.dtype != torch.float32 or rstd.numel() != M or not rstd.is_contiguous() or rstd.device != A.device:
        raise ValueError(f"rstd must be a contiguous float32 vector of length {M} on {A.device}")
    if norm not in _NORMS:
        raise ValueError("norm must be 'layernorm' or 'rmsnorm'")
    gamma = _vec(gamma, N, "gamma", A.device)
    beta = _vec(beta, N, "beta", A.device)
    dev = A.device
    out = {"dA": torch.empty((M, K), dtype=torch.bfloat16, device=dev) if "dA" in need else None,
           "dB": torch.empty((K, N), dtype=torch.bfloat16, device=dev) if "dB" in need else None,
           "dgamma": torch.empty(N, dtype=torch.float32, device=dev) if "dgamma" in need else None,
           "dbeta": torch.empty(N, dtype=torch.float32, device=dev) if "dbeta" in need else None}
    out["dH"] = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    part = torch.empty(2 * N * ((M + 31) // 32), dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        ws = _workspace(M, N, dev) if workspace and N > 1024 else None
        _check(lib().fnorm_gemm_postnorm_backward_regrouped(
            _ptr(G), _ptr(W), J, 1 if trans_w else 0, _ptr(A), _ptr(B), _ptr(C), _NORMS[norm], _ptr(gamma),
            _ptr(beta), _ptr(rstd), _ptr(out["dA"]), _ptr(out["dB"]), _ptr(out["dgamma"]), _ptr(out["dbeta"]),
            _ptr(out["dH"]), _ptr(part), _ptr(ws), 0 if ws is None else ws.numel(), M, N, K, _stream(dev)))
    return out


def gemm_add_postnorm(A: torch.Tensor, B: torch.Tensor, R: torch.Tensor, norm="rmsnorm",
                      gamma: Optional[torch.Tensor] = None, beta: Optional[torch.Tensor] = None, eps: float = 1e-5,
                      out: Optional[torch.Tensor] = None, return_stats: bool = False):
    """C = norm(A @ B + R) * gamma + beta: the residual R [M, N] is added to the
    fp32 accumulator before the post-norm.  With ``return_stats`` also returns
    {"rstd", "mean" (LayerNorm)} of the rows of A @ B + R."""
    M, N, K = _ab(A, B)
    _mat(R, "R")
    if tuple(R.shape) != (M, N) or R.device != A.device:
        raise ValueError(f"R must have shape {(M, N)} on {A.device}")
    if norm not in _NORMS:
        raise ValueError("norm must be 'layernorm' or 'rmsnorm'")
    nid = _NORMS[norm]
    gamma = _vec(gamma, N, "gamma", A.device)
    beta = _vec(beta, N, "beta", A.device)
    C = _out(out, (M, N), A.device)
    stats = {}
    if return_stats:
        stats["rstd"] = _stat(M, A.device)
        stats["mean"] = _stat(M, A.device) if nid == LAYERNORM else None
    with torch.cuda.device(A.device):
        _check(lib().fnorm_gemm_add_postnorm(
            _ptr(A), _ptr(B), _ptr(R), _ptr(C), M, N, K, nid, _ptr(gamma), _ptr(beta), float(eps),
            _ptr(stats.get("mean")), _ptr(stats.get("rstd")), _stream(A.device)))
    return (C, stats) if return_stats else C


def fold_prenorm_affine(B: torch.Tensor, gamma: Optional[torch.Tensor] = None, beta: Optional[torch.Tensor] = None,
                        out: Optional[torch.Tensor] = None, colsum_out: Optional[torch.Tensor] = None,
                        bias_out: Optional[torch.Tensor] = None):
    """Fold a pre-norm's fixed affine into the weight B [K, N] it feeds.

    Returns (B_folded, colsum, bias): B_folded = bf16(diag(gamma) B) [K, N],
    colsum = column sums of B_folded (fp32 [N]) and bias = beta @ B (fp32 [N],
    None without beta).  ``out`` may be B itself (fold in place);
    ``colsum_out`` / ``bias_out`` receive the sums when given.
    """
    _mat(B, "B")
    K, N = B.shape
    gamma = _vec(gamma, K, "gamma", B.device)
    beta = _vec(beta, K, "beta", B.device)
    Bf = _out(out, (K, N), B.device, "out")
    colsum = _fvec(colsum_out, N, "colsum_out", B.device)
    if colsum is None:
        colsum = torch.empty(N, dtype=torch.float32, device=B.device)
    bias = None
    if beta is not None:
        bias = _fvec(bias_out, N, "bias_out", B.device)
        if bias is None:
            bias = torch.empty(N, dtype=torch.float32, device=B.device)
    with torch.cuda.device(B.device):
        _check(lib().fnorm_fold_prenorm_affine(_ptr(B), K, N, _ptr(gamma), _ptr(beta), _ptr(Bf), _ptr(colsum),
                                               _ptr(bias), _stream(B.device)))
    return Bf, colsum, bias


def prenorm_gemm(A: torch.Tensor, B_folded: torch.Tensor, norm="layernorm", colsum: Optional[torch.Tensor] = None,
                 bias: Optional[torch.Tensor] = None, eps: float = 1e-5, out: Optional[torch.Tensor] = None,
                 return_stats: bool = False):
    """C = (norm(A) * gamma + beta) @ B on the weight folded by
    ``fold_prenorm_affine``: rstd * (A @ B' - mean * colsum) + bias for
    LayerNorm, rstd * (A @ B') + bias for RMSNorm.  With ``return_stats`` also
    returns {"rstd", "mean" (LayerNorm)} of the rows of A."""
    M, N, K = _ab(A, B_folded)
    if norm not in _NORMS:
        raise ValueError("norm must be 'layernorm' or 'rmsnorm'")
    nid = _NORMS[norm]
    colsum = _fvec(colsum, N, "colsum", A.device)
    bias = _fvec(bias, N, "bias", A.device)
    C = _out(out, (M, N), A.device)
    stats = {}
    if return_stats:
        stats["rstd"] = _stat(M, A.device)
        stats["mean"] = _stat(M, A.device) if nid == LAYERNORM else None
    with torch.cuda.device(A.device):
        _check(lib().fnorm_prenorm_gemm(
            _ptr(A), _ptr(B_folded), _ptr(C), M, N, K, nid, _ptr(colsum), _ptr(bias), float(eps),
            _ptr(stats.get("mean")), _ptr(stats.get("rstd")), _stream(A.device)))
    return (C, stats) if return_stats else C


def rmsnorm(X: torch.Tensor, gamma: Optional[torch.Tensor] = None, eps: float = 1e-6,
            out: Optional[torch.Tensor] = None, return_rstd: bool = False):
    """Standalone row RMSNorm (the unfused comparison kernel)."""
    _mat(X, "X")
    M, N = X.shape
    gamma = _vec(gamma, N, "gamma", X.device)
    Y = _out(out, (M, N), X.device)
    rstd = _stat(M, X.device) if return_rstd else None
    with torch.cuda.device(X.device):
        _check(lib().fnorm_rmsnorm(_ptr(X), _ptr(Y), M, N, _ptr(gamma), float(eps), _ptr(rstd),
                                   _stream(X.device)))
    return (Y, rstd) if return_rstd else Y


def layernorm(X: torch.Tensor, gamma: Optional[torch.Tensor] = None, beta: Optional[torch.Tensor] = None,
              eps: float = 1e-5, out: Optional[torch.Tensor] = None, return_stats: bool = False):
    """Standalone row LayerNorm (the unfused comparison kernel)."""
    _mat(X, "X")
    M, N = X.shape
    gamma = _vec(gamma, N, "gamma", X.device)
    beta = _vec(beta, N, "beta", X.device)
    Y = _out(out, (M, N), X.device)
    mean = _stat(M, X.device) if return_stats else None
    rstd = _stat(M, X.device) if return_stats else None
    with torch.cuda.device(X.device):
        _check(lib().fnorm_layernorm(_ptr(X), _ptr(Y), M, N, _ptr(gamma), _ptr(beta), float(eps), _ptr(mean),
                                     _ptr(rstd), _stream(X.device)))
    return (Y, {"mean": mean, "rstd": rstd}) if return_stats else Y


def add_rownorm(X: torch.Tensor, R: torch.Tensor, norm="rmsnorm", gamma: Optional[torch.Tensor] = None,
                beta: Optional[torch.Tensor] = None, eps: float = 1e-5, out: Optional[torch.Tensor] = None,
                return_stats: bool = False):
    """Standalone norm(X + R) * gamma + beta (the unfused residual-add norm)."""
    _mat(X, "X")
    _mat(R, "R")
    M, N = X.shape
    if tuple(R.shape) != (M, N) or R.device != X.device:
        raise ValueError(f"R must have shape {(M, N)} on {X.device}")
    if norm not in _NORMS:
        raise ValueError("norm must be 'layernorm' or 'rmsnorm'")
    nid = _NORMS[norm]
    gamma = _vec(gamma, N, "gamma", X.device)
    beta = _vec(beta, N, "beta", X.device)
    Y = _out(out, (M, N), X.device)
    stats = {}
    if return_stats:
        stats["rstd"] = _stat(M, X.device)
        stats["mean"] = _stat(M, X.device) if nid == LAYERNORM else None
    with torch.cuda.device(X.device):
        _check(lib().fnorm_add_rownorm(_ptr(X), _ptr(R), _ptr(Y), M, N, nid, _ptr(gamma), _ptr(beta), float(eps),
                                       _ptr(stats.get("mean")), _ptr(stats.get("rstd")), _stream(X.device)))
    return (Y, stats) if return_stats else Y


def check_status(device=None) -> None:
    """Synchronise the current stream and raise FnormError if a kernel timed out."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        _check(lib().fnorm_check_status(_stream(dev)))


def set_wait_limit_ns(ns: int) -> None:
    _check(lib().fnorm_set_wait_limit_ns(int(ns)))


def postnorm_plan(N: int) -> tuple[int, int]:
    """(CTAs per cluster along N, columns per CTA) used by gemm_postnorm for width N."""
    c = ctypes.c_int(0)
    w = ctypes.c_int(0)
    _check(lib().fnorm_postnorm_plan(int(N), ctypes.byref(c), ctypes.byref(w)))
    return c.value, w.value


def set_postnorm_cluster(cluster_size: int) -> None:
    """Force the post-norm cluster size (0 = automatic)."""
    _check(lib().fnorm_set_postnorm_cluster(int(cluster_size)))


def set_pair_mma(mode: int) -> None:
    """When 256-column GEMM tiles run as two-CTA MMAs: -1 automatic, 0 never, 1 always (see fnorm_set_pair_mma)."""
    _check(lib().fnorm_set_pair_mma(int(mode)))


def set_b_multicast(mode: int) -> None:
    """When 256-column tiles share B over a 2-CTA cluster (TMA multicast): -1 automatic, 0 never,
    1 always (see fnorm_set_b_multicast)."""
    _check(lib().fnorm_set_b_multicast(int(mode)))


def debug_cluster_shape(cluster: int, device=None) -> None:
    """Launch the cluster-shape self test (see fnorm_debug_cluster_shape)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        _check(lib().fnorm_debug_cluster_shape(int(cluster), _stream(dev)))


def debug_wait_timeout(limit_ns: int = 50_000_000, device=None) -> None:
    """Launch the bounded-wait self test (see fnorm_debug_wait_timeout)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        _check(lib().fnorm_debug_wait_timeout(int(limit_ns), _stream(dev)))
