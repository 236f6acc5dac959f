"""Host-side checks of the C ABI (no GPU needed, no compute launched).

* libfnorm.so loads and exports every function include/fnorm.h declares;
* argument validation returns FNORM_ERR_INVALID_ARG / FNORM_ERR_UNSUPPORTED
  before touching the device (fake non-NULL pointers are never dereferenced);
* the post-norm planner's cluster choices.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build()
    import normalization_gemm_tcgen05_gb300 as fn
    return fn.lib()


def _header_functions():
    src = open(os.path.join(ROOT, "include", "fnorm.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fnorm_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = _header_functions()
    for required in ("fnorm_gemm", "fnorm_lazy_prenorm_gemm", "fnorm_gemm_postnorm", "fnorm_rmsnorm",
                     "fnorm_layernorm", "fnorm_check_status", "fnorm_last_error", "fnorm_gemm_add_postnorm",
                     "fnorm_fold_prenorm_affine", "fnorm_prenorm_gemm", "fnorm_lazy_prenorm_gemm_backward",
                     "fnorm_gemm_ex", "fnorm_rmsnorm_backward", "fnorm_gemm_postnorm_backward",
                     "fnorm_gemm_postnorm_noalloc", "fnorm_gemm_postnorm_ws", "fnorm_postnorm_workspace_size",
                     "fnorm_gemm_postnorm_backward_regrouped"):
        assert required in names


def test_library_exports_every_declared_symbol(L):
    import normalization_gemm_tcgen05_gb300 as fn
    names = _header_functions()
    for n in names:
        assert hasattr(L, n), f"{n} declared in fnorm.h but not exported"
    assert sorted(fn.EXPORTED_SYMBOLS) == names, "binding and header disagree"
    assert L.fnorm_version() == 100


FAKE = ctypes.c_void_p(0x10000)  # aligned, never dereferenced: validation fails first


@pytest.mark.parametrize("M,N,K", [(-1, 64, 64), (128, 60, 64), (128, 64, 60), (128, 0, 64), (128, 64, 0),
                                   (1 << 31, 64, 64)])
def test_gemm_rejects_bad_sizes(L, M, N, K):
    assert L.fnorm_gemm(FAKE, FAKE, FAKE, M, N, K, None) == 1
    assert L.fnorm_last_error()


def test_gemm_rejects_null_and_misaligned(L):
    assert L.fnorm_gemm(None, FAKE, FAKE, 128, 64, 64, None) == 1
    assert b"A" in L.fnorm_last_error()
    assert L.fnorm_gemm(FAKE, ctypes.c_void_p(0x10008), FAKE, 128, 64, 64, None) == 1
    assert b"aligned" in L.fnorm_last_error()


def test_prenorm_rejects_bad_eps(L):
    for eps in (0.0, -1.0, float("inf"), float("nan")):
        assert L.fnorm_lazy_prenorm_gemm(FAKE, FAKE, FAKE, 128, 64, 64, eps, None, None) == 1


def test_postnorm_argument_rules(L):
    f = L.fnorm_gemm_postnorm
    # unknown norm
    assert f(FAKE, FAKE, FAKE, 128, 64, 64, 7, None, None, 1e-5, 0, 1e-6, None, None, None, None) == 1
    # mean_out with RMSNorm
    assert f(FAKE, FAKE, FAKE, 128, 64, 64, 0, None, None, 1e-5, 0, 1e-6, FAKE, None, None, None) == 1
    # pre_rstd_out without the pre-norm
    assert f(FAKE, FAKE, FAKE, 128, 64, 64, 1, None, None, 1e-5, 0, 1e-6, None, None, FAKE, None) == 1
    # pre_rmsnorm flag out of range and a bad pre_eps
    assert f(FAKE, FAKE, FAKE, 128, 64, 64, 1, None, None, 1e-5, 2, 1e-6, None, None, None, None) == 1
    assert f(FAKE, FAKE, FAKE, 128, 64, 64, 1, None, None, 1e-5, 1, 0.0, None, None, None, None) == 1
    # misaligned gamma
    assert f(FAKE, FAKE, FAKE, 128, 64, 64, 1, ctypes.c_void_p(0x10002), None, 1e-5, 0, 1e-6, None, None, None,
             None) == 1


def test_add_postnorm_argument_rules(L):
    f = L.fnorm_gemm_add_postnorm
    ok = (FAKE, FAKE, ctypes.c_void_p(0x200000), ctypes.c_void_p(0x400000))  # A, B, R, C: R and C disjoint
    # unknown norm, mean_out with RMSNorm, bad eps
    assert f(*ok, 128, 64, 64, 7, None, None, 1e-5, None, None, None) == 1
    assert f(*ok, 128, 64, 64, 0, None, None, 1e-5, FAKE, None, None) == 1
    assert f(*ok, 128, 64, 64, 0, None, None, 0.0, None, None, None) == 1
    # R missing, misaligned, or overlapping C
    assert f(FAKE, FAKE, None, ok[3], 128, 64, 64, 0, None, None, 1e-5, None, None, None) == 1
    assert b"R" in L.fnorm_last_error()
    assert f(FAKE, FAKE, ctypes.c_void_p(0x200008), ok[3], 128, 64, 64, 0, None, None, 1e-5, None, None, None) == 1
    assert f(FAKE, FAKE, ctypes.c_void_p(0x400000 + 128 * 64), ok[3], 128, 64, 64, 0, None, None, 1e-5, None, None,
             None) == 1
    assert b"overlap" in L.fnorm_last_error()


def test_fold_argument_rules(L):
    f = L.fnorm_fold_prenorm_affine
    out = ctypes.c_void_p(0x400000)
    # sizes: K and N multiples of 8
    assert f(FAKE, 60, 64, None, None, out, None, None, None) == 1
    assert f(FAKE, 64, 12, None, None, out, None, None, None) == 1
    # bias exactly when beta
    assert f(FAKE, 64, 64, None, FAKE, out, None, None, None) == 1
    assert f(FAKE, 64, 64, None, None, out, None, FAKE, None) == 1
    # colsum / bias must be 16-byte aligned
    assert f(FAKE, 64, 64, None, None, out, ctypes.c_void_p(0x10004), None, None) == 1
    # partial overlap of B_folded with B (in place, B_folded == B, is allowed)
    assert f(FAKE, 64, 64, None, None, ctypes.c_void_p(0x10000 + 64), None, None, None) == 1
    assert b"overlap" in L.fnorm_last_error()


def test_prenorm_gemm_argument_rules(L):
    f = L.fnorm_prenorm_gemm
    # LayerNorm needs the column sums
    assert f(FAKE, FAKE, FAKE, 128, 64, 64, 1, None, None, 1e-5, None, None, None) == 1
    assert b"colsum" in L.fnorm_last_error()
    # mean_out only for LayerNorm; unknown norm; bad eps
    assert f(FAKE, FAKE, FAKE, 128, 64, 64, 0, None, None, 1e-5, FAKE, None, None) == 1
    assert f(FAKE, FAKE, FAKE, 128, 64, 64, 3, FAKE, None, 1e-5, None, None, None) == 1
    assert f(FAKE, FAKE, FAKE, 128, 64, 64, 1, FAKE, None, -1.0, None, None, None) == 1
    # misaligned colsum / bias
    assert f(FAKE, FAKE, FAKE, 128, 64, 64, 1, ctypes.c_void_p(0x10004), None, 1e-5, None, None, None) == 1
    assert f(FAKE, FAKE, FAKE, 128, 64, 64, 0, None, ctypes.c_void_p(0x10008), 1e-5, None, None, None) == 1
    # M == 0 is an empty call that touches nothing
    assert f(None, None, None, 0, 64, 64, 1, FAKE, None, 1e-5, None, None, None) == 0


def test_backward_argument_rules(L):
    f = L.fnorm_lazy_prenorm_gemm_backward
    W = ctypes.c_void_p(0x800000)  # workspace, disjoint from FAKE
    # neither gradient asked for; workspaces missing; misaligned rstd; dCs over dC
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, None, None, W, W, 128, 64, 64, None) == 1
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, W, 128, 64, 64, None) == 1
    assert b"dCs" in L.fnorm_last_error()
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, W, None, 128, 64, 64, None) == 1
    assert f(FAKE, FAKE, FAKE, FAKE, ctypes.c_void_p(0x10002), None, FAKE, W, W, 128, 64, 64, None) == 1
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, W, 128, 64, 64, None) == 1
    assert b"overlap" in L.fnorm_last_error()
    # dB reads A^T: M must be a multiple of 8; bad sizes
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, W, W, 100, 64, 64, None) == 1
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, W, W, 128, 60, 64, None) == 1
    h = L.fnorm_gemm_postnorm_backward
    # no gradient asked; unknown norm; dH workspace missing; dB with M % 8 != 0
    assert h(FAKE, FAKE, FAKE, FAKE, 1, None, None, FAKE, None, None, None, None, None, W, 128, 64, 64, None) == 1
    assert h(FAKE, FAKE, FAKE, FAKE, 3, None, None, FAKE, FAKE, None, None, None, W, W, 128, 64, 64, None) == 1
    assert h(FAKE, FAKE, FAKE, FAKE, 1, None, None, FAKE, FAKE, None, None, None, None, W, 128, 64, 64, None) == 1
    assert b"dH" in L.fnorm_last_error()
    assert h(FAKE, FAKE, FAKE, FAKE, 1, None, None, FAKE, None, FAKE, None, None, W, W, 100, 64, 64, None) == 1
    g = L.fnorm_gemm_ex
    assert g(FAKE, FAKE, FAKE, 100, 64, 64, 1, 0, None) == 1      # A^T needs M % 8 == 0
    assert g(FAKE, FAKE, FAKE, 128, 64, 64, 2, 0, None) == 1
    assert g(FAKE, FAKE, FAKE, 128, 64, 64, 0, -1, None) == 1
    assert L.fnorm_rmsnorm_backward(FAKE, FAKE, FAKE, FAKE, 16, 32768, None) == 1
    assert L.fnorm_rmsnorm_backward(FAKE, FAKE, None, FAKE, 16, 64, None) == 1


def test_regrouped_backward_rejects_bad_arguments(L):
    h = L.fnorm_gemm_postnorm_backward_regrouped
    W = FAKE

    def call(G=FAKE, J=64, trans_w=0, norm=1, dA=FAKE, dB=FAKE, dgamma=None, dbeta=None, dH=FAKE, part=None,
             ws=None, ws_bytes=0, M=128, N=256, K=64):
        return h(G, W, J, trans_w, FAKE, FAKE, FAKE, norm, None, None, FAKE, dA, dB, dgamma, dbeta, dH, part, ws,
                 ws_bytes, M, N, K, None)

    assert call(J=60) == 1 and b"J" in L.fnorm_last_error()
    assert call(trans_w=2) == 1
    assert call(norm=3) == 1
    assert call(N=60) == 1
    # rows wider than a cluster of 4 x 256 columns exchange grid-wide: without a
    # workspace they are refused, with too small a one it is an argument error,
    # both before any device work
    assert call(N=1032) == 2 and b"workspace" in L.fnorm_last_error()
    assert call(N=4096, ws=FAKE, ws_bytes=1024) == 1 and b"workspace" in L.fnorm_last_error()
    assert call(M=100) == 1 and b"multiple of 8" in L.fnorm_last_error()    # dB reads dH transposed
    assert call(dH=None) == 1 and b"dH" in L.fnorm_last_error()
    assert call(dgamma=FAKE) == 1 and b"part" in L.fnorm_last_error()
    assert call(G=ctypes.c_void_p(0x10002)) == 1 and b"G" in L.fnorm_last_error()
    assert call(dgamma=ctypes.c_void_p(0x10002), part=FAKE) == 1
    # a forced cluster size that leaves more than 256 columns per CTA
    L.fnorm_set_postnorm_cluster(2)
    try:
        assert call(N=1024) == 2
    finally:
        L.fnorm_set_postnorm_cluster(0)


def test_norm_rejects_bad_sizes(L):
    assert L.fnorm_add_rownorm(FAKE, None, FAKE, 16, 64, 0, None, None, 1e-5, None, None, None) == 1
    assert L.fnorm_add_rownorm(FAKE, FAKE, FAKE, 16, 64, 0, None, None, 1e-5, FAKE, None, None) == 1
    assert L.fnorm_add_rownorm(FAKE, FAKE, FAKE, 16, 64, 5, None, None, 1e-5, None, None, None) == 1
    assert L.fnorm_rmsnorm(FAKE, FAKE, 16, 12, None, 1e-6, None, None) == 1
    assert L.fnorm_layernorm(FAKE, FAKE, 16, 65536, None, None, 1e-5, None, None, None) == 1
    assert L.fnorm_layernorm(FAKE, FAKE, 16, 64, ctypes.c_void_p(0x10002), None, 1e-5, None, None, None) == 1


@pytest.mark.parametrize("N,cluster,cols", [(8, 1, 64), (64, 1, 64), (128, 1, 128), (200, 1, 256), (256, 1, 256),
                                            (320, 2, 256), (512, 2, 256), (1024, 4, 256), (1032, 4, 512),
                                            (2048, 4, 512), (2056, 4, 768), (3000, 4, 768), (4096, 4, 1024),
                                            (8192, 4, 2048), (16384, 4, 4096)])
def test_postnorm_plan(L, N, cluster, cols):
    # without a workspace: one CTA, a resident cluster, or the spill layout on
    # a cluster of 4 (ceil(N / 1024) slices of 256 columns per CTA)
    import normalization_gemm_tcgen05_gb300 as fn
    assert fn.postnorm_plan(N) == (cluster, cols)


@pytest.mark.parametrize("M,N", [(16384, 8192), (16384, 4096), (300, 1032), (1, 2048), (16384, 1024), (0, 4096),
                                 (65536, 256), (128 * 16384, 2048), (128 * 16384 + 1, 2048)])
def test_postnorm_workspace_size(L, M, N):
    # a 256-byte header, 16384 row-block counters, then 1 KB per (128-row
    # block, 256-column tile); nothing for rows a cluster holds (N <= 1024)
    # or an empty call
    import normalization_gemm_tcgen05_gb300 as fn
    rb, tiles = -(-M // 128), -(-N // 256)
    want = 256 + 8 * 16384 + rb * tiles * 1024 if (N > 1024 and 0 < M and rb <= 16384) else 0
    assert fn.postnorm_workspace_size(M, N) == want


def test_postnorm_workspace_size_follows_a_forced_cluster(L):
    import normalization_gemm_tcgen05_gb300 as fn
    try:
        fn.set_postnorm_cluster(4)
        assert fn.postnorm_workspace_size(1024, 4096) == 0   # the forced cluster spill needs none
    finally:
        fn.set_postnorm_cluster(0)
    assert fn.postnorm_workspace_size(1024, 4096) > 0


def test_postnorm_ws_argument_rules(L):
    f = L.fnorm_gemm_postnorm_ws
    W = ctypes.c_void_p(0x800000)
    need = 256 + 8 * 16384 + (4 * 16) * 1024   # M = 512, N = 4096
    # too small, misaligned
    assert f(FAKE, FAKE, FAKE, 512, 4096, 64, 1, None, None, 1e-5, 0, 1e-6, None, None, None, W, need - 1, None) == 1
    assert b"workspace" in L.fnorm_last_error()
    assert f(FAKE, FAKE, FAKE, 512, 4096, 64, 1, None, None, 1e-5, 0, 1e-6, None, None, None,
             ctypes.c_void_p(0x800008), need, None) == 1
    # the shared post-norm rules still apply
    assert f(FAKE, FAKE, FAKE, 512, 4096, 64, 0, None, None, 1e-5, 0, 1e-6, FAKE, None, None, W, need, None) == 1
    # M == 0: nothing to do, no workspace needed
    assert f(None, None, None, 0, 4096, 64, 1, None, None, 1e-5, 0, 1e-6, None, None, None, None, 0, None) == 0
    n = ctypes.c_size_t(0)
    assert L.fnorm_postnorm_workspace_size(512, 4096, ctypes.byref(n)) == 0 and n.value == need
    assert L.fnorm_postnorm_workspace_size(512, 4096, None) == 1
    assert L.fnorm_postnorm_workspace_size(512, 4092, ctypes.byref(n)) == 1


def test_no_call_allocates_or_synchronises():
    # No entry point may allocate device memory or synchronise the host,
    # except fnorm_check_status (which synchronises its stream by contract):
    # the library's sources name no allocation or device-wide synchronisation
    # at all, and the only blocking copies are in the status read.
    csrc = os.path.join(ROOT, "normalization_gemm_tcgen05_gb300", "csrc")
    banned = re.compile(r"\b(cudaMalloc\w*|cudaFree\w*|cudaDeviceSynchronize|cudaMallocAsync|cudaHostAlloc|"
                        r"cudaMallocHost|cuMemAlloc\w*|cudaMemset|cudaStreamSynchronize|cudaMemcpy)\s*\(")
    allowed = {("runtime.cu", "cudaStreamSynchronize"), ("runtime.cu", "cudaMemcpy")}
    for name in sorted(os.listdir(csrc)):
        if not name.endswith((".cu", ".cuh", ".h")):
            continue
        text = open(os.path.join(csrc, name)).read()
        code = re.sub(r"//[^\n]*", "", re.sub(r"/\*.*?\*/", "", text, flags=re.S))
        for m in banned.finditer(code):
            assert (name, m.group(1)) in allowed, f"{name} calls {m.group(1)}"
    # and the blocking calls that remain sit in the status read alone
    rt = open(os.path.join(csrc, "runtime.cu")).read()
    body = rt[rt.index("fnorm_status_t read_and_clear_status"):]
    body = body[:body.index("\n}\n") + 3]
    code = re.sub(r"//[^\n]*", "", rt.replace(body, ""))
    assert not re.search(r"\b(cudaStreamSynchronize|cudaMemcpy)\s*\(", code)


def test_forced_cluster(L):
    import normalization_gemm_tcgen05_gb300 as fn
    try:
        fn.set_postnorm_cluster(8)
        assert fn.postnorm_plan(1024) == (8, 128)
        with pytest.raises(fn.FnormError):             # 8 CTAs hold at most 128 columns each
            fn.postnorm_plan(2048)
        fn.set_postnorm_cluster(2)
        assert fn.postnorm_plan(1024) == (2, 512)      # spill: two 256-column slices per CTA
        fn.set_postnorm_cluster(1)
        assert fn.postnorm_plan(1024) == (1, 1024)
        assert fn.postnorm_plan(256) == (1, 256)       # resident, one CTA
        for bad in (3, 16, -1):
            with pytest.raises(fn.FnormError):
                fn.set_postnorm_cluster(bad)
    finally:
        fn.set_postnorm_cluster(0)
    assert fn.postnorm_plan(1024) == (4, 256)


def test_pair_mma_setter(L):
    import normalization_gemm_tcgen05_gb300 as fn
    try:
        for mode in (-1, 0, 1):
            fn.set_pair_mma(mode)
        for bad in (2, -2, 16):
            with pytest.raises(fn.FnormError):
                fn.set_pair_mma(bad)
    finally:
        fn.set_pair_mma(-1)


def test_wait_limit_setter(L):
    assert L.fnorm_set_wait_limit_ns(0) == 0
    assert L.fnorm_set_wait_limit_ns(5_000_000) == 0
    assert L.fnorm_set_wait_limit_ns(0) == 0


def test_cluster_shape_self_test_rejects_bad_sizes(L):
    for bad in (0, 3, -1, 8):
        assert L.fnorm_debug_cluster_shape(bad, None) == 1


def test_product_path_has_no_fallback():
    # the binding must fail loudly when the library cannot be loaded
    import normalization_gemm_tcgen05_gb300 as fn
    src = open(fn.__file__).read()
    assert "oracle" not in src.replace("no fallback", "")
    saved = fn._lib, fn.LIB_PATH
    try:
        fn._lib = None
        fn.LIB_PATH = os.path.join(ROOT, "does-not-exist.so")
        with pytest.raises(fn.FnormError):
            fn.lib()
    finally:
        fn._lib, fn.LIB_PATH = saved
