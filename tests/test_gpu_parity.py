"""GPU parity: the CUDA path (through the C ABI binding) against the fp64 oracle.

Small cases the oracle finishes in seconds, spanning several tiles, ragged
tails in M, N and K, every post-norm cluster plan, the degenerate rows of the
method (zero rows, constant rows, outlier rows) and empty inputs.
"""
import numpy as np
import pytest
import torch

import normalization_gemm_tcgen05_gb300 as fn
import oracle
from gpu_util import assert_mean_close, assert_out_close, assert_rstd_close, np64
from workloads import WORKLOADS, make_inputs, to_f64

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


def _case(base: str, seed: int, **kw):
    w = WORKLOADS[base].scaled(**kw)
    return w, make_inputs(w, seed)


def _dev(t):
    return None if t is None else t.to(DEV)


# ----------------------------------------------------------------------------
# plain GEMM (the unfused comparison's GEMM half, same mainloop)
# ----------------------------------------------------------------------------
GEMM_SHAPES = [(128, 64, 64), (256, 128, 512), (200, 136, 72), (300, 256, 1000), (129, 320, 64),
               (1, 8, 8), (513, 520, 264), (384, 1024, 2048), (1000, 4096, 128)]


@pytest.mark.parametrize("M,N,K", GEMM_SHAPES, ids=lambda v: str(v))
def test_gemm(M, N, K):
    w, d = _case("cfg3", M * 7 + N, M=M, N=N, K=K, b_std=1.0 / np.sqrt(K), a_row_scale=False)
    C = fn.gemm(_dev(d["A"]), _dev(d["B"]))
    assert_out_close(C, oracle.gemm(to_f64(d["A"]), to_f64(d["B"])), f"gemm {M}x{N}x{K}")
    fn.check_status(DEV)


def test_gemm_identity_B():
    # B = I: C must reproduce A exactly (every product is exact in fp32)
    w, d = _case("cfg3", 3, M=256, N=192, K=192, a_row_scale=False)
    eye = torch.eye(192, dtype=torch.bfloat16)
    C = fn.gemm(_dev(d["A"]), _dev(eye))
    assert torch.equal(C.cpu(), d["A"]), "A @ I != A"


# ----------------------------------------------------------------------------
# Lazy Pre-RMSNorm GEMM
# ----------------------------------------------------------------------------
# the last two give more tiles than two per CTA: the paired tile order, whose
# second tile reuses the first one's row sums (and a partial last round)
PRE_SHAPES = [(256, 128, 512), (200, 64, 72), (333, 256, 1024), (128, 520, 256), (1, 8, 8), (640, 4096, 256),
              (8192, 2048, 128), (2560, 4096, 64)]


@pytest.mark.parametrize("M,N,K", PRE_SHAPES, ids=lambda v: str(v))
def test_lazy_prenorm(M, N, K):
    w, d = _case("cfg1", M + 11 * K, M=M, N=N, K=K, b_std=1.0 / np.sqrt(K))
    C, rstd = fn.lazy_prenorm_gemm(_dev(d["A"]), _dev(d["B"]), w.eps, return_rstd=True)
    Cr, rr = oracle.lazy_prenorm_gemm(to_f64(d["A"]), to_f64(d["B"]), w.eps)
    assert_out_close(C, Cr, "prenorm C")
    assert_rstd_close(rstd, rr, "prenorm rstd")
    fn.check_status(DEV)


def test_lazy_prenorm_cfg1_exact_config():
    w = WORKLOADS["cfg1"]
    d = make_inputs(w, 0)
    C, rstd = fn.lazy_prenorm_gemm(_dev(d["A"]), _dev(d["B"]), w.eps, return_rstd=True)
    Cr, rr = oracle.lazy_prenorm_gemm(to_f64(d["A"]), to_f64(d["B"]), w.eps)
    assert_out_close(C, Cr)
    assert_rstd_close(rstd, rr)


def test_lazy_prenorm_special_rows():
    # zero row -> rstd = 1/sqrt(eps) and C row = 0; constant row c -> rstd = 1/sqrt(c^2 + eps)
    w, d = _case("cfg1", 5, M=300, N=128, K=512)
    A = d["A"].clone()
    A[7] = 0
    A[8] = 3.0
    A[299] = -0.5
    eps = 1e-2
    C, rstd = fn.lazy_prenorm_gemm(_dev(A), _dev(d["B"]), eps, return_rstd=True)
    Cr, rr = oracle.lazy_prenorm_gemm(to_f64(A), to_f64(d["B"]), eps)
    assert_out_close(C, Cr)
    assert_rstd_close(rstd, rr)
    r = np64(rstd)
    assert abs(r[7] - 1 / np.sqrt(eps)) <= 1e-4 / np.sqrt(eps)
    assert abs(r[8] - 1 / np.sqrt(9 + eps)) <= 1e-4 / np.sqrt(9 + eps)
    assert np.all(np64(C)[7] == 0)


def test_lazy_prenorm_identity_B_is_rmsnorm():
    # B = I reduces the fused form to the standalone RMSNorm (both kernels)
    w, d = _case("cfg1", 6, M=256, N=256, K=256)
    eye = torch.eye(256, dtype=torch.bfloat16)
    C = fn.lazy_prenorm_gemm(_dev(d["A"]), _dev(eye), w.eps)
    Y = fn.rmsnorm(_dev(d["A"]), None, w.eps)
    ref, _ = oracle.rmsnorm(to_f64(d["A"]), None, None, w.eps)
    assert_out_close(C, ref, "prenorm with B = I")
    assert_out_close(Y, ref, "standalone rmsnorm")


# ----------------------------------------------------------------------------
# GEMM + post-norm, one CTA per row block (N <= 256)
# ----------------------------------------------------------------------------
POST1 = [("layernorm", 64), ("layernorm", 128), ("rmsnorm", 64), ("rmsnorm", 128), ("layernorm", 192),
         ("layernorm", 256), ("rmsnorm", 256), ("layernorm", 200), ("rmsnorm", 8)]


def _post(w, d, norm, pre=False, affine=True, workspace=True):
    gamma = d["gamma"] if affine else None
    beta = d["beta"] if (affine and norm == "layernorm") else None
    C, st = fn.gemm_postnorm(_dev(d["A"]), _dev(d["B"]), norm, _dev(gamma), _dev(beta), w.eps,
                             pre_rmsnorm=pre, pre_eps=w.pre_eps, return_stats=True, workspace=workspace)
    fn.check_status(DEV)  # a kernel that gave up on a wait is reported as such, before any comparison
    ref = oracle.gemm_postnorm(to_f64(d["A"]), to_f64(d["B"]), norm, to_f64(gamma), to_f64(beta), w.eps,
                               pre_rmsnorm=pre, pre_eps=w.pre_eps)
    assert_out_close(C, ref["C"], f"post-{norm} C")
    assert_rstd_close(st["rstd"], ref["rstd"], f"post-{norm} rstd")
    if norm == "layernorm":
        assert_mean_close(st["mean"], ref["mean"], ref["rstd"], "post-LN mean")
    if pre:
        assert_rstd_close(st["pre_rstd"], ref["pre_rstd"], "pre rstd")
    fn.check_status(DEV)
    return C, st


@pytest.mark.parametrize("norm,N", POST1, ids=lambda v: str(v))
def test_postnorm_single_cta(norm, N):
    w, d = _case("cfg2_n64", N + 3, M=1000, N=N, K=1024)
    assert fn.postnorm_plan(N)[0] == 1
    _post(w, d, norm)


def test_postnorm_no_affine_and_ragged_K():
    w, d = _case("cfg2_n128", 9, M=257, N=128, K=200)
    _post(w, d, "layernorm", affine=False)
    _post(w, d, "rmsnorm", affine=False)


@pytest.mark.parametrize("norm", ["layernorm", "rmsnorm"])
def test_pre_and_post_in_one_kernel(norm):
    w, d = _case("cfg5", 12, M=1500)
    assert d["outliers"].size == 15
    _post(w, d, norm, pre=True)


# every one-CTA tile width with the norm warps present (pre-RMS + post-norm):
# 64, 128, 192 (three 32-column subtiles per half, loaded one at a time) and
# 256 columns, full and ragged
PRE_POST1 = [64, 120, 128, 136, 184, 192, 200, 256]


@pytest.mark.parametrize("N", PRE_POST1)
@pytest.mark.parametrize("norm", ["layernorm", "rmsnorm"])
def test_pre_and_post_every_tile_width(norm, N):
    w, d = _case("cfg5", 14 + N, M=1809, N=N, K=1312, b_std=1.0 / np.sqrt(1312))
    assert fn.postnorm_plan(N)[0] == 1
    _post(w, d, norm, pre=True)


# ----------------------------------------------------------------------------
# GEMM + post-norm over a cluster along N (DSMEM row-statistics exchange)
# ----------------------------------------------------------------------------
CLUSTER_N = [320, 512, 640, 1024]                  # resident slices, 2 or 4 CTAs
WIDE_N = [1032, 2048, 3000, 4096, 8192, 12288]     # grid exchange (5..48 tiles a row) or, with no
                                                   # workspace, the spill layout (4 CTAs, 2..12 slices)


@pytest.mark.parametrize("N", CLUSTER_N)
@pytest.mark.parametrize("norm", ["layernorm", "rmsnorm"])
def test_postnorm_cluster(norm, N):
    w, d = _case("cfg4_n1024_ln", N + (norm == "rmsnorm"), M=300, N=N, K=256)
    c, cols = fn.postnorm_plan(N)
    assert c > 1 and c * cols >= N and cols <= 256
    _post(w, d, norm)


@pytest.mark.parametrize("N", WIDE_N)
@pytest.mark.parametrize("norm", ["layernorm", "rmsnorm"])
def test_postnorm_grid_exchange(norm, N):
    # with a workspace: 256-column tiles resident in tensor memory over the
    # whole grid, the row statistics exchanged through the workspace
    w, d = _case("cfg4_n4096_ln", N + 7 * (norm == "rmsnorm"), M=520, N=N, K=192)
    assert fn.postnorm_workspace_size(520, N) > 0
    _post(w, d, norm)


@pytest.mark.parametrize("N", WIDE_N)
@pytest.mark.parametrize("norm", ["layernorm", "rmsnorm"])
def test_postnorm_spill(norm, N):
    # without a workspace (fnorm_gemm_postnorm): the spill layout on a cluster
    w, d = _case("cfg4_n4096_ln", N + 7 * (norm == "rmsnorm"), M=520, N=N, K=192)
    c, cols = fn.postnorm_plan(N)
    assert c == 4 and cols > 256
    _post(w, d, norm, workspace=False)


@pytest.mark.parametrize("N", [1032, 4096, 8192])
@pytest.mark.parametrize("norm", ["layernorm", "rmsnorm"])
def test_postnorm_spill_on_a_forced_cluster(norm, N):
    # a forced cluster size takes the spill layout even where a workspace is
    # offered (the binding then passes none)
    w, d = _case("cfg4_n4096_ln", N + 3 * (norm == "rmsnorm"), M=300, N=N, K=128)
    try:
        fn.set_postnorm_cluster(4)
        assert fn.postnorm_plan(N)[0] == 4
        assert fn.postnorm_workspace_size(300, N) == 0
        _post(w, d, norm)
    finally:
        fn.set_postnorm_cluster(0)


def test_grid_exchange_repeats_and_replays():
    # back-to-back calls reuse the grid-exchange counters (a new generation
    # each call), and a CUDA graph replays the same launch: every result is
    # the same as the first, bit for bit, and the status stays clean
    w, d = _case("cfg4_n4096_ln", 31, M=128 * 170 + 5, N=2048, K=128)
    A, B, g, b = _dev(d["A"]), _dev(d["B"]), _dev(d["gamma"]), _dev(d["beta"])
    assert fn.postnorm_workspace_size(w.M, 2048) > 0
    C0 = fn.gemm_postnorm(A, B, "layernorm", g, b, w.eps)
    C1 = fn.gemm_postnorm(A, B, "layernorm", g, b, w.eps)
    fn.check_status(DEV)
    assert torch.equal(C0, C1)
    ref = oracle.gemm_postnorm(to_f64(d["A"]), to_f64(d["B"]), "layernorm", to_f64(d["gamma"]),
                               to_f64(d["beta"]), w.eps)
    assert_out_close(C0, ref["C"], "grid exchange vs oracle")
    stream = torch.cuda.Stream(DEV)
    out = torch.empty_like(C0)
    with torch.cuda.stream(stream):
        fn.gemm_postnorm(A, B, "layernorm", g, b, w.eps, out=out)  # the stream's workspace, before capture
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        fn.gemm_postnorm(A, B, "layernorm", g, b, w.eps, out=out)
    for _ in range(3):
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, C0)
    fn.check_status(DEV)


def test_postnorm_cluster_with_pre():
    w, d = _case("cfg5", 13, M=400, N=1024, K=256)
    _post(w, d, "layernorm", pre=True)


@pytest.mark.parametrize("workspace", [True, False])
def test_postnorm_wide_with_pre_and_no_affine(workspace):
    w, d = _case("cfg5", 14, M=300, N=4096, K=256)
    _post(w, d, "layernorm", pre=True, workspace=workspace)
    _post(w, d, "rmsnorm", pre=True, affine=False, workspace=workspace)


@pytest.mark.parametrize("workspace", [True, False])
def test_postnorm_wide_many_row_blocks(workspace):
    # more row blocks than CTAs: the grid exchange's CTAs hold a tile of one
    # row block while computing the next; the spill layout's CTAs carry a
    # pending normalisation across row blocks
    w, d = _case("cfg4_n4096_ln", 15, M=128 * 160 + 37, N=3072, K=64)
    _post(w, d, "layernorm", workspace=workspace)


def test_grid_exchange_and_spill_agree():
    # the two wide-row layouts split the row statistics differently: equal up
    # to fp32 summation order
    w, d = _case("cfg4_n4096_ln", 41, M=384, N=4096, K=256)
    _, s1 = _post(w, d, "layernorm", workspace=True)
    _, s2 = _post(w, d, "layernorm", workspace=False)
    assert np.max(np.abs(np64(s1["rstd"]) - np64(s2["rstd"])) / np64(s2["rstd"])) < 1e-5


@pytest.mark.parametrize("M", [1, 127, 129])
@pytest.mark.parametrize("norm", ["layernorm", "rmsnorm"])
def test_grid_exchange_few_rows(norm, M):
    # one (partial) row block or two: as many CTAs as tiles of the row, the
    # rows past M zero-filled and never stored
    w, d = _case("cfg4_n4096_ln", 50 + M, M=M, N=2048, K=256)
    _post(w, d, norm)
    _post(w, d, norm, affine=False)


def test_grid_exchange_row_wider_than_the_grid():
    # a row of more 256-column tiles than SMs cannot be exchanged grid-wide
    # (a CTA would hold two tiles of the row block it waits on): the call
    # takes the spill layout even with a workspace, and is still correct
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    N = 256 * (sms + 1)
    w, d = _case("cfg4_n4096_ln", 43, M=130, N=N, K=64)
    _post(w, d, "rmsnorm", workspace=True)


def test_one_workspace_serves_calls_of_any_shape():
    # one caller workspace, zero-filled once, through calls whose row-block
    # and tile counts differ (the counters and generation word stay where
    # every call looks for them), each checked against the oracle
    shapes = [(520, 12288, "rmsnorm"), (520, 1032, "layernorm"), (130, 4096, "rmsnorm"), (1000, 2048, "layernorm"),
              (520, 12288, "rmsnorm"), (128 * 40 + 3, 1536, "layernorm")]
    need = max(fn.postnorm_workspace_size(M, N) for M, N, _ in shapes)
    ws = torch.zeros(need, dtype=torch.uint8, device=DEV)
    L = fn.lib()
    for i, (M, N, norm) in enumerate(shapes):
        w, d = _case("cfg4_n4096_ln", 200 + i, M=M, N=N, K=128)
        A, B, g = _dev(d["A"]), _dev(d["B"]), _dev(d["gamma"])
        b = _dev(d["beta"]) if norm == "layernorm" else None
        C = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
        st = L.fnorm_gemm_postnorm_ws(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, 128,
                                      fn.LAYERNORM if norm == "layernorm" else fn.RMSNORM, g.data_ptr(),
                                      None if b is None else b.data_ptr(), w.eps, 0, 1e-6, None, None, None,
                                      ws.data_ptr(), need, torch.cuda.current_stream(DEV).cuda_stream)
        assert st == fn.OK, fn.last_error()
        fn.check_status(DEV)
        ref = oracle.gemm_postnorm(to_f64(d["A"]), to_f64(d["B"]), norm, to_f64(d["gamma"]),
                                   to_f64(d["beta"]) if norm == "layernorm" else None, w.eps)
        assert_out_close(C, ref["C"], f"call {i}: {norm} {M}x{N}")


def test_postnorm_without_workspace_allocates_nothing_and_captures():
    # fnorm_gemm_postnorm on a fresh stream, through the C ABI: no device
    # memory changes hands, and its very first call captures into a CUDA
    # graph whose replays equal the eager result bit for bit
    w, d = _case("cfg4_n4096_ln", 47, M=512, N=4096, K=256)
    A, B, g, b = _dev(d["A"]), _dev(d["B"]), _dev(d["gamma"]), _dev(d["beta"])
    C0 = torch.empty(512, 4096, dtype=torch.bfloat16, device=DEV)
    C1 = torch.empty_like(C0)
    L = fn.lib()

    def call(C, stream):
        st = L.fnorm_gemm_postnorm(A.data_ptr(), B.data_ptr(), C.data_ptr(), 512, 4096, 256, fn.LAYERNORM,
                                   g.data_ptr(), b.data_ptr(), w.eps, 0, 1e-6, None, None, None,
                                   stream.cuda_stream)
        assert st == fn.OK, fn.last_error()

    call(C0, torch.cuda.current_stream(DEV))  # loads the kernel (lazy module loading takes device memory)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info(DEV)
    alloc0 = torch.cuda.memory_allocated(DEV)
    s1 = torch.cuda.Stream(DEV)
    call(C0, s1)
    s1.synchronize()
    free1, _ = torch.cuda.mem_get_info(DEV)
    assert free1 == free0 and torch.cuda.memory_allocated(DEV) == alloc0
    s2 = torch.cuda.Stream(DEV)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s2):
        call(C1, s2)
    for _ in range(2):
        C1.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(C1, C0)
    fn.check_status(DEV)
    ref = oracle.gemm_postnorm(to_f64(d["A"]), to_f64(d["B"]), "layernorm", to_f64(d["gamma"]),
                               to_f64(d["beta"]), w.eps)
    assert_out_close(C0, ref["C"], "fnorm_gemm_postnorm, no workspace")


@pytest.mark.parametrize("norm", ["layernorm", "rmsnorm"])
def test_cluster_sizes_agree(norm):
    # the statistics split into per-CTA partials: cluster sizes 1 and 2 (spill
    # layout) and 4 and 8 (resident) must give the same row statistics up to
    # fp32 summation order
    w, d = _case("cfg4_n1024_ln", 21, M=256, N=1024, K=512)
    outs = {}
    try:
        for c in (1, 2, 4, 8):
            fn.set_postnorm_cluster(c)
            assert fn.postnorm_plan(1024)[0] == c
            outs[c] = _post(w, d, norm)
    finally:
        fn.set_postnorm_cluster(0)
    r4 = np64(outs[4][1]["rstd"])
    for c in (1, 2, 8):
        rc = np64(outs[c][1]["rstd"])
        assert np.max(np.abs(rc - r4) / r4) < 1e-5, f"cluster {c} rstd differs from cluster 4"


def test_cluster_size_one_vs_two_small_N():
    w, d = _case("cfg2_n128", 22, M=384, N=256, K=512)
    try:
        fn.set_postnorm_cluster(1)
        C1, s1 = _post(w, d, "layernorm")
        fn.set_postnorm_cluster(2)
        C2, s2 = _post(w, d, "layernorm")
    finally:
        fn.set_postnorm_cluster(0)
    assert np.max(np.abs(np64(s1["rstd"]) - np64(s2["rstd"])) / np64(s1["rstd"])) < 1e-5


# ----------------------------------------------------------------------------
# standalone norms (unfused comparison kernels)
# ----------------------------------------------------------------------------
NORM_SHAPES = [(1000, 64), (1000, 128), (257, 1024), (64, 4096), (33, 8192), (7, 8), (100, 1000), (3, 32768)]


@pytest.mark.parametrize("M,N", NORM_SHAPES, ids=lambda v: str(v))
def test_standalone_norms(M, N):
    w, d = _case("cfg2_n64", M + N, M=1, K=8, N=N)
    rng = np.random.default_rng(M * 31 + N)
    X = torch.from_numpy((rng.standard_normal((M, N)) * 2 + 0.5).astype(np.float32)).to(torch.bfloat16)
    Y, st = fn.layernorm(_dev(X), _dev(d["gamma"]), _dev(d["beta"]), 1e-5, return_stats=True)
    ref, mu, r = oracle.layernorm(to_f64(X), to_f64(d["gamma"]), to_f64(d["beta"]), 1e-5)
    assert_out_close(Y, ref, "layernorm")
    assert_rstd_close(st["rstd"], r)
    assert_mean_close(st["mean"], mu, r)
    Y, rs = fn.rmsnorm(_dev(X), _dev(d["gamma"]), 1e-6, return_rstd=True)
    ref, r = oracle.rmsnorm(to_f64(X), to_f64(d["gamma"]), None, 1e-6)
    assert_out_close(Y, ref, "rmsnorm")
    assert_rstd_close(rs, r)


# ----------------------------------------------------------------------------
# edge cases and failure detection
# ----------------------------------------------------------------------------
def test_empty_M_is_a_no_op():
    A = torch.empty((0, 64), dtype=torch.bfloat16, device=DEV)
    B = torch.randn(64, 128, device=DEV).to(torch.bfloat16)
    assert fn.gemm(A, B).shape == (0, 128)
    assert fn.lazy_prenorm_gemm(A, B).shape == (0, 128)
    assert fn.gemm_postnorm(A, B, "rmsnorm").shape == (0, 128)
    assert fn.rmsnorm(A).shape == (0, 64)
    fn.check_status(DEV)


def test_invalid_arguments_launch_nothing():
    A = torch.randn(128, 60, device=DEV).to(torch.bfloat16)   # K not a multiple of 8
    B = torch.randn(60, 64, device=DEV).to(torch.bfloat16)
    with pytest.raises(fn.FnormError) as e:
        fn.gemm(A, B)
    assert e.value.status == fn.INVALID_ARG
    A = torch.randn(128, 64, device=DEV).to(torch.bfloat16)
    B = torch.randn(64, 64, device=DEV).to(torch.bfloat16)
    with pytest.raises(fn.FnormError) as e:
        fn.lazy_prenorm_gemm(A, B, eps=0.0)
    assert e.value.status == fn.INVALID_ARG
    g = torch.ones(80, dtype=torch.bfloat16, device=DEV)[1:65]  # gamma 2 bytes off a 16-byte boundary
    with pytest.raises(fn.FnormError) as e:
        fn.gemm_postnorm(A, B, "layernorm", g)
    assert e.value.status == fn.INVALID_ARG
    try:
        fn.set_postnorm_cluster(8)
        Bw = torch.randn(64, 2048, device=DEV).to(torch.bfloat16)
        with pytest.raises(fn.FnormError) as e:
            fn.gemm_postnorm(A, Bw, "layernorm")
        assert e.value.status == fn.UNSUPPORTED
    finally:
        fn.set_postnorm_cluster(0)
    fn.check_status(DEV)


def test_bounded_wait_timeout_is_reported_and_context_survives():
    fn.debug_wait_timeout(20_000_000, DEV)          # a wait nothing will satisfy, 20 ms bound
    with pytest.raises(fn.FnormError) as e:
        fn.check_status(DEV)
    assert e.value.status == fn.TIMEOUT
    fn.check_status(DEV)                            # cleared
    w, d = _case("cfg1", 30, M=128, N=64, K=64)     # the context is still usable
    C = fn.gemm(_dev(d["A"]), _dev(d["B"]))
    assert_out_close(C, oracle.gemm(to_f64(d["A"]), to_f64(d["B"])))
    fn.check_status(DEV)


def test_cluster_shape_check_is_reported_and_context_survives():
    # every clustered kernel first checks that it runs in clusters of the size
    # it expects (a launch path can drop the cluster shape: profilers replay
    # a cooperative launch without its clusters); a mismatch is recorded and
    # the kernel returns before any cluster operation
    fn.debug_cluster_shape(2, DEV)                  # the expected shape: nothing recorded
    fn.check_status(DEV)
    fn.debug_cluster_shape(1, DEV)                  # clusters of one CTA where two are expected
    with pytest.raises(fn.FnormError) as e:
        fn.check_status(DEV)
    assert e.value.status == fn.CUDA_ERROR
    assert "cluster" in str(e.value)
    fn.check_status(DEV)                            # cleared
    w, d = _case("cfg1", 31, M=384, N=256, K=64)    # a clustered GEMM (B multicast) still runs
    C = fn.gemm(_dev(d["A"]), _dev(d["B"]))
    assert_out_close(C, oracle.gemm(to_f64(d["A"]), to_f64(d["B"])))
    fn.check_status(DEV)


def test_grid_exchange_timeout_is_reported_and_context_survives():
    # The grid exchange's counter of row block 0 starts at 1 instead of 0, so
    # it can never read its target: the polling lane's bounded wait runs out,
    # every CTA stops, the call reports a timeout, the last CTA still zeroes
    # the counters, and the context and the workspace stay usable.
    M, N, K = 256, 2048, 64
    w, d = _case("cfg4_n4096_ln", 37, M=M, N=N, K=K)
    A, B = _dev(d["A"]), _dev(d["B"])
    C = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    size = fn.postnorm_workspace_size(M, N)
    ws = torch.zeros(size, dtype=torch.uint8, device=DEV)
    ws[256:264].view(torch.int64).fill_(1)  # the first row block's counter, after the 256-byte header

    def call():
        st = fn.lib().fnorm_gemm_postnorm_ws(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, 1, None, None,
                                             w.eps, 0, 1e-6, None, None, None, ws.data_ptr(), size,
                                             torch.cuda.current_stream(DEV).cuda_stream)
        assert st == 0

    fn.set_wait_limit_ns(20_000_000)
    try:
        call()
        with pytest.raises(fn.FnormError) as e:
            fn.check_status(DEV)
        assert e.value.status == fn.TIMEOUT
    finally:
        fn.set_wait_limit_ns(0)
    fn.check_status(DEV)                            # cleared
    assert torch.count_nonzero(ws[:256 + 8 * 2]) == 0  # the finish count and both row blocks' counters were
                                                    # zeroed on the way out
    call()                                          # the same workspace serves the next call
    fn.check_status(DEV)
    ref = oracle.gemm_postnorm(to_f64(d["A"]), to_f64(d["B"]), "layernorm", None, None, w.eps)
    assert_out_close(C, ref["C"], "grid exchange after a timeout")


def test_stream_and_graph_capture():
    # calls run on the caller's stream and replay from a CUDA graph
    w, d = _case("cfg2_n128", 31, M=512, N=128, K=1024)
    A, B, g, b = _dev(d["A"]), _dev(d["B"]), _dev(d["gamma"]), _dev(d["beta"])
    out = torch.empty((512, 128), dtype=torch.bfloat16, device=DEV)
    fn.gemm_postnorm(A, B, "layernorm", g, b, w.eps, out=out)   # first call loads the kernels
    torch.cuda.synchronize()
    ref = out.clone()
    out.zero_()
    s = torch.cuda.Stream(DEV)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            fn.gemm_postnorm(A, B, "layernorm", g, b, w.eps, out=out)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref)


# ----------------------------------------------------------------------------
# B resident in shared memory (N <= tile width, short K, more row blocks than SMs)
# ----------------------------------------------------------------------------
BRES_CASES = [("gemm", 64, 1024), ("gemm", 128, 512), ("gemm", 256, 256), ("prenorm", 256, 256),
              ("layernorm", 256, 256), ("rmsnorm", 128, 512), ("layernorm", 64, 1000), ("pre+layernorm", 256, 256)]


@pytest.mark.parametrize("kind,N,K", BRES_CASES, ids=lambda v: str(v))
def test_resident_B(kind, N, K):
    M = 128 * 170 + 45  # more row blocks than the 152 SMs, ragged tail
    w, d = _case("cfg5", 40 + N + K, M=M, N=N, K=K, b_std=1.0 / np.sqrt(K))
    A, B = _dev(d["A"]), _dev(d["B"])
    if kind == "gemm":
        assert_out_close(fn.gemm(A, B), oracle.gemm(to_f64(d["A"]), to_f64(d["B"])))
    elif kind == "prenorm":
        C, r = fn.lazy_prenorm_gemm(A, B, 1e-6, return_rstd=True)
        Cr, rr = oracle.lazy_prenorm_gemm(to_f64(d["A"]), to_f64(d["B"]), 1e-6)
        assert_out_close(C, Cr)
        assert_rstd_close(r, rr)
    elif kind == "pre+layernorm":
        _post(w, d, "layernorm", pre=True)
    else:
        _post(w, d, kind)
    fn.check_status(DEV)


def test_without_programmatic_dependent_launch():
    # the same kernels launched without programmatic serialisation
    import os
    import subprocess
    import sys
    here = os.path.dirname(os.path.abspath(__file__))
    code = (
        "import sys; sys.path.insert(0, %r); sys.path.insert(0, %r)\n"
        "import torch\n"
        "import normalization_gemm_tcgen05_gb300 as fn, oracle\n"
        "from workloads import WORKLOADS, make_inputs, to_f64\n"
        "from gpu_util import assert_out_close\n"
        "w = WORKLOADS['cfg4_n4096_ln'].scaled(M=300, K=128)\n"
        "d = make_inputs(w, 3)\n"
        "dev = torch.device('cuda', 0)\n"
        "C = fn.gemm_postnorm(d['A'].to(dev), d['B'].to(dev), 'layernorm', d['gamma'].to(dev), d['beta'].to(dev), w.eps)\n"
        "ref = oracle.gemm_postnorm(to_f64(d['A']), to_f64(d['B']), 'layernorm', to_f64(d['gamma']), to_f64(d['beta']), w.eps)\n"
        "assert_out_close(C, ref['C'])\n"
        "Y = fn.layernorm(C, None, None, 1e-5)\n"
        "assert_out_close(Y, oracle.layernorm(to_f64(C.cpu()), None, None, 1e-5)[0])\n"
        "fn.check_status(dev)\n"
        "print('ok')\n"
    ) % (os.path.dirname(here), here)
    env = dict(os.environ, FNORM_PDL="0")
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout + r.stderr
