"""Benchmark of the fused normalization + GEMM path on one GB300 (or N replicas).

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                [--workload main|cfg1|cfg2|cfg3|cfg4|cfg5|res|preaff|bwd|all]

Workload groups: main (the default: all five configurations in one step),
cfg1..cfg5 (one configuration each), res (residual-add post-norm), preaff
(pre-norm with its affine folded into B), bwd (backward of the Lazy
Pre-RMSNorm GEMM and of the GEMM + post-LayerNorm), all (main, res, preaff,
bwd: one line each).

Default workload (one JSON line on stdout): one step is one fused launch of
every sub-workload of the five configurations: the Lazy Pre-RMSNorm GEMMs
(256x512x128 and 8192x4096x4096), the GEMM + post-LayerNorm at N = 64 and
128, the GEMM + post-LayerNorm and post-RMSNorm of A[16384,2048] at N = 1024,
4096 and 8192, and the pre-RMSNorm + post-LayerNorm block at 65536x256x256.
Metric: fused norm-GEMM TFLOP/s (2*M*N*K per launch, summed over the step),
with the roofline of the dominant kernel (the one with the largest share of
the step), per sub-workload the fraction of the unfused norm's latency that
fusion hides and its own roofline fraction, an end-to-end number through the
public API with host buffers, and the fp64 oracle timed on the host cores.

Timing: W eager warm-up steps, then exactly K steps replayed from CUDA graphs,
bracketed by a barrier and torch.cuda.synchronize() on both sides and timed
with CUDA events on the launching stream.  For the per-sub-workload
comparison (latency_hidden) each leg (the fused call and the unfused pieces it
is compared with) is then timed as a graph of min(K, 20) launches in six
rounds, the legs of a sub-workload back to back within a round, in reverse
order every other round, and reports its median round: the GPU runs at its
power cap on the long legs, and legs compared with one another then see the
same clocks (short legs, and the alternating order, keep a drift of the clock
within a round from favouring one leg).  Inputs and outputs rotate over R
copies whose total exceeds 2x the L2 cache, so no step reads what the previous
one left in L2.  Under torchrun every rank runs the same per-GPU workload (weak
scaling, independent replicas: rows of the path never interact) and the time
is the maximum over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

if "OPENBLAS_NUM_THREADS" not in os.environ and "OMP_NUM_THREADS" not in os.environ:
    _ncores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    os.environ["OPENBLAS_NUM_THREADS"] = str(_ncores)
    os.environ["OMP_NUM_THREADS"] = str(_ncores)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from workloads import WORKLOADS, Workload, make_inputs  # noqa: E402

METRIC = "fused norm-GEMM TFLOP/s and % of roofline; % unfused-norm latency hidden (1×GB300)"

MAIN = ["cfg1", "cfg2_n64", "cfg2_n128", "cfg3", "cfg4_n1024_ln", "cfg4_n1024_rms", "cfg4_n4096_ln",
        "cfg4_n4096_rms", "cfg4_n8192_ln", "cfg4_n8192_rms", "cfg5"]
GROUPS = {
    "main": MAIN,
    "cfg1": ["cfg1"],
    "cfg2": ["cfg2_n64", "cfg2_n128"],
    "cfg3": ["cfg3"],
    "cfg4": ["cfg4_n1024_ln", "cfg4_n1024_rms", "cfg4_n4096_ln", "cfg4_n4096_rms", "cfg4_n8192_ln",
             "cfg4_n8192_rms"],
    "cfg5": ["cfg5"],
    "res": ["res_ln_n128", "res_rms_n1024"],
    "preaff": ["preln_affine", "prerms_gamma"],
    "bwd": ["prenorm_bwd", "postnorm_bwd", "postnorm_bwd_rg", "postnorm_bwd_rg_n4096"],
}
GROUP_TEXT = {
    "main": "the five configurations, one fused launch of each sub-workload per step: Lazy Pre-RMSNorm GEMM "
            "256x512x128 and 8192x4096x4096; GEMM + post-LayerNorm(affine) A[16384,1024] @ B[1024,N], N in "
            "{64,128}; GEMM + post-LayerNorm(affine) and post-RMSNorm(gamma) A[16384,2048] @ B[2048,N], N in "
            "{1024,4096,8192}; pre-RMSNorm + GEMM + post-LayerNorm(affine) A[65536,256] @ B[256,256]",
    "cfg1": "Lazy Pre-RMSNorm GEMM, A[256,512] @ B[512,128], eps 1e-6",
    "cfg2": "GEMM + post-LayerNorm(affine), A[16384,1024] @ B[1024,N], N in {64,128}, eps 1e-5",
    "cfg3": "Lazy Pre-RMSNorm GEMM, A[8192,4096] @ B[4096,4096], eps 1e-6",
    "cfg4": "GEMM + post-LayerNorm and post-RMSNorm of rows split over CTAs (a cluster at N = 1024, the "
            "grid-wide exchange beyond), A[16384,2048] @ B[2048,N], N in {1024,4096,8192}",
    "cfg5": "pre-RMSNorm + GEMM + post-LayerNorm(affine) in one kernel, A[65536,256] @ B[256,256]",
    "res": "GEMM + residual + post-norm: LayerNorm(affine) A[16384,1024] @ B[1024,128] + R, "
           "RMSNorm(gamma) A[16384,2048] @ B[2048,1024] + R",
    "preaff": "pre-norm with affine folded into B + GEMM, A[8192,4096] @ B[4096,4096]: LayerNorm(gamma, beta), "
              "RMSNorm(gamma)",
    "bwd": "backward of the Lazy Pre-RMSNorm GEMM, A[8192,4096] @ B[4096,4096], and of GEMM + post-LayerNorm, "
           "A[16384,2048] @ B[2048,1024]: from a given dC, and regrouped onto the consuming layer's data-gradient "
           "GEMM G[16384,2048] @ W^T (also at N = 4096)",
}
KERNEL_SOURCES = ["fused_gemm.cuh", "ptx.cuh", "fused_launch.cuh", "rownorm.cu"]


# --------------------------------------------------------------------------
# distributed plumbing (N > 1 under torchrun: independent replicas)
# --------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Maximum of a per-rank scalar (a time) over all ranks."""
    if world <= 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------
# helpers
# --------------------------------------------------------------------------
def kernel_source_hash() -> str:
    """Hash of the kernel sources' code: whole-line // comments and blank lines
    are left out, so that editing a comment does not count as a new kernel."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "normalization_gemm_tcgen05_gb300", "csrc", name), "rb") as f:
            for line in f.read().splitlines():
                t = line.strip()
                if t and not t.startswith(b"//"):
                    h.update(line + b"\n")
    return h.hexdigest()[:16]


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def load_traffic(name: str):
    """dram read+write bytes per launch from the committed ncu summary, or None
    when it is missing or was taken on kernel sources other than these."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(name)
    if not e or e.get("kernel_source_hash") != kernel_source_hash():
        return None
    return e.get("bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks, throttle reasons and the board's power limit, sampled every 100 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,power.limit")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()
        return False

    def summary(self) -> dict:
        rows = []
        limits = []
        for line in (self.out or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append({"sm": float(parts[1]), "max": float(parts[2]), "power": float(parts[3]),
                             "hw": parts[5], "hwt": parts[6], "swt": parts[7], "pcap": parts[8]})
            except ValueError:
                continue
            try:
                limits.append(float(parts[9]))
            except (IndexError, ValueError):
                pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        loaded = [r for r in rows if r["power"] > 250.0] or rows
        reasons = set()
        for r in rows:
            for key, label in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                               ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(label)
        return {"sm_mhz": statistics.median(r["sm"] for r in loaded), "sm_max_mhz": max(r["max"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows), "samples_under_load": len(loaded),
                "power_w_max": max(r["power"] for r in rows), "power_limit_w": max(limits) if limits else None}


# --------------------------------------------------------------------------
# the GPU arm
# --------------------------------------------------------------------------
class Case:
    """One sub-workload on the device: R rotating copies of its buffers."""

    def __init__(self, w: Workload, device, l2_bytes: int, seed: int = 0):
        import normalization_gemm_tcgen05_gb300 as fn
        self.fn = fn
        self.w = w
        self.dev = device
        d = make_inputs(w, seed)
        self.host = d
        fp = 2 * (w.M * w.K + w.K * w.N + 2 * w.M * w.N)
        self.R = max(2, math.ceil(2 * l2_bytes / fp))
        self.A = [d["A"].to(device) for _ in range(self.R)]
        self.B = [d["B"].to(device) for _ in range(self.R)]
        self.g = None if d["gamma"] is None else d["gamma"].to(device)
        self.b = None if d["beta"] is None else d["beta"].to(device)
        # residual-add post-norm: R rotates with A
        self.Rres = None if d["R"] is None else [d["R"].to(device) for _ in range(self.R)]
        # pre-norm with affine: the weight is folded once per copy (a one-time
        # preparation of a fixed weight, outside the timed step)
        self.fold = None
        if w.kind == "prenorm_affine":
            self.fold = [fn.fold_prenorm_affine(Bj, self.g, self.b) for Bj in self.B]
        # backward: the forward's saved output and rstd per copy, the upstream
        # gradient, and the gradients' buffers
        if w.kind == "prenorm_backward":
            fwd = [fn.lazy_prenorm_gemm(Aj, Bj, w.eps, return_rstd=True) for Aj, Bj in zip(self.A, self.B)]
            self.Cf = [c for c, _ in fwd]
            self.rstd = [r for _, r in fwd]
            self.dC = [d["dC"].to(device) for _ in range(self.R)]
            self.dA = [torch.empty((w.M, w.K), dtype=torch.bfloat16, device=device) for _ in range(self.R)]
            self.dB = [torch.empty((w.K, w.N), dtype=torch.bfloat16, device=device) for _ in range(self.R)]
            self.G = [torch.empty((w.M, w.K), dtype=torch.bfloat16, device=device) for _ in range(self.R)]
            self.work = [(torch.empty((w.M, w.N), dtype=torch.bfloat16, device=device),
                          torch.empty(w.M, dtype=torch.float32, device=device)) for _ in range(self.R)]
        if w.kind in ("postnorm_backward", "postnorm_regrouped_backward"):
            fwd = [fn.gemm_postnorm(Aj, Bj, w.norm, self.g, self.b, w.eps, return_stats=True)
                   for Aj, Bj in zip(self.A, self.B)]
            self.Cf = [c for c, _ in fwd]
            self.rstd = [st["rstd"] for _, st in fwd]
            if w.kind == "postnorm_backward":
                self.dC = [d["dC"].to(device) for _ in range(self.R)]
            else:
                # the consumer's gradient and weight; dC is materialised only
                # by the unfused comparison
                self.Gr = [d["G"].to(device) for _ in range(self.R)]
                self.Wr = [d["W"].to(device) for _ in range(self.R)]
                self.dC = [fn.gemm_ex(Gj, Wj, trans_b=True) for Gj, Wj in zip(self.Gr, self.Wr)]
        self.C = [torch.empty((w.M, w.N), dtype=torch.bfloat16, device=device) for _ in range(self.R)]
        self.Y = [torch.empty((w.M, w.N), dtype=torch.bfloat16, device=device) for _ in range(self.R)]
        nst = 3
        self.stats = [[torch.empty(w.M, dtype=torch.float32, device=device) for _ in range(nst)]
                      for _ in range(self.R)]
        # the unfused norm reads a C produced by the GEMM: rotate it too
        self.Rn = max(2, math.ceil(2 * l2_bytes / (4 * w.M * w.N)))
        self.Cn = [torch.randn((w.M, w.N), device=device).to(torch.bfloat16) for _ in range(self.Rn)]
        self.Yn = [torch.empty((w.M, w.N), dtype=torch.bfloat16, device=device) for _ in range(self.Rn)]
        self.An = self.A  # the pre-norm's input rotates with A

    # one launch of the fused kernel on copy i
    def fused(self, i: int):
        w, fn, j = self.w, self.fn, i % self.R
        st = self.stats[j]
        if w.kind == "prenorm":
            fn.lazy_prenorm_gemm(self.A[j], self.B[j], w.eps, out=self.C[j])
        elif w.kind == "prenorm_affine":
            Bf, cs, bias = self.fold[j]
            fn.prenorm_gemm(self.A[j], Bf, w.norm, cs, bias, w.eps, out=self.C[j])
        elif w.kind == "prenorm_backward":
            fn.lazy_prenorm_gemm_backward(self.A[j], self.B[j], self.Cf[j], self.dC[j], self.rstd[j],
                                          dA=self.dA[j], dB=self.dB[j], work=self.work[j])
        elif w.kind == "postnorm_backward":
            fn.gemm_postnorm_backward(self.A[j], self.B[j], self.Cf[j], self.dC[j], self.rstd[j], w.norm, self.g,
                                      self.b)
        elif w.kind == "postnorm_regrouped_backward":
            fn.gemm_postnorm_backward_regrouped(self.Gr[j], self.Wr[j], self.A[j], self.B[j], self.Cf[j],
                                                self.rstd[j], w.norm, self.g, self.b)
        elif w.residual:
            fn.gemm_add_postnorm(self.A[j], self.B[j], self.Rres[j], w.norm, self.g, self.b, w.eps, out=self.C[j])
        elif w.kind == "postnorm":
            fn.gemm_postnorm(self.A[j], self.B[j], w.norm, self.g, self.b, w.eps, pre_rmsnorm=w.pre_rmsnorm,
                             pre_eps=w.pre_eps, out=self.C[j])
        else:
            fn.gemm(self.A[j], self.B[j], out=self.C[j])
        del st

    def gemm_only(self, i: int):
        j = i % self.R
        if self.w.kind == "postnorm_regrouped_backward":  # the consumer's G @ W^T, then the two GEMMs
            self.fn.gemm_ex(self.Gr[j], self.Wr[j], trans_b=True, out=self.dC[j])
            self.fn.gemm_ex(self.dC[j], self.B[j], trans_b=True)
            self.fn.gemm_ex(self.A[j], self.dC[j], trans_a=True)
            return
        if self.w.kind == "postnorm_backward":  # the two GEMMs: dH @ B^T, A^T @ dH (dH: dC's shape)
            self.fn.gemm_ex(self.dC[j], self.B[j], trans_b=True)
            self.fn.gemm_ex(self.A[j], self.dC[j], trans_a=True)
            return
        if self.w.kind == "prenorm_backward":  # the two GEMMs of the backward: dC @ B^T, A^T @ dC
            self.fn.gemm_ex(self.dC[j], self.B[j], trans_b=True, out=self.G[j])
            self.fn.gemm_ex(self.A[j], self.dC[j], trans_a=True, out=self.dB[j])
            return
        self.fn.gemm(self.A[j], self.B[j], out=self.C[j])

    def cublas_gemm(self, i: int):
        """The same GEMM(s) by cuBLAS (torch.matmul): context for the GEMM half of
        the unfused comparison, not a product path."""
        w, j = self.w, i % self.R
        if w.kind in ("postnorm_backward", "prenorm_backward", "postnorm_regrouped_backward"):
            if w.kind == "postnorm_regrouped_backward":
                torch.matmul(self.Gr[j], self.Wr[j].t(), out=self.dC[j])
            if self._cub is None:
                self._cub = (torch.empty((w.M, w.K), dtype=torch.bfloat16, device=self.dev),
                             torch.empty((w.K, w.N), dtype=torch.bfloat16, device=self.dev))
            torch.matmul(self.dC[j], self.B[j].t(), out=self._cub[0])
            torch.matmul(self.A[j].t(), self.dC[j], out=self._cub[1])
            return
        torch.matmul(self.A[j], self.B[j], out=self.C[j])

    _cub = None

    def norm_only(self, i: int):
        """The standalone norm kernel(s) the fusion replaces, on rotating inputs."""
        w, fn, j = self.w, self.fn, i % self.Rn
        if w.kind == "prenorm":
            k = i % self.R
            fn.rmsnorm(self.A[k], None, w.eps, out=self._pre_out(k))
        elif w.kind == "prenorm_affine":
            k = i % self.R
            self._pre_norm(k, self.A[k], self._pre_out(k))
        elif w.kind in ("postnorm_backward", "postnorm_regrouped_backward"):
            # the norm backward's passes alone (dH, dgamma and dbeta)
            k = i % self.R
            fn.gemm_postnorm_backward(self.A[k], self.B[k], self.Cf[k], self.dC[k], self.rstd[k], w.norm, self.g,
                                      self.b, need=("dgamma", "dbeta"))
        elif w.kind == "prenorm_backward":
            # the normalised A materialised for dB, and the RMSNorm backward for dA
            k = i % self.R
            fn.rmsnorm(self.A[k], None, w.eps, out=self._pre_out(k))
            fn.rmsnorm_backward(self.G[k], self.A[k], self.rstd[k], out=self.dA[k])
        elif w.residual:
            k = i % self.R
            fn.add_rownorm(self.Cn[j], self.Rres[k], w.norm, self.g, self.b, w.eps, out=self.Yn[j])
        else:
            if w.pre_rmsnorm:
                k = i % self.R
                fn.rmsnorm(self.A[k], None, w.pre_eps, out=self._pre_out(k))
            if w.norm == "layernorm":
                fn.layernorm(self.Cn[j], self.g, self.b, w.eps, out=self.Yn[j])
            else:
                fn.rmsnorm(self.Cn[j], self.g, w.eps, out=self.Yn[j])

    def unfused_pipeline(self, i: int):
        """GEMM and the standalone norm(s) back to back, as an unfused model runs them."""
        w, fn, j = self.w, self.fn, i % self.R
        if w.kind == "prenorm":
            fn.rmsnorm(self.A[j], None, w.eps, out=self._pre_out(j))
            fn.gemm(self._pre_out(j), self.B[j], out=self.C[j])
        elif w.kind == "prenorm_affine":
            self._pre_norm(j, self.A[j], self._pre_out(j))
            fn.gemm(self._pre_out(j), self.B[j], out=self.C[j])
        elif w.kind == "postnorm_backward":
            # the same decomposition: the norm backward's passes, then the GEMMs
            fn.gemm_postnorm_backward(self.A[j], self.B[j], self.Cf[j], self.dC[j], self.rstd[j], w.norm, self.g,
                                      self.b)
        elif w.kind == "postnorm_regrouped_backward":
            # the consumer's GEMM writes dC, then the unfused post-norm backward
            fn.gemm_ex(self.Gr[j], self.Wr[j], trans_b=True, out=self.dC[j])
            fn.gemm_postnorm_backward(self.A[j], self.B[j], self.Cf[j], self.dC[j], self.rstd[j], w.norm, self.g,
                                      self.b)
        elif w.kind == "prenorm_backward":
            fn.rmsnorm(self.A[j], None, w.eps, out=self._pre_out(j))
            fn.gemm_ex(self.dC[j], self.B[j], trans_b=True, out=self.G[j])
            fn.gemm_ex(self._pre_out(j), self.dC[j], trans_a=True, out=self.dB[j])
            fn.rmsnorm_backward(self.G[j], self.A[j], self.rstd[j], out=self.dA[j])
        elif w.residual:
            fn.gemm(self.A[j], self.B[j], out=self.C[j])
            fn.add_rownorm(self.C[j], self.Rres[j], w.norm, self.g, self.b, w.eps, out=self.Y[j])
        else:
            if w.pre_rmsnorm:
                fn.rmsnorm(self.A[j], None, w.pre_eps, out=self._pre_out(j))
                fn.gemm(self._pre_out(j), self.B[j], out=self.C[j])
            else:
                fn.gemm(self.A[j], self.B[j], out=self.C[j])
            if w.norm == "layernorm":
                fn.layernorm(self.C[j], self.g, self.b, w.eps, out=self.Y[j])
            else:
                fn.rmsnorm(self.C[j], self.g, w.eps, out=self.Y[j])

    def _pre_norm(self, j, X, out):
        """The standalone pre-norm with its affine over rows of length K."""
        w, fn = self.w, self.fn
        if w.norm == "layernorm":
            fn.layernorm(X, self.g, self.b, w.eps, out=out)
        else:
            fn.rmsnorm(X, self.g, w.eps, out=out)

    _pre = None

    def _pre_out(self, j):
        if self._pre is None:
            self._pre = [torch.empty((self.w.M, self.w.K), dtype=torch.bfloat16, device=self.dev)
                         for _ in range(self.R)]
        return self._pre[j]

    def launches_per_call(self, what: str) -> int:
        w = self.w
        if w.kind == "prenorm_backward":
            return {"fused": 3, "gemm": 2, "norm": 2}.get(what, 4)
        if w.kind == "postnorm_backward":
            return {"fused": 4, "gemm": 2, "norm": 2}.get(what, 4)
        if w.kind == "postnorm_regrouped_backward":
            # fused: the GEMM with the norm backward's epilogue, the column sum, dA, dB
            return {"fused": 4, "gemm": 3, "norm": 2}.get(what, 5)
        if what == "fused" or what == "gemm":
            return 1
        if what == "norm":
            return 1 + (1 if (w.kind == "postnorm" and w.pre_rmsnorm) else 0)
        return 2 + (1 if (w.kind == "postnorm" and w.pre_rmsnorm) else 0)


def build_graphs(step, K: int, stream, chunk: int = 200) -> list:
    """Capture `step(i)` for i in [0, K) into CUDA graphs (uploaded by one
    untimed replay)."""
    graphs = []
    i = 0
    with torch.cuda.stream(stream):
        # one eager step on this stream first: per-stream resources (the
        # wide post-norm's workspace) exist before the capture
        step(0)
        stream.synchronize()
        while i < K:
            n = min(chunk, K - i)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for k in range(i, i + n):
                    step(k)
            graphs.append(g)
            i += n
        for g in graphs:          # one untimed replay: graph upload
            g.replay()
    torch.cuda.synchronize()
    return graphs


def time_graphs(graphs, stream, world: int, device) -> float:
    """Time one replay of `graphs` (K launches) between a barrier and a
    synchronize on each side; returns seconds (max over ranks)."""
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    with torch.cuda.stream(stream):
        for g in graphs:
            g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    t = e0.elapsed_time(e1) / 1e3
    return max_over_ranks(t, world, device)


# The step (the fused launch of every sub-workload) is timed once, K steps.
# For latency_hidden every leg of every sub-workload is then timed in ROUNDS
# rounds, the legs of a sub-workload back to back within a round (so the
# fused kernel and the unfused pieces it is compared with run in the same
# thermal and power state of the GPU), in reverse order every other round (so
# a drift of the clock within a round favours no leg), and each leg reports
# its median round.  The legs are graphs of LEG_LAUNCHES launches whatever K
# is: a leg of a few hundred launches runs long enough for the clock to settle
# differently under the power cap from one leg to the next, which the
# comparison of per-launch times should not see.
ROUNDS = 6
LEG_LAUNCHES = 20


def run_ours(args, names, world, rank, local):
    import normalization_gemm_tcgen05_gb300 as fn
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    props = torch.cuda.get_device_properties(device)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2**20))
    peaks = load_peaks()
    cases = [Case(WORKLOADS[n], device, l2) for n in names]
    stream = torch.cuda.Stream(device)
    K, W = args.steps, args.warmup

    for c in cases:                      # warm-up (loads kernels, first-use set-up)
        for i in range(W):
            c.fused(i)
            c.gemm_only(i)
            c.norm_only(i)
            c.unfused_pipeline(i)
            c.cublas_gemm(i)
    torch.cuda.synchronize()
    fn.check_status(device)

    KL = min(K, LEG_LAUNCHES)
    steps = [build_graphs(c.fused, K, stream) for c in cases]
    legs = [[build_graphs(f, KL, stream) for f in (c.fused, c.gemm_only, c.norm_only, c.unfused_pipeline,
                                                   c.cublas_gemm)] for c in cases]
    rounds = [[[] for _ in range(5)] for _ in cases]
    with ClockSampler(local) as clk:
        step_t = [time_graphs(steps[k], stream, world, device) for k in range(len(cases))]
        for r in range(ROUNDS):
            for k in range(len(cases)):
                for j in (range(5) if r % 2 == 0 else range(4, -1, -1)):
                    rounds[k][j].append(time_graphs(legs[k][j], stream, world, device))
    del legs, steps
    fn.check_status(device)
    med = [[statistics.median(rounds[k][j]) for j in range(5)] for k in range(len(cases))]
    fused_t, gemm_t, norm_t, pipe_t, cub_t = ([med[k][j] for k in range(len(cases))] for j in range(5))

    # ---- end to end through the public API with pinned host buffers ----
    e2e = run_e2e(cases, K, W, world, device)

    flops_step = sum(c.w.flops for c in cases)
    t_step = sum(step_t) / K
    value = world * flops_step / t_step / 1e12
    dom = max(range(len(cases)), key=lambda k: step_t[k])
    dc = cases[dom]
    per_launch = step_t[dom] / K
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)

    def roofline_of(w, t):
        """(bound, achieved, peak, unit) of one launch of w taking t seconds."""
        if w.flops / w.algorithmic_bytes < ridge:
            return "hbm", w.algorithmic_bytes / t / 1e9, peaks["hbm_gbs"], "GB/s"
        return "tensor", w.flops / t / 1e12, peaks["bf16_tflops"], "TFLOP/s"

    bound, achieved, peak, unit = roofline_of(dc.w, per_launch)
    roof = {"bound": bound, "achieved": round(achieved, 1), "peak": peak, "unit": unit}
    roof["frac"] = round(roof["achieved"] / roof["peak"], 4)
    if bound == "tensor":
        # context: the same against the measured sustained (power-capped) rate
        roof["frac_of_sustained"] = round(achieved / peaks["bf16_tflops_sustained"], 4)
    roof["traffic"] = load_traffic(dc.w.name)
    roof["kernel"] = (f"fused backward (row pass + dgrad + wgrad: one call, three launches), {dc.w.name}"
                      if dc.w.kind == "prenorm_backward" else f"fused kernel, {dc.w.name}")
    roof["algorithmic_bytes"] = dc.w.algorithmic_bytes
    roof["peak_source"] = peaks["source"] + (" (burst)" if roof["bound"] == "tensor" else "")

    hidden = {}
    for k, c in enumerate(cases):
        tf, tg, tn, tp = fused_t[k] / KL, gemm_t[k] / KL, norm_t[k] / KL, pipe_t[k] / KL
        tc = cub_t[k] / KL
        b_k, a_k, p_k, _ = roofline_of(c.w, tf)
        hidden[c.w.name] = {
            "t_fused_us": round(tf * 1e6, 3), "t_gemm_us": round(tg * 1e6, 3), "t_norm_us": round(tn * 1e6, 3),
            "t_unfused_pipeline_us": round(tp * 1e6, 3),
            "hidden_vs_standalone_norm": round((tg + tn - tf) / tn, 4),
            "hidden_vs_pipeline": round((tp - tf) / (tp - tg), 4) if tp > tg else None,
            "fused_tflops": round(c.w.flops / tf / 1e12, 2),
            "fused_gbs": round(c.w.algorithmic_bytes / tf / 1e9, 1),
            "roofline": {"bound": b_k, "frac": round(a_k / p_k, 4)},
            # context only, not the product path: the same GEMM by cuBLAS
            # (torch.matmul), and "hidden" against cuBLAS + this library's
            # standalone norm
            "context_t_cublas_gemm_us": round(tc * 1e6, 3),
            "context_hidden_vs_cublas_plus_norm": round((tc + tn - tf) / tn, 4),
        }
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": round(t_step * 1e3, 6), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: seeded inputs with the workload table's shapes and distributions",
        "config": {"workload": args.workload + ": " + GROUP_TEXT.get(args.workload, ""),
                   "sub_workloads": names, "l2": f"inputs/outputs rotate over >= 2x L2 ({l2 >> 20} MiB)",
                   "timing": f"CUDA graphs, CUDA events on the launching stream: the step once, K launches; "
                             f"for latency_hidden each leg of each sub-workload as a graph of {KL} launches in "
                             f"{ROUNDS} rounds, the legs of a sub-workload back to back in a round, in reverse "
                             f"order every other round, the median round reported",
                   "parallelism": f"{world} independent replica(s)"},
        "roofline": roof,
        "latency_hidden": hidden,
        "e2e": e2e,
        "gpu_launches": K * sum(c.launches_per_call("fused") for c in cases),
        "clocks": clk.summary(),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(names, args.cpu_seconds)
    return line


def link_rates(device, nbytes: int = 64 << 20, reps: int = 5) -> tuple:
    """Best-of-`reps` GB/s of one pinned host -> device and one device -> host
    copy of `nbytes` (tensor.copy_, i.e. cudaMemcpyAsync), CUDA events."""
    h = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d = torch.empty(nbytes, dtype=torch.uint8, device=device)
    best = [float("inf"), float("inf")]
    for _ in range(reps):
        for k, (dst, src) in enumerate(((d, h), (h, d))):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record()
            dst.copy_(src, non_blocking=True)
            e1.record()
            torch.cuda.synchronize()
            best[k] = min(best[k], e0.elapsed_time(e1) / 1e3)
    return nbytes / best[0] / 1e9, nbytes / best[1] / 1e9


def run_e2e(cases, K, W, world, device) -> dict:
    """K steps through the public API: H2D copy of every input from pinned
    host memory, the fused call, D2H copy of the output, per step."""
    import normalization_gemm_tcgen05_gb300 as fn
    host = []
    for c in cases:
        hA = c.host["A"].pin_memory()
        hB = c.host["B"].pin_memory()
        hg = None if c.host["gamma"] is None else c.host["gamma"].pin_memory()
        hb = None if c.host["beta"] is None else c.host["beta"].pin_memory()
        hR = None if c.host["R"] is None else c.host["R"].pin_memory()
        hC = torch.empty((c.w.M, c.w.N), dtype=torch.bfloat16).pin_memory()
        bwd = None
        if c.w.kind.endswith("_backward"):
            # the backward's inputs in (forward output, rstd, and the upstream
            # gradient: dC, or for the regrouped form G and W), dA and dB out
            ins = [(c.Cf[0].cpu().pin_memory(), c.Cf[0]), (c.rstd[0].cpu().pin_memory(), c.rstd[0])]
            if c.w.kind == "postnorm_regrouped_backward":
                ins += [(c.host["G"].pin_memory(), c.Gr[0]), (c.host["W"].pin_memory(), c.Wr[0])]
            else:
                ins += [(c.host["dC"].pin_memory(), c.dC[0])]
            bwd = (ins, (torch.empty((c.w.M, c.w.K), dtype=torch.bfloat16).pin_memory(),
                         torch.empty((c.w.K, c.w.N), dtype=torch.bfloat16).pin_memory()))
            hC = None
        host.append((hA, hB, hg, hb, hR, hC, bwd))
    h2d = sum(t.numel() * t.element_size() for h in host for t in h[:5] if t is not None)
    h2d += sum(t.numel() * t.element_size() for h in host if h[6] is not None for t, _ in h[6][0])
    d2h = sum(h[5].numel() * h[5].element_size() for h in host if h[5] is not None)
    d2h += sum(t.numel() * t.element_size() for h in host if h[6] is not None for t in h[6][1])

    # Three streams, so that the host link carries inputs in and results out
    # at the same time and the kernels run meanwhile: per sub-workload, the
    # H2D copies of its inputs (after its previous call has read them), the
    # fused call (after its inputs are in and its previous output has been
    # read back), then the D2H copy of its output.
    s_in, s_cmp, s_out = (torch.cuda.Stream(device) for _ in range(3))
    ev_in = [torch.cuda.Event() for _ in cases]
    ev_cmp = [torch.cuda.Event() for _ in cases]
    ev_out = [torch.cuda.Event() for _ in cases]
    for k in range(len(cases)):
        for ev, st in ((ev_in[k], s_in), (ev_cmp[k], s_cmp), (ev_out[k], s_out)):
            ev.record(st)

    def step():
        for k, (c, (hA, hB, hg, hb, hR, hC, bwd)) in enumerate(zip(cases, host)):
            dA, dB = c.A[0], c.B[0]
            w = c.w
            s_in.wait_event(ev_cmp[k])
            with torch.cuda.stream(s_in):
                dA.copy_(hA, non_blocking=True)
                dB.copy_(hB, non_blocking=True)
                if hg is not None:
                    c.g.copy_(hg, non_blocking=True)
                if hb is not None:
                    c.b.copy_(hb, non_blocking=True)
                if hR is not None:
                    c.Rres[0].copy_(hR, non_blocking=True)
                if bwd is not None:
                    for src, dst in bwd[0]:
                        dst.copy_(src, non_blocking=True)
                ev_in[k].record(s_in)
            s_cmp.wait_event(ev_in[k])
            s_cmp.wait_event(ev_out[k])
            with torch.cuda.stream(s_cmp):
                if bwd is not None:
                    if w.kind == "prenorm_backward":
                        fn.lazy_prenorm_gemm_backward(dA, dB, c.Cf[0], c.dC[0], c.rstd[0], dA=c.dA[0], dB=c.dB[0],
                                                      work=c.work[0])
                        outs = (c.dA[0], c.dB[0])
                    elif w.kind == "postnorm_regrouped_backward":
                        g = fn.gemm_postnorm_backward_regrouped(c.Gr[0], c.Wr[0], dA, dB, c.Cf[0], c.rstd[0],
                                                                w.norm, c.g, c.b, need=("dA", "dB"))
                        outs = (g["dA"], g["dB"])
                    else:
                        g = fn.gemm_postnorm_backward(dA, dB, c.Cf[0], c.dC[0], c.rstd[0], w.norm, c.g, c.b,
                                                      need=("dA", "dB"))
                        outs = (g["dA"], g["dB"])
                elif w.kind == "prenorm":
                    fn.lazy_prenorm_gemm(dA, dB, w.eps, out=c.C[0])
                    outs = (c.C[0],)
                elif w.kind == "prenorm_affine":
                    # the weight arrives from the host every step: fold, then the fused GEMM
                    Bf, cs, bias = c.fold[0]
                    fn.fold_prenorm_affine(dB, c.g, c.b, out=Bf, colsum_out=cs, bias_out=bias)
                    fn.prenorm_gemm(dA, Bf, w.norm, cs if w.norm == "layernorm" else None, bias, w.eps,
                                    out=c.C[0])
                    outs = (c.C[0],)
                elif w.residual:
                    fn.gemm_add_postnorm(dA, dB, c.Rres[0], w.norm, c.g, c.b, w.eps, out=c.C[0])
                    outs = (c.C[0],)
                else:
                    fn.gemm_postnorm(dA, dB, w.norm, c.g, c.b, w.eps, pre_rmsnorm=w.pre_rmsnorm,
                                     pre_eps=w.pre_eps, out=c.C[0])
                    outs = (c.C[0],)
                ev_cmp[k].record(s_cmp)
            s_out.wait_event(ev_cmp[k])
            with torch.cuda.stream(s_out):
                dsts = bwd[1] if bwd is not None else (hC,)
                for dst, src in zip(dsts, outs):
                    src.record_stream(s_out)  # (the backward's outputs are fresh allocations)
                    dst.copy_(src, non_blocking=True)
                ev_out[k].record(s_out)

    def join():
        # the default stream waits for the three streams' work so far
        cur = torch.cuda.current_stream(device)
        for st in (s_in, s_cmp, s_out):
            cur.wait_stream(st)

    for _ in range(W):
        step()
    join()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for st in (s_in, s_cmp, s_out):  # nothing of the timed steps starts before e0
        st.wait_stream(torch.cuda.current_stream(device))
    for _ in range(K):
        step()
    join()
    e1.record()
    torch.cuda.synchronize()
    barrier(world)
    t = max_over_ranks(e0.elapsed_time(e1) / 1e3, world, device)
    flops = sum(c.w.flops for c in cases)
    h2d_gbs, d2h_gbs = link_rates(device)
    return {"value": round(world * K * flops / t / 1e12, 4), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(t / K * 1e3, 4),
            # the host link, measured on this machine: one 64 MiB pinned copy each
            # way, and the step's copies at those rates (each direction on its
            # own stream, the two directions overlapping)
            "h2d_gbs": round(h2d_gbs, 1), "d2h_gbs": round(d2h_gbs, 1),
            "h2d_ms_at_link_rate": round(h2d / h2d_gbs / 1e6, 4),
            "d2h_ms_at_link_rate": round(d2h / d2h_gbs / 1e6, 4),
            "streams": "inputs in, compute and results out on three streams"}


# --------------------------------------------------------------------------
# the oracle on the host cores
# --------------------------------------------------------------------------
def oracle_step(w: Workload, d: dict, rows: np.ndarray):
    import oracle
    A = d["A64"][rows]
    if w.kind == "prenorm":
        oracle.lazy_prenorm_gemm(A, d["B64"], w.eps)
    elif w.kind == "prenorm_backward":
        oracle.lazy_prenorm_gemm_backward(A, d["B64"], d["dC64"][rows], w.eps)
    elif w.kind == "postnorm_backward":
        oracle.gemm_postnorm_backward(A, d["B64"], d["dC64"][rows], w.norm, d["g64"], d["b64"], w.eps)
    elif w.kind == "postnorm_regrouped_backward":
        oracle.gemm_postnorm_backward_regrouped(d["G64"][rows], d["W64"], A, d["B64"], w.norm, d["g64"], d["b64"],
                                                w.eps)
    elif w.kind == "prenorm_affine":
        oracle.prenorm_affine_gemm(A, d["B64"], w.norm, d["g64"], d["b64"], w.eps)
    elif w.residual:
        oracle.gemm_add_postnorm(A, d["B64"], d["R64"][rows], w.norm, d["g64"], d["b64"], w.eps)
    elif w.kind == "postnorm":
        oracle.gemm_postnorm(A, d["B64"], w.norm, d["g64"], d["b64"], w.eps, pre_rmsnorm=w.pre_rmsnorm,
                             pre_eps=w.pre_eps)
    else:
        oracle.gemm(A, d["B64"])


def _oracle_inputs(names):
    from workloads import to_f64
    out = []
    for n in names:
        w = WORKLOADS[n]
        d = make_inputs(w, 0)
        out.append((w, {"A64": to_f64(d["A"]), "B64": to_f64(d["B"]), "g64": to_f64(d["gamma"]),
                        "b64": to_f64(d["beta"]), "R64": to_f64(d["R"]), "dC64": to_f64(d["dC"]),
                        "G64": to_f64(d["G"]), "W64": to_f64(d["W"])}))
    return out


def _cores() -> int:
    v = os.environ.get("OPENBLAS_NUM_THREADS") or os.environ.get("OMP_NUM_THREADS")
    return int(v) if v else (os.cpu_count() or 1)


def _sample_rows(w: Workload, budget_flops: float) -> np.ndarray:
    per_row = w.flops / w.M
    n = int(max(1, min(w.M, budget_flops // per_row)))
    return np.linspace(0, w.M - 1, n).astype(np.int64)


def cpu_baseline(names, seconds: float) -> dict:
    """The fp64 oracle as it stands, on a bounded row sample of each sub-workload."""
    inputs = _oracle_inputs(names)
    flops = 0.0
    t_total = 0.0
    samples = []
    for w, d in inputs:
        rows = _sample_rows(w, 4e9)
        t0 = time.perf_counter()
        reps = 0
        while True:
            oracle_step(w, d, rows)
            reps += 1
            if time.perf_counter() - t0 >= seconds / len(inputs):
                break
        dt = time.perf_counter() - t0
        flops += reps * len(rows) * w.flops / w.M
        t_total += dt
        samples.append(f"{w.name}: {reps} x {len(rows)} of {w.M} rows")
    return {"value": round(flops / t_total / 1e12, 6), "unit": "TFLOP/s", "cores": _cores(), "kind": "oracle",
            "sample": "; ".join(samples) + " (fp64 numpy oracle, all N columns of each sampled row)"}


def run_reference(args, names, world, rank):
    """--impl reference: the oracle on the host cores, K timed steps each a bounded row sample."""
    if world > 1 and rank != 0:
        return None
    inputs = _oracle_inputs(names)
    budget = 2e9 / len(inputs)
    sampled = [(w, d, _sample_rows(w, budget)) for w, d in inputs]
    for _ in range(args.warmup):
        for w, d, rows in sampled:
            oracle_step(w, d, rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        for w, d, rows in sampled:
            oracle_step(w, d, rows)
    t = time.perf_counter() - t0
    flops = args.steps * sum(len(rows) * w.flops / w.M for w, d, rows in sampled)
    value = flops / t / 1e12
    sample = "; ".join(f"{w.name}: {len(rows)} of {w.M} rows" for w, d, rows in sampled)
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic: seeded inputs with the workload table's shapes and distributions",
        "config": {"workload": args.workload + ": " + GROUP_TEXT.get(args.workload, ""), "sub_workloads": names},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": _cores(), "kind": "oracle",
                         "sample": sample + " per step (fp64 numpy oracle on the host cores)"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def profile_case(args):
    """Eager launches of one kernel on one sub-workload (a small, bounded ncu target)."""
    import normalization_gemm_tcgen05_gb300 as fn
    device = torch.device("cuda", 0)
    props = torch.cuda.get_device_properties(device)
    c = Case(WORKLOADS[args.profile_case], device, int(getattr(props, "L2_cache_size", 126 * 2**20)))
    step = {"fused": c.fused, "gemm": c.gemm_only, "norm": c.norm_only}[args.profile_kernel]
    for i in range(args.warmup + args.steps):
        step(i)
    torch.cuda.synchronize()
    fn.check_status(device)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="main", choices=sorted(GROUPS) + ["all"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--profile-case", default=None, choices=sorted(WORKLOADS),
                    help="for ncu: run W + K eager launches of one kernel of one sub-workload and exit")
    ap.add_argument("--profile-kernel", default="fused", choices=["fused", "gemm", "norm"])
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_env()
    if args.profile_case:
        profile_case(args)
        return
    if args.impl == "ours":
        if not torch.cuda.is_available():
            raise SystemExit("bench.py needs a CUDA device (the fused path has no CPU fallback)")
        torch.cuda.set_device(local)
        init_dist(world, "nccl")
    groups = ["main", "res", "preaff", "bwd"] if args.workload == "all" else [args.workload]
    for gname in groups:
        args.workload = gname
        names = GROUPS[gname]
        if args.impl == "reference":
            line = run_reference(args, names, world, rank)
        else:
            line = run_ours(args, names, world, rank, local)
        if line is not None and rank == 0:
            print(json.dumps(line), flush=True)
    if world > 1 and torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
