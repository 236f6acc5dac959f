"""Helpers shared by the GPU parity tests: tolerances and comparisons.

Tolerances (stated by the benchmark spec for this path and written here once):
* outputs:  max |C_gpu - C_ref| <= 2e-2 * max |C_ref| + 1e-3 over the compared
  elements (bf16 output, fp32 accumulation);
* rstd:     |r_gpu - r_ref| <= 1e-4 * |r_ref| per row;
* mean:     |mu_gpu - mu_ref| <= 1e-4 * (|mu_ref| + sigma_ref) per row, with
  sigma_ref = 1 / rstd_ref (the row's own scale: a LayerNorm row mean is near 0
  here, so a purely relative test would be ill-posed).
"""
from __future__ import annotations

import numpy as np
import torch

OUT_REL = 2e-2
OUT_ABS = 1e-3
STAT_REL = 1e-4


def np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().double().cpu().numpy()


def assert_out_close(got: torch.Tensor, ref: np.ndarray, what: str = "C") -> float:
    g = np64(got)
    assert g.shape == ref.shape, f"{what}: shape {g.shape} != {ref.shape}"
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    err = float(np.max(np.abs(g - ref))) if g.size else 0.0
    bound = OUT_REL * float(np.max(np.abs(ref))) + OUT_ABS if ref.size else OUT_ABS
    assert err <= bound, f"{what}: max |err| {err:.4e} > bound {bound:.4e}"
    return err


def assert_rstd_close(got: torch.Tensor, ref: np.ndarray, what: str = "rstd") -> None:
    g = np64(got)
    rel = np.abs(g - ref) / np.abs(ref)
    worst = int(np.argmax(rel))
    assert rel[worst] <= STAT_REL, f"{what}: row {worst} rel err {rel[worst]:.3e} (got {g[worst]}, ref {ref[worst]})"


def assert_mean_close(got: torch.Tensor, ref_mean: np.ndarray, ref_rstd: np.ndarray, what: str = "mean") -> None:
    g = np64(got)
    scale = np.abs(ref_mean) + 1.0 / ref_rstd
    rel = np.abs(g - ref_mean) / scale
    worst = int(np.argmax(rel))
    assert rel[worst] <= STAT_REL, f"{what}: row {worst} err {rel[worst]:.3e} of the row scale"
