"""Helpers shared by the GPU parity tests (comparison, conversions)."""

import numpy as np
import torch

# Tolerances (normwise: max|got - ref| <= tol * max|ref|).
#   fp32 paths: 1e-5; bf16 outputs and grads at fp32 accumulation: 1e-2.
F32_TOL = 1e-5
BF16_TOL = 1e-2


def np64(t: torch.Tensor) -> np.ndarray:
    t = t.detach()
    if t.dtype in (torch.bfloat16, torch.float16):
        t = t.float()
    a = t.cpu().numpy()
    return a.astype(np.float64) if a.dtype.kind == "f" else a.astype(np.int64)


def assert_normwise(got, ref, tol, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, f"{what}: shape {got.shape} vs {ref.shape}"
    if ref.size == 0:
        return
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    scale = float(np.max(np.abs(ref)))
    err = float(np.max(np.abs(got - ref)))
    if scale == 0.0:
        assert err == 0.0, f"{what}: expected zeros, max|got| = {err:.3e}"
        return
    assert err <= tol * scale, f"{what}: max|diff| {err:.3e} > {tol} * max|ref| {scale:.3e}"


def tol_for(dtype: str) -> float:
    return F32_TOL if dtype == "f32" else BF16_TOL


def torch_dtype(dtype: str):
    return torch.float32 if dtype == "f32" else torch.bfloat16
