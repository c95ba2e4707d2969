"""Helpers shared by the GPU parity tests (comparison, conversions)."""

import inspect

import numpy as np
import torch

# Tolerances (normwise: max|got - ref| <= tol * max|ref|).
#   fp32 paths: 1e-5; bf16 outputs and grads at fp32 accumulation: 1e-2.
F32_TOL = 1e-5
BF16_TOL = 1e-2

# Unit roundoff of fp32 (round to nearest).
U32 = 2.0 ** -24


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


def ulp(x, dtype: str) -> np.ndarray:
    """Spacing of the storage format at |x|: 2^(floor(log2|x|) - p + 1) with
    p = 8 significand bits for bf16 and 24 for fp32, and the subnormal
    spacing (2^-133 for bf16, 2^-149 for fp32) at the bottom of the range."""
    p, tiny = (8, 2.0 ** -133) if dtype == "bf16" else (24, 2.0 ** -149)
    m, e = np.frexp(np.abs(np.asarray(x, dtype=np.float64)))  # |x| = m 2^e, m in [0.5, 1)
    sp = np.ldexp(1.0, e - p)
    return np.maximum(np.where(m == 0.0, 0.0, sp), tiny)


def assert_elementwise(got, ref, mag, n_roundings: int, dtype: str, what=""):
    """Per-element bound for an output that the kernel accumulates in fp32
    with n_roundings rounded operations per element and stores with one
    rounding to `dtype`, against the oracle's exact sum rounded to fp32 and
    then to `dtype`:
        |got - ref| <= ulp_dtype(max(|got|, |ref|)) + (n_roundings + 2) u32 mag
    where mag is the element's sum of absolute terms and u32 = 2^-24.  The
    fp32 sum differs from the exact one by at most n u32 mag (recursive
    summation, one rounding per operation); rounding is monotone, so the two
    stored values differ by at most that plus one step of the format."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    mag = np.asarray(mag, dtype=np.float64)
    assert got.shape == ref.shape == mag.shape, f"{what}: shapes {got.shape} {ref.shape} {mag.shape}"
    if ref.size == 0:
        return
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    bound = ulp(np.maximum(np.abs(got), np.abs(ref)), dtype) + (n_roundings + 2) * U32 * mag
    bad = np.abs(got - ref) > bound
    if bad.any():
        i = np.unravel_index(int(np.argmax(np.abs(got - ref) - bound)), got.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {got.size} elements past the per-element bound; "
            f"worst at {i}: got {got[i]!r} ref {ref[i]!r} bound {bound[i]:.3e}")


def assert_bitwise(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, f"{what}: shape {got.shape} vs {ref.shape}"
    bad = got != ref
    assert not bad.any(), f"{what}: {int(bad.sum())} of {got.size} elements differ"


def tol_for(dtype: str) -> float:
    return F32_TOL if dtype == "f32" else BF16_TOL


def torch_dtype(dtype: str):
    return torch.float32 if dtype == "f32" else torch.bfloat16


class StatusChecked:
    """The binding module, with the device status word of every call that
    takes one checked: a call made without a ``dev_status`` gets a fresh
    zeroed word, and after the call (``moe_check_status`` synchronises the
    stream) the word must still read MOE_OK.  Calls given their own word are
    passed through unchanged, so tests that expect an error check it
    themselves."""

    def __init__(self, mod):
        self._m = mod
        self._wrapped = {}

    def __getattr__(self, name):
        f = getattr(self._m, name)
        if not (name.startswith("moe_") and callable(f)):
            return f
        try:
            sig = inspect.signature(f)
        except (TypeError, ValueError):
            return f
        if "dev_status" not in sig.parameters:
            return f
        if name not in self._wrapped:
            m = self._m

            def checked(*args, **kw):
                if sig.bind_partial(*args, **kw).arguments.get("dev_status") is not None:
                    return f(*args, **kw)
                st = m.new_status()
                kw["dev_status"] = st
                out = f(*args, **kw)
                rc = m.moe_check_status(st)
                assert rc == m.MOE_OK, f"{name}: device status {rc} ({m.status_name(rc)})"
                return out

            checked.__name__ = name
            self._wrapped[name] = checked
        return self._wrapped[name]
