"""Shared helpers for the test suite (tolerances, device transfer)."""
from __future__ import annotations

import numpy as np
import pytest

# fp32 path: max abs error on outputs and final state.
F32_ATOL = 1e-4
# bf16-input path: per (sequence, head) max|x - x*| / max(max|x*|, 1e-6).
BF16_REL = 2e-2


def cuda_or_skip():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def ensure_built():
    from linear_attention_recurrence_02_gb300 import build
    return build.build_library()


def to_dev(a, dtype, torch, device="cuda"):
    """numpy float32/float64 -> torch tensor of `dtype` on the device."""
    t = torch.from_numpy(np.ascontiguousarray(np.asarray(a, dtype=np.float32)))
    return t.to(device=device, dtype=dtype).contiguous()


def to_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def rel_err_per_unit(got, ref, unit_axes):
    """max|got-ref| / max(max|ref|, 1e-6) over the non-unit axes, per unit."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    red = tuple(i for i in range(ref.ndim) if i not in unit_axes)
    num = np.max(np.abs(got - ref), axis=red)
    den = np.maximum(np.max(np.abs(ref), axis=red), 1e-6)
    return num / den


def assert_close(got, ref, dtype_is_bf16, unit_axes, what=""):
    if dtype_is_bf16:
        r = rel_err_per_unit(got, ref, unit_axes)
        assert np.all(np.isfinite(got)), f"{what}: non-finite values"
        assert r.max() <= BF16_REL, f"{what}: max per-unit relative error {r.max():.3e} > {BF16_REL}"
        return float(r.max())
    err = np.max(np.abs(np.asarray(got, np.float64) - np.asarray(ref, np.float64))) if np.size(ref) else 0.0
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    assert err <= F32_ATOL, f"{what}: max abs error {err:.3e} > {F32_ATOL}"
    return float(err)


def row_rel_err(got, ref, floor=1e-6):
    """Per-row relative error of [..., D] arrays: max_j |got - ref| / max(max_j |ref|, floor)
    for every row (a (token, head) or (sequence, head) output vector)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    num = np.max(np.abs(got - ref), axis=-1)
    den = np.maximum(np.max(np.abs(ref), axis=-1), floor)
    return (num / den).ravel()


def report_rows(got, ref, what):
    """Print the 99.9th percentile and the maximum of the per-row relative
    error (a report beside the per-(sequence, head) gate, not a gate). Rows
    whose reference is ~0 (below 1e-3 of the largest row) are left out: their
    relative error measures only rounding of a vanishing value."""
    ref = np.asarray(ref, np.float64)
    rmax = np.max(np.abs(ref), axis=-1).ravel()
    keep = rmax >= 1e-3 * max(float(rmax.max()) if rmax.size else 0.0, 1e-30)
    r = row_rel_err(got, ref)[keep]
    if r.size:
        print(f"{what}: per-row relative error p99.9 {np.percentile(r, 99.9):.3e}, max {r.max():.3e} "
              f"({r.size} rows)")
    return r
