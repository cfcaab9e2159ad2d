"""Comparison helpers for GPU-vs-oracle parity tests.

Tolerances (the method fixes fp32 and bf16 bars; their reading):
  - fp32 inputs: max |gpu - oracle| <= 1e-4, element by element.
  - bf16 inputs (fp32 accumulation, bf16 output): for every output row
    (one position of one head), max_c |gpu - oracle| <= 2e-2 * max_c |oracle|.
    The row-wise max norm keeps the bar relative for late positions of long
    sequences, whose outputs are far smaller than those of early positions.
Gradients (dq, dk, dv) take the same bars, read for tensors that are not
bounded by the values as outputs are: bf16, the same row-relative 2e-2;
fp32, max |gpu - oracle| <= 1e-4 * max(1, max |oracle|) per head.  A row
whose exact gradient cancels to zero (e.g. dq at position 0, or any row when
all values are equal) has no relative scale of its own, so the bf16 row bar
is taken against max(row max, floor) with floor = 1e-4 * max|dout| * max|v|,
the natural scale of the gradient terms that cancel there.
"""
from __future__ import annotations

import numpy as np
import torch

F32_ABS_TOL = 1e-4
BF16_ROW_REL_TOL = 2e-2


def np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def assert_f32_close(got, ref, tol=F32_ABS_TOL, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.max(np.abs(got - ref)) if got.size else 0.0
    assert err <= tol, f"{what}: max abs err {err:.3e} > {tol:.1e}"
    return err


def row_rel_err(got, ref):
    """max over rows of max_c|g - o| / max_c|o| (rows = last axis)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    num = np.max(np.abs(got - ref), axis=-1)
    den = np.maximum(np.max(np.abs(ref), axis=-1), 1e-30)
    return float(np.max(num / den)) if num.size else 0.0


def assert_bf16_rows_close(got, ref, tol=BF16_ROW_REL_TOL, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    e = row_rel_err(got, ref)
    assert e <= tol, f"{what}: row-relative err {e:.3e} > {tol:.1e}"
    return e


def assert_close(got, ref, dtype: str, what=""):
    if dtype == "f32":
        return assert_f32_close(got, ref, what=what)
    return assert_bf16_rows_close(got, ref, what=what)


def assert_grad_close(got, ref, dtype: str, what="", floor=0.0):
    """Gradient tensors [..., heads, N, cols]: bf16 row-relative 2e-2 against
    max(row max, floor); fp32 1e-4 relative to max(1, the head's largest
    |entry|)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite gradient"
    if dtype != "f32":
        num = np.max(np.abs(got - ref), axis=-1)
        den = np.maximum(np.max(np.abs(ref), axis=-1), max(floor, 1e-30))
        e = float(np.max(num / den)) if num.size else 0.0
        assert e <= BF16_ROW_REL_TOL, f"{what}: row-relative err {e:.3e} > {BF16_ROW_REL_TOL:.1e}"
        return e
    g = got.reshape(-1, got.shape[-2] * got.shape[-1])
    r = ref.reshape(g.shape)
    err = np.max(np.abs(g - r), axis=1) / np.maximum(np.max(np.abs(r), axis=1), 1.0)
    e = float(np.max(err)) if err.size else 0.0
    assert e <= F32_ABS_TOL, f"{what}: fp32 gradient err {e:.3e} > {F32_ABS_TOL:.1e}"
    return e


def assert_state_close(got, ref, rtol, what=""):
    """Memories S, z: max abs error relative to the largest |entry| per head."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    g = got.reshape(got.shape[0] * got.shape[1], -1)
    r = ref.reshape(ref.shape[0] * ref.shape[1], -1)
    err = np.max(np.abs(g - r), axis=1) / np.maximum(np.max(np.abs(r), axis=1), 1e-30)
    assert float(np.max(err)) <= rtol, f"{what}: state rel err {np.max(err):.3e} > {rtol:.1e}"
    return float(np.max(err))
