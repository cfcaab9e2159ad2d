"""Comparison helpers for GPU-vs-oracle parity tests.

Tolerances (the method fixes fp32 and bf16 bars; their reading):
  - fp32 inputs: max |gpu - oracle| <= 1e-4, element by element.
  - bf16 inputs (fp32 accumulation, bf16 output): for every output row
    (one position of one head), max_c |gpu - oracle| <= 2e-2 * max_c |oracle|.
    The row-wise max norm keeps the bar relative for late positions of long
    sequences, whose outputs are far smaller than those of early positions.
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
