"""Helpers shared by the GPU parity tests: tensor -> float64 numpy, tolerances."""

from __future__ import annotations

import numpy as np
import torch

# bf16 storage path gate; FP8/FP4 storage path gate; float32 path internal target
TOL_BF16 = 2e-2
TOL_MIXED = 6e-2
TOL_F32 = 1e-4
TOL_SCORES_REL = 1e-3


def f64(t) -> np.ndarray:
    if isinstance(t, np.ndarray):
        return t.astype(np.float64)
    if t.dtype in (torch.uint8, torch.int32, torch.int64):
        return t.cpu().numpy()
    return t.detach().float().cpu().numpy().astype(np.float64)


def host(x: dict) -> dict:
    """numpy copies of an input dict (bf16 widened exactly to float64)."""
    return {k: f64(v) for k, v in x.items()}


def assert_close(got, ref, atol, rtol, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    err = np.abs(got - ref)
    bound = atol + rtol * np.abs(ref)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} elements out of tolerance; "
                             f"worst at {i}: got {got[i]!r} ref {ref[i]!r} (max abs err "
                             f"{err.max():.3g})")


def assert_scores_close(got_row, ref_row, what=""):
    """Indexer row parity: identical -inf pattern, |dI| <= 1e-3 * max|I_ref| on the rest."""
    got_row = np.asarray(got_row, dtype=np.float64)
    ref_row = np.asarray(ref_row, dtype=np.float64)
    ninf_g, ninf_r = np.isneginf(got_row), np.isneginf(ref_row)
    assert np.array_equal(ninf_g, ninf_r), f"{what}: -inf pattern differs"
    fin = ~ninf_r
    if fin.any():
        scale = np.abs(ref_row[fin]).max()
        err = np.abs(got_row[fin] - ref_row[fin]).max()
        assert err <= TOL_SCORES_REL * scale + 1e-30, f"{what}: max err {err:.3g} vs {scale:.3g}"
