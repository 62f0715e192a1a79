"""Parity criteria between the CUDA path and the float64 oracle.

Output: relative L2 error ||gpu - oracle|| / ||oracle|| <= 2e-3 over the compared
outputs, and max |gpu - oracle| <= 1e-2, against the unrounded float64 oracle.
LSE: |gpu - oracle| <= 1e-4 * max(1, |oracle|). Rows with no visible key must come out
as out == 0 and lse == -inf on both sides.
"""
from __future__ import annotations

import numpy as np
import torch

REL_L2 = 2e-3
MAX_ABS = 1e-2
LSE_REL = 1e-4


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def compare(out_gpu, lse_gpu, out_ref, lse_ref, what=""):
    og = to_np(out_gpu) if isinstance(out_gpu, torch.Tensor) else np.asarray(out_gpu, np.float64)
    lg = to_np(lse_gpu) if isinstance(lse_gpu, torch.Tensor) else np.asarray(lse_gpu, np.float64)
    og = og.reshape(out_ref.shape)
    lg = lg.reshape(lse_ref.shape)
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lg), empty), f"{what}: -inf lse pattern differs"
    assert np.all(og[empty] == 0), f"{what}: rows without visible keys must be zero"
    assert np.all(np.isfinite(og)), f"{what}: non-finite outputs"
    denom = np.linalg.norm(out_ref)
    rel = np.linalg.norm(og - out_ref) / denom if denom > 0 else np.linalg.norm(og)
    mx = float(np.max(np.abs(og - out_ref))) if og.size else 0.0
    fin = ~empty
    lse_err = np.abs(lg[fin] - lse_ref[fin]) / np.maximum(1.0, np.abs(lse_ref[fin]))
    lmax = float(lse_err.max()) if lse_err.size else 0.0
    assert rel <= REL_L2, f"{what}: rel L2 {rel:.3e} > {REL_L2}"
    assert mx <= MAX_ABS, f"{what}: max abs {mx:.3e} > {MAX_ABS}"
    assert lmax <= LSE_REL, f"{what}: lse rel {lmax:.3e} > {LSE_REL}"
    return dict(rel_l2=float(rel), max_abs=mx, lse_rel=lmax)
