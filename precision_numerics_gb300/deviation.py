"""Numeric-deviation statistics of a result against a reference (NumPy).

Holds no attention arithmetic: it compares two arrays of the same shape and
reports max-abs, mean-abs, signed mean (rounding bias) and relative L2 error
-- the figures used to compare the tiled kernel and the naive BF16 attention
against the FP64 definition ("Is Flash Attention Stable?", abstract: numeric
deviation of Flash Attention versus Baseline Attention at BF16; "Why
Low-Precision Transformer Training Fails", Figure 6: signed error of O).
"""
from __future__ import annotations

import numpy as np


def deviation(x, ref) -> dict:
    """Error statistics of `x` against `ref` (both converted to FP64)."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if x.shape != ref.shape:
        raise ValueError(f"shape mismatch {x.shape} vs {ref.shape}")
    if x.size == 0:
        return {"max_abs": 0.0, "mean_abs": 0.0, "signed_mean": 0.0, "rel_l2": 0.0, "max_rel": 0.0}
    err = x - ref
    nref = float(np.linalg.norm(ref))
    aref = float(np.abs(ref).max())
    return {
        "max_abs": float(np.abs(err).max()),
        "mean_abs": float(np.abs(err).mean()),
        "signed_mean": float(err.mean()),
        "rel_l2": float(np.linalg.norm(err) / nref) if nref > 0 else float(np.linalg.norm(err)),
        "max_rel": float(np.abs(err).max() / aref) if aref > 0 else float(np.abs(err).max()),
    }
