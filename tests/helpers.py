"""Shared helpers for the parity tests (test code only)."""
from __future__ import annotations

import json
import os

import numpy as np
import torch

# Tolerances of the parity bar: max |Δ| / max |ref| per (b, h) head.
TOL_F32 = 1e-4
TOL_BF16 = 2e-2


def head_rel_err(got, ref):
    """Per-head normwise error max|got − ref| / max|ref| over the trailing
    (n, d) or (d,) axes.  Returns an array over the leading head axes."""
    g = got.detach().double().cpu().numpy() if isinstance(got, torch.Tensor) else np.asarray(got)
    r = ref.detach().double().cpu().numpy() if isinstance(ref, torch.Tensor) else np.asarray(ref)
    assert g.shape == r.shape, (g.shape, r.shape)
    axes = tuple(range(2, r.ndim))
    num = np.abs(g - r).max(axis=axes)
    den = np.abs(r).max(axis=axes)
    den = np.where(den > 0, den, 1.0)
    return num / den


def log_parity(what, worst, tol, heads):
    """With LA_PARITY_LOG set, appends one JSON line per check: the worst
    head's error and its bar."""
    log = os.environ.get("LA_PARITY_LOG")
    if log:
        with open(log, "a") as f:
            f.write(json.dumps({"check": what, "worst_head_err": float(worst), "tol": tol,
                                "heads": int(heads)}) + "\n")


def assert_parity(got, ref, tol, what=""):
    err = head_rel_err(got, ref)
    worst = float(err.max()) if err.size else 0.0
    log_parity(what, worst, tol, err.size)
    assert np.all(np.isfinite(err)), f"{what}: non-finite error"
    assert worst <= tol, f"{what}: worst head error {worst:.3e} > {tol:.1e}"
    return worst


def to_cuda(inputs, device):
    return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in inputs.items()}
