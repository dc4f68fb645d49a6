"""Comparison of the CUDA path with the fp64 oracle.

The floating-point bar is the one the attention core is held to: max-abs
error <= 2e-2 and relative L2 error <= 1e-2 against the fp64 result.
"""
from __future__ import annotations

import numpy as np
import torch

MAX_ABS = 2e-2
REL_L2 = 1e-2


def to_f64(x) -> np.ndarray:
    if isinstance(x, torch.Tensor):
        return x.detach().float().cpu().numpy().astype(np.float64)
    return np.asarray(x, dtype=np.float64)


def check_close(got, want, what: str = "", max_abs: float = MAX_ABS, rel_l2: float = REL_L2):
    g, w = to_f64(got), to_f64(want)
    assert g.shape == w.shape, f"{what}: shape {g.shape} vs {w.shape}"
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    err = float(np.max(np.abs(g - w))) if g.size else 0.0
    rel = float(np.linalg.norm(g - w) / max(np.linalg.norm(w), 1e-30)) if g.size else 0.0
    assert err <= max_abs and rel <= rel_l2, f"{what}: max-abs {err:.3e}, rel-L2 {rel:.3e}"
    return err, rel


def bf16_ulp_diff(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    """Distance in bf16 units in the last place between two bit-pattern arrays."""
    def ordered(x):
        x = x.astype(np.int32)
        return np.where(x & 0x8000, 0x8000 - (x & 0x7FFF), 0x8000 + x)
    return np.abs(ordered(a_bits) - ordered(b_bits))


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp64 to bf16 (round to nearest even) directly, returning bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    f = x.astype(np.float32)  # exact enough: the two-step rounding is allowed 1 ulp in tests
    u = f.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)
