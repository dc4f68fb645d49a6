"""Comparison of the CUDA path with the fp64 oracle.

The floating-point bar is the one the attention core is held to: max-abs
error <= 2e-2 and relative L2 error <= 1e-2 against the fp64 result.

With the silu output gate (gate_attn_act_mode = silu, Spark-X2.5 architecture
§3) a head's output is the attention result times silu(g) = g * sigmoid(g),
which exceeds 1 for logits above ~1.28.  The output is a bf16 tensor, and
its final rounding alone errs by up to 2^-9 of the value: above |out| ~ 10
that is more than 2e-2, whatever the kernel does.  So for the silu gate the
max-abs bar is applied per unit of gate factor, |got - want| <= 2e-2 *
max(1, |silu(g)|) element by element, while the relative-L2 bar (which does
not depend on scale) is applied to the raw outputs.  Under the sigmoid gate
the factor is below 1 and this is exactly the plain bar.
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


def check_close(got, want, what: str = "", max_abs: float = MAX_ABS, rel_l2: float = REL_L2,
                unit=None):
    """Asserts the bar; returns (max-abs, rel-L2).  `unit` (broadcastable to
    the outputs, >= 1) is the gate factor of the silu gate: the max-abs bar
    then holds for (got - want) / unit, the relative-L2 bar for the raw
    outputs, and the returned max-abs is the scaled one."""
    g, w = to_f64(got), to_f64(want)
    assert g.shape == w.shape, f"{what}: shape {g.shape} vs {w.shape}"
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    diff = g - w
    if unit is not None:
        u = np.broadcast_to(np.asarray(unit, np.float64), diff.shape)
        assert np.all(u >= 1.0), f"{what}: gate unit below 1"
        diff_scaled = diff / u
    else:
        diff_scaled = diff
    err = float(np.max(np.abs(diff_scaled))) if g.size else 0.0
    rel = float(np.linalg.norm(diff) / max(np.linalg.norm(w), 1e-30)) if g.size else 0.0
    assert err <= max_abs and rel <= rel_l2, f"{what}: max-abs {err:.3e}, rel-L2 {rel:.3e}"
    return err, rel


def silu_gate_unit(gate, head_dim: int = 256) -> np.ndarray:
    """max(1, |silu(g)|) per output element for gate logits [..., H]: the
    factor by which the silu gate scales a head's output (and the bf16
    rounding error of that output), repeated over the head's dims."""
    g = to_f64(gate)
    act = np.abs(g / (1.0 + np.exp(-g)))
    return np.repeat(np.maximum(1.0, act), head_dim, axis=-1)


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


def bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> exact fp64 values."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def check_rotated_bf16(got_bits: np.ndarray, exact: np.ndarray, x_scale, what: str = ""):
    """A RoPE output stored as bf16 against the exact fp64 rotation.

    The GPU rotates in fp32 with angles good to ~2e-7 rad, then rounds to
    bf16.  Where the two terms of a rotation nearly cancel the result is tiny
    and those fp32 errors, small against the inputs, exceed one bf16 ulp of
    the result; so the bound is one bf16 ulp of the value (2^-8 relative) plus
    2e-6 of the input magnitude x_scale (per row, broadcastable)."""
    got = bits_to_f64(got_bits)
    bound = np.abs(exact) * 2.0 ** -8 + 2e-6 * np.asarray(x_scale, dtype=np.float64)
    bad = np.abs(got - exact) > bound
    assert not np.any(bad), f"{what}: {int(bad.sum())} rotated values off (first at {np.argwhere(bad)[0]})"
