"""Pins of the fp64 oracle: checks against what the pages and mathematics fix.

Each ``pin_*`` takes an ``oracle.OracleLib`` and raises AssertionError when the
oracle disagrees.  ``test_oracle.py`` runs them on the real oracle and on
copies of the oracle with a planted mistake (each planted mistake must be
caught by at least one pin).

Sources (page title, section):
  * Spark-X2.5 architecture (4B / 1.7B): §2 masks (causal / sliding window 512),
    §3 Eq. 1 (softmax(QK^T/sqrt(d)) V times the per-head sigmoid gate), §4
    layered-RoPE table (theta 5e6 with 64 rotated dims; theta 1e4 with 256).
  * MiniMax-M2 chapter §13.3 of the translated LLM-architecture notes: partial
    RoPE rotates the first rotary_dim channels and leaves the others as-is.
  * Spark-X2.5-4B hybrid-attention explainer (lshu.cn): sliding layers keep
    only the latest 512 tokens in their KV cache.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import brute

D = 256
FULL, SLIDING = 0, 1


def bf16_inputs(seed: int, shape, scale: float = 1.0):
    """Random bf16 tensor: returns (bits uint16, exact fp64 values)."""
    g = torch.Generator("cpu").manual_seed(seed)
    t = (torch.randn(shape, generator=g) * scale).to(torch.bfloat16)
    bits = t.view(torch.int16).numpy().view(np.uint16).copy()
    return bits, t.to(torch.float64).numpy()


def to_bits(x64: np.ndarray) -> np.ndarray:
    """fp64 values already representable in bf16 -> uint16 patterns."""
    t = torch.from_numpy(np.ascontiguousarray(x64)).to(torch.bfloat16)
    assert np.array_equal(t.to(torch.float64).numpy(), x64), "not bf16-exact"
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def round_bits(x64: np.ndarray):
    """Round fp64 to bf16 (RNE): (bits, exact fp64 of the rounded values)."""
    t = torch.from_numpy(np.ascontiguousarray(x64)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy(), t.to(torch.float64).numpy()


def gates(seed: int, shape, std=1.0):
    g = torch.Generator("cpu").manual_seed(seed)
    return (torch.randn(shape, generator=g) * std).numpy().astype(np.float32)


# --------------------------------------------------------------------------
# brute force on tiny inputs

BRUTE_CASES = [
    # kind, window, rot_dim, theta, H, Hkv, B, T, positions
    (FULL, 0, 64, 5e6, 4, 1, 1, 8, "arange"),
    (SLIDING, 3, 256, 1e4, 4, 2, 2, 8, "random"),
    (SLIDING, 1, 256, 1e4, 2, 2, 1, 5, "offset"),
    (FULL, 0, 0, 1e4, 8, 2, 1, 7, "arange"),
    (SLIDING, 8, 64, 5e6, 4, 4, 1, 8, "random"),
    (FULL, 0, 128, 1e4, 16, 4, 1, 3, "random"),
    (SLIDING, 2, 256, 1e4, 8, 2, 2, 6, "offset"),
]


def _positions(kind: str, B: int, T: int, seed: int):
    if kind == "arange":
        return np.tile(np.arange(T, dtype=np.int32), (B, 1))
    if kind == "offset":
        return np.tile(np.arange(T, dtype=np.int32) + 1000, (B, 1))
    rng = np.random.default_rng(seed)
    return rng.integers(0, 1 << 20, size=(B, T)).astype(np.int32)


def pin_brute_force(orc):
    # fp64 angles near 1e6 rad carry ~1e-10 rad of rounding, hence 1e-9.
    for n, (kind, W, r, theta, H, Hkv, B, T, pk) in enumerate(BRUTE_CASES):
        bits, x = bf16_inputs(100 + n, (B, T, (H + 2 * Hkv) * D))
        g = gates(200 + n, (B, T, H))
        pos = _positions(pk, B, T, 300 + n)
        got = orc.prefill(bits, g, pos, kind, W, theta, r, H, Hkv)
        want = brute.prefill(x, g.astype(np.float64), pos, kind, W, theta, r, H, Hkv)
        err = np.max(np.abs(got - want))
        assert err < 1e-9, f"brute case {n}: max abs diff {err}"


def pin_decode_brute_force(orc):
    """Decode with rotation, ragged positions and a ring, against brute force."""
    for n, (kind, W, r, theta, cap, posl) in enumerate([
            (FULL, 0, 64, 5e6, 40, [0, 5, 39]),
            (SLIDING, 6, 256, 1e4, 6, [0, 3, 5, 6, 13, 1048575]),
            (SLIDING, 5, 256, 1e4, 9, [4, 9, 10, 23])]):
        H, Hkv = 4, 2
        B = len(posl)
        pos = np.array(posl, np.int32)
        bits, x = bf16_inputs(400 + n, (B, (H + 2 * Hkv) * D))
        kb, kx = bf16_inputs(500 + n, (B, Hkv, cap, D))
        vb, vx = bf16_inputs(600 + n, (B, Hkv, cap, D))
        g = gates(700 + n, (B, H))
        got, _, _ = orc.decode(bits, g, pos, kb, vb, kind, W, theta, r, H, Hkv)
        want = brute.decode(x, g.astype(np.float64), pos, kx, vx, kind, W, theta, r, H, Hkv)
        err = np.max(np.abs(got - want))
        assert err < 1e-9, f"decode brute case {n}: max abs diff {err}"


# --------------------------------------------------------------------------
# special cases with closed forms


def pin_window_ge_T_is_full(orc):
    """A window at least T wide masks nothing the causal mask keeps."""
    H, Hkv, B, T = 4, 2, 1, 12
    bits, _ = bf16_inputs(11, (B, T, (H + 2 * Hkv) * D))
    g = gates(12, (B, T, H))
    pos = _positions("random", B, T, 13)
    full = orc.prefill(bits, g, pos, FULL, 0, 1e4, 256, H, Hkv)
    for W in (T, T + 5, 1 << 20):
        sl = orc.prefill(bits, g, pos, SLIDING, W, 1e4, 256, H, Hkv)
        assert np.array_equal(sl, full), f"window {W} differs from causal"
    sl = orc.prefill(bits, g, pos, SLIDING, T - 1, 1e4, 256, H, Hkv)
    assert not np.array_equal(sl[:, -1], full[:, -1]), "window T-1 must drop a key"


def pin_window_one_is_gated_self_value(orc):
    """Window 1: each query sees only itself, so out = sigmoid(g) * v_self."""
    H, Hkv, B, T = 4, 2, 2, 9
    G = H // Hkv
    bits, x = bf16_inputs(21, (B, T, (H + 2 * Hkv) * D))
    g = gates(22, (B, T, H))
    pos = _positions("random", B, T, 23)
    out = orc.prefill(bits, g, pos, SLIDING, 1, 1e4, 256, H, Hkv).reshape(B, T, H, D)
    v = x[:, :, (H + Hkv) * D:].reshape(B, T, Hkv, D)
    for h in range(H):
        want = v[:, :, h // G, :] / (1.0 + np.exp(-g[:, :, h].astype(np.float64)))[..., None]
        assert np.allclose(out[:, :, h, :], want, rtol=1e-14, atol=0), f"head {h}"


def pin_layout_identity(orc):
    """No rotation, window 1, gate +40 (sigmoid == 1.0 in fp64): out is exactly
    the bf16 V slice of the head's KV group, head h at columns [h*256,(h+1)*256).
    Pins the Q||K||V split, the head-to-group map and the output layout."""
    for H, Hkv in ((4, 2), (8, 2), (4, 4), (6, 3)):
        G = H // Hkv
        B, T = 2, 5
        bits, x = bf16_inputs(31 + H, (B, T, (H + 2 * Hkv) * D))
        g = np.full((B, T, H), 40.0, np.float32)
        pos = _positions("arange", B, T, 0)
        out = orc.prefill(bits, g, pos, SLIDING, 1, 1e4, 0, H, Hkv)
        for h in range(H):
            gk = h // G
            v = x[:, :, (H + Hkv + gk) * D:(H + Hkv + gk + 1) * D]
            assert np.array_equal(out[:, :, h * D:(h + 1) * D], v), f"H={H} head {h}"


def pin_gate_zero_halves(orc):
    """sigmoid(0) = 1/2 exactly, so gate 0 gives half of the ungated output."""
    H, Hkv, B, T = 4, 1, 1, 10
    bits, _ = bf16_inputs(41, (B, T, (H + 2 * Hkv) * D))
    pos = _positions("arange", B, T, 0)
    ungated = orc.prefill(bits, np.full((B, T, H), 40.0, np.float32), pos, FULL, 0,
                          5e6, 64, H, Hkv)
    half = orc.prefill(bits, np.zeros((B, T, H), np.float32), pos, FULL, 0, 5e6, 64,
                       H, Hkv)
    assert np.array_equal(half, 0.5 * ungated)


def pin_zero_query_mean_of_window(orc):
    """Q = 0 makes every visible score 0, so the output is sigmoid(g) times the
    plain mean of the visible values.  With v_j[0] = j and v_j[1] = 1 the mean
    index of the band is (lo + i)/2 with lo = max(0, i - W + 1) (sliding) or 0
    (causal): this pins the band edges exactly."""
    H, Hkv, B, T = 2, 1, 1, 40
    qkv = np.zeros((B, T, (H + 2 * Hkv) * D))
    rng = np.random.default_rng(5)
    qkv[:, :, H * D:(H + Hkv) * D] = to_bits_exact(rng.standard_normal((B, T, Hkv * D)))
    vbase = (H + Hkv) * D
    qkv[0, :, vbase + 0] = np.arange(T)
    qkv[0, :, vbase + 1] = 1.0
    bits = to_bits(qkv)
    g = gates(51, (B, T, H))
    pos = _positions("random", B, T, 52)
    for kind, W in ((FULL, 0), (SLIDING, 7), (SLIDING, 1), (SLIDING, 39)):
        out = orc.prefill(bits, g, pos, kind, W, 1e4, 256, H, Hkv).reshape(B, T, H, D)
        for i in range(T):
            lo = max(0, i - W + 1) if kind == SLIDING else 0
            for h in range(H):
                s = 1.0 / (1.0 + math.exp(-float(g[0, i, h])))
                assert abs(out[0, i, h, 0] - s * (lo + i) / 2.0) < 1e-12, (kind, W, i)
                assert abs(out[0, i, h, 1] - s) < 1e-14, (kind, W, i)


def to_bits_exact(x):
    """Round fp64 to bf16 and return the exact fp64 of the rounded values."""
    return round_bits(x)[1]


def pin_gqa_group_map(orc):
    """Q = 0 and V of KV head g equal to g+1 everywhere: head h must output
    sigmoid(gate) * (floor(h / G) + 1)."""
    for H, Hkv in ((8, 2), (8, 4), (16, 4), (4, 1)):
        G = H // Hkv
        B, T = 1, 6
        qkv = np.zeros((B, T, (H + 2 * Hkv) * D))
        for gk in range(Hkv):
            qkv[:, :, (H + Hkv + gk) * D:(H + Hkv + gk + 1) * D] = gk + 1
        bits = to_bits(qkv)
        g = gates(61 + H, (B, T, H))
        pos = _positions("arange", B, T, 0)
        out = orc.prefill(bits, g, pos, FULL, 0, 5e6, 64, H, Hkv).reshape(B, T, H, D)
        for h in range(H):
            s = 1.0 / (1.0 + np.exp(-g[0, :, h].astype(np.float64)))
            want = s[:, None] * (h // G + 1)
            assert np.allclose(out[0, :, h, :], want, rtol=1e-14, atol=0), (H, Hkv, h)


# --------------------------------------------------------------------------
# RoPE


def pin_rope_partial_passthrough(orc):
    """Dims at or above rot_dim leave RoPE bit-identical (partial RoPE)."""
    _, x = bf16_inputs(71, (50, D))
    pos = np.random.default_rng(1).integers(0, 1 << 20, 50).astype(np.int32)
    for r in (0, 2, 64, 128):
        y = orc.rope(x, pos, r, 5e6)
        assert np.array_equal(y[:, r:], x[:, r:]), f"rot_dim {r}"


def pin_rope_pair_norm(orc):
    """Each rotated pair (k, k + r/2) keeps its Euclidean norm."""
    _, x = bf16_inputs(72, (50, D))
    pos = np.random.default_rng(2).integers(0, 1 << 20, 50).astype(np.int32)
    for r, theta in ((64, 5e6), (256, 1e4)):
        y = orc.rope(x, pos, r, theta)
        h = r // 2
        nx = np.hypot(x[:, :h], x[:, h:r])
        ny = np.hypot(y[:, :h], y[:, h:r])
        assert np.allclose(nx, ny, rtol=1e-13, atol=1e-14)


def pin_rope_position_zero_identity(orc):
    _, x = bf16_inputs(73, (20, D))
    y = orc.rope(x, np.zeros(20, np.int32), 256, 1e4)
    assert np.array_equal(x, y)


def pin_rope_relative_position(orc):
    """<R(p+d) q, R(p'+d) k> = <R(p) q, R(p') k>: scores depend on p - p' only."""
    _, q = bf16_inputs(74, (30, D))
    _, k = bf16_inputs(75, (30, D))
    rng = np.random.default_rng(3)
    p1 = rng.integers(0, 500000, 30).astype(np.int32)
    p2 = rng.integers(0, 500000, 30).astype(np.int32)
    dl = rng.integers(0, 500000, 30).astype(np.int32)
    for r, theta in ((64, 5e6), (256, 1e4)):
        a = np.sum(orc.rope(q, p1, r, theta) * orc.rope(k, p2, r, theta), axis=1)
        b = np.sum(orc.rope(q, p1 + dl, r, theta) * orc.rope(k, p2 + dl, r, theta), axis=1)
        assert np.allclose(a, b, rtol=0, atol=1e-8)


def pin_rope_basis_closed_form(orc):
    """Rotating unit vectors gives the rotate_half closed form:
    e_k -> cos(a) e_k + sin(a) e_{k+r/2};  e_{k+r/2} -> -sin(a) e_k + cos(a) e_{k+r/2},
    a = pos * theta^(-2k/r), with r the rotated width (not the head width)."""
    for r, theta in ((64, 5e6), (256, 1e4), (32, 10.0)):
        h = r // 2
        for k in (0, 1, h // 2, h - 1):
            for p in (1, 7, 1048575):
                a = p * math.exp(-(2.0 * k / r) * math.log(theta))
                e1 = np.zeros((1, D)); e1[0, k] = 1.0
                e2 = np.zeros((1, D)); e2[0, k + h] = 1.0
                y1 = orc.rope(e1, np.array([p], np.int32), r, theta)[0]
                y2 = orc.rope(e2, np.array([p], np.int32), r, theta)[0]
                tol = 1e-9
                assert abs(y1[k] - math.cos(a)) < tol and abs(y1[k + h] - math.sin(a)) < tol, \
                    (r, k, p)
                assert abs(y2[k] + math.sin(a)) < tol and abs(y2[k + h] - math.cos(a)) < tol, \
                    (r, k, p)
                others = np.delete(y1, [k, k + h])
                assert not np.any(others), (r, k, p)


# --------------------------------------------------------------------------
# decode


def pin_decode_equals_prefill_last_row(orc):
    """Without rotation the cache holds the raw keys, so a decode step at
    position T-1 over a cache of tokens 0..T-2 equals prefill row T-1."""
    H, Hkv, B, T = 4, 2, 2, 11
    bits, _ = bf16_inputs(81, (B, T, (H + 2 * Hkv) * D))
    g = gates(82, (B, T, H))
    pos = _positions("arange", B, T, 0)
    for kind, W, cap in ((FULL, 0, T + 3), (SLIDING, 4, 4), (SLIDING, 4, 7)):
        pre = orc.prefill(bits, g, pos, kind, W, 1e4, 0, H, Hkv)
        kc = np.zeros((B, Hkv, cap, D), np.uint16)
        vc = np.zeros((B, Hkv, cap, D), np.uint16)
        kc[...] = 0x4480  # 1024.0: poison in slots the step must not read
        vc[...] = 0x4480
        for t in range(T - 1):
            slot = t % cap if kind == SLIDING else t
            if kind == SLIDING and t < T - 1 - cap:
                continue
            for gk in range(Hkv):
                kc[:, gk, slot] = bits[:, t, (H + gk) * D:(H + gk + 1) * D]
                vc[:, gk, slot] = bits[:, t, (H + Hkv + gk) * D:(H + Hkv + gk + 1) * D]
        out, _, _ = orc.decode(bits[:, T - 1], g[:, T - 1], pos[:, T - 1], kc, vc, kind, W,
                               1e4, 0, H, Hkv)
        assert np.allclose(out, pre[:, T - 1], rtol=0, atol=1e-13), (kind, W, cap)


def pin_decode_ring_wrap(orc):
    """The 512-slot ring at the wrap points: decode equals the prefill row of
    the same token with the 512 window (no rotation, so cached keys are raw)."""
    H, Hkv, B = 2, 1, 1
    W = 512
    for p in (0, 1, 511, 512, 513, 1023, 1024):
        T = p + 1
        bits, _ = bf16_inputs(90 + p, (B, T, (H + 2 * Hkv) * D))
        g = gates(91, (B, T, H))
        pos = _positions("arange", B, T, 0)
        want = orc.prefill(bits, g, pos, SLIDING, W, 1e4, 0, H, Hkv,
                           rows=np.array([p], np.int64))
        kc = np.full((B, Hkv, W, D), 0x4480, np.uint16)
        vc = np.full((B, Hkv, W, D), 0x4480, np.uint16)
        for t in range(max(0, p - W), p):
            kc[0, 0, t % W] = bits[0, t, H * D:(H + 1) * D]
            vc[0, 0, t % W] = bits[0, t, (H + 1) * D:(H + 2) * D]
        out, _, _ = orc.decode(bits[:, p], g[:, p], pos[:, p], kc, vc, SLIDING, W, 1e4, 0,
                               H, Hkv)
        assert np.allclose(out, want, rtol=0, atol=1e-13), p


def pin_decode_new_entries(orc):
    """The step stores RoPE(k_new, pos) and v_new at the slot of pos."""
    H, Hkv, B = 4, 2, 3
    bits, x = bf16_inputs(95, (B, (H + 2 * Hkv) * D))
    kb, _ = bf16_inputs(96, (B, Hkv, 16, D))
    g = gates(97, (B, H))
    pos = np.array([0, 9, 15], np.int32)
    _, kn, vn = orc.decode(bits, g, pos, kb, kb, FULL, 0, 5e6, 64, H, Hkv)
    k = x[:, H * D:(H + Hkv) * D].reshape(B, Hkv, D)
    v = x[:, (H + Hkv) * D:].reshape(B, Hkv, D)
    want = brute.rope_complex(k, pos[:, None], 64, 5e6)
    assert np.allclose(kn, want, rtol=0, atol=1e-12)
    assert np.array_equal(vn, v)


def pin_silu_gate(orc):
    """The silu gate (gate_attn_act_mode, §3): brute force agrees, a zero logit
    gives exactly zero, and a logit of 40 (sigmoid == 1 in fp64) gives 40x the
    ungated output."""
    H, Hkv, B, T = 4, 2, 2, 7
    bits, x = bf16_inputs(111, (B, T, (H + 2 * Hkv) * D))
    g = gates(112, (B, T, H), std=2.0)
    pos = _positions("random", B, T, 113)
    got = orc.prefill(bits, g, pos, SLIDING, 3, 1e4, 256, H, Hkv, gate_mode=1)
    want = brute.prefill(x, g.astype(np.float64), pos, SLIDING, 3, 1e4, 256, H, Hkv, gate_mode=1)
    assert np.max(np.abs(got - want)) < 1e-9
    zero = orc.prefill(bits, np.zeros_like(g), pos, FULL, 0, 5e6, 64, H, Hkv, gate_mode=1)
    assert not np.any(zero)
    big = orc.prefill(bits, np.full_like(g, 40.0), pos, FULL, 0, 5e6, 64, H, Hkv, gate_mode=1)
    ungated = orc.prefill(bits, np.full_like(g, 40.0), pos, FULL, 0, 5e6, 64, H, Hkv)
    assert np.allclose(big, 40.0 * ungated, rtol=1e-15, atol=0)
    kb, kx = bf16_inputs(114, (B, Hkv, 9, D))
    dpos = np.array([8, 3], np.int32)
    dg = gates(115, (B, H), std=2.0)
    got, _, _ = orc.decode(bits[:, 0], dg, dpos, kb, kb, FULL, 0, 5e6, 64, H, Hkv, gate_mode=1)
    want = brute.decode(x[:, 0], dg.astype(np.float64), dpos, kx, kx, FULL, 0, 5e6, 64, H, Hkv,
                        gate_mode=1)
    assert np.max(np.abs(got - want)) < 1e-9


ALL_PINS = [
    pin_brute_force,
    pin_decode_brute_force,
    pin_window_ge_T_is_full,
    pin_window_one_is_gated_self_value,
    pin_layout_identity,
    pin_gate_zero_halves,
    pin_zero_query_mean_of_window,
    pin_gqa_group_map,
    pin_rope_partial_passthrough,
    pin_rope_pair_norm,
    pin_rope_position_zero_identity,
    pin_rope_relative_position,
    pin_rope_basis_closed_form,
    pin_decode_equals_prefill_last_row,
    pin_decode_ring_wrap,
    pin_decode_new_entries,
    pin_silu_gate,
]
