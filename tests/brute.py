"""Brute-force restatement of the attention core for tiny inputs (T <= 8).

Written independently of the C oracle, through different routes, so that a
mistake in one is unlikely to be repeated in the other:
  * RoPE as complex multiplication: the pair (x_k, x_{k+r/2}) is the complex
    number x_k + i x_{k+r/2}, multiplied by exp(i * pos * theta^(-2k/r));
    this is the rotate_half convention of the layered-RoPE section (§4) of the
    Spark-X2.5 architecture page, partial RoPE as the MiniMax-M2 chapter §13.3
    of the translated architecture notes defines it (first r dims rotated).
  * the mask as an explicit boolean matrix; softmax and sigmoid from scipy;
  * attention as dense matrix products (Eq. 1 of §3 of the same page).
"""
from __future__ import annotations

import numpy as np
from scipy.special import expit, softmax

D = 256


def rope_complex(x: np.ndarray, pos: np.ndarray, rot_dim: int, theta: float):
    """x [..., 256] fp64, pos broadcastable to x[..., 0]."""
    if rot_dim == 0:
        return x.copy()
    half = rot_dim // 2
    z = x[..., :half] + 1j * x[..., half:rot_dim]
    k = np.arange(half, dtype=np.float64)
    freq = np.power(float(theta), -2.0 * k / rot_dim)
    z = z * np.exp(1j * np.asarray(pos, np.float64)[..., None] * freq)
    return np.concatenate([z.real, z.imag, x[..., rot_dim:]], axis=-1)


def visible(kind: int, window: int, T: int) -> np.ndarray:
    """Boolean [T, T]: True where query i may attend key j."""
    i = np.arange(T)[:, None]
    j = np.arange(T)[None, :]
    m = j <= i
    if kind == 1:
        m &= (i - j) < window
    return m


def gate_activation(g, gate_mode: int):
    """sigmoid (mode 0) or silu = g * sigmoid(g) (mode 1), from scipy's expit."""
    return expit(g) if gate_mode == 0 else g * expit(g)


def prefill(qkv: np.ndarray, gate: np.ndarray, pos: np.ndarray, kind: int,
            window: int, theta: float, rot_dim: int, H: int, Hkv: int, gate_mode: int = 0):
    """qkv fp64 [B,T,(H+2Hkv)*256], gate [B,T,H], pos [B,T] -> fp64 [B,T,H*256]."""
    B, T, _ = qkv.shape
    G = H // Hkv
    q = qkv[:, :, :H * D].reshape(B, T, H, D)
    k = qkv[:, :, H * D:(H + Hkv) * D].reshape(B, T, Hkv, D)
    v = qkv[:, :, (H + Hkv) * D:].reshape(B, T, Hkv, D)
    q = rope_complex(q, pos[:, :, None], rot_dim, theta)
    k = rope_complex(k, pos[:, :, None], rot_dim, theta)
    mask = visible(kind, window, T)
    out = np.zeros((B, T, H, D))
    for b in range(B):
        for h in range(H):
            g = h // G
            s = q[b, :, h, :] @ k[b, :, g, :].T / np.sqrt(D)
            s = np.where(mask, s, -np.inf)
            p = softmax(s, axis=-1)
            out[b, :, h, :] = (p @ v[b, :, g, :]) * gate_activation(gate[b, :, h], gate_mode)[:, None]
    return out.reshape(B, T, H * D)


def decode(qkv: np.ndarray, gate: np.ndarray, pos: np.ndarray, k_cache: np.ndarray,
           v_cache: np.ndarray, kind: int, window: int, theta: float, rot_dim: int,
           H: int, Hkv: int, gate_mode: int = 0):
    """One decode step by brute force.

    qkv fp64 [B,(H+2Hkv)*256]; gate [B,H]; pos [B]; caches fp64 [B,Hkv,cap,256]
    (post-RoPE keys).  Token j lives at slot j (full) or j mod cap (ring).
    Returns fp64 [B, H*256].
    """
    B = qkv.shape[0]
    cap = k_cache.shape[2]
    G = H // Hkv
    out = np.zeros((B, H, D))
    for b in range(B):
        p = int(pos[b])
        toks = np.arange(0, p + 1)
        if kind == 1:
            toks = toks[p - toks < window]
        q = rope_complex(qkv[b, :H * D].reshape(H, D), np.full(H, p), rot_dim, theta)
        kn = rope_complex(qkv[b, H * D:(H + Hkv) * D].reshape(Hkv, D), np.full(Hkv, p),
                          rot_dim, theta)
        vn = qkv[b, (H + Hkv) * D:].reshape(Hkv, D)
        for h in range(H):
            g = h // G
            keys = np.stack([kn[g] if t == p else k_cache[b, g, t % cap if kind == 1 else t]
                             for t in toks])
            vals = np.stack([vn[g] if t == p else v_cache[b, g, t % cap if kind == 1 else t]
                             for t in toks])
            w = softmax(keys @ q[h] / np.sqrt(D))
            out[b, h] = (w @ vals) * gate_activation(gate[b, h], gate_mode)
    return out.reshape(B, H * D)
