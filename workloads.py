"""Seeded synthetic inputs for the Spark-X2.5 attention core.

This module serves both the fp64 oracle and the CUDA library (through the
tests and the benchmark).  It holds shapes, layer presets and random-number
recipes only: none of the method's arithmetic lives here.

Shapes and presets come from the Spark-X2.5 architecture page (4B / 1.7B):
§1 config table (H=16/8, Hkv=4/2, head_dim 256, window 512), §3 (fused
q_k_v_proj output width H*256 + 2*Hkv*256), §4 layered-RoPE table
(full_attention: theta 5e6, 64 rotated dims; sliding_attention: theta 1e4,
all 256 dims).  The pages publish no dataset or benchmark input for this path,
so every input is synthetic: normal bf16 activations and fp32 gate logits at
the pages' model shapes.

Recipe (all seeded):
  * CPU tensors: ``torch.Generator('cpu').manual_seed(seed)``, ``randn`` in
    fp32, times the stated standard deviation, then rounded to bf16 (RNE);
    qkv first, then gate logits, drawn in that order from one generator.
  * The 65,536-token case multiplies the K slice of qkv by 0.5 in fp32 before
    the bf16 rounding (exact, a power of two).
  * Decode caches above a few GB are filled on the GPU with a seeded CUDA
    generator in fixed chunks (one chunk per (b, kv-head) row block, in order).
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass

import torch

HEAD_DIM = 256

FULL = 0
SLIDING = 1


@dataclass(frozen=True)
class Layer:
    """Layer-type descriptor: mask kind, window, RoPE base and rotated dims."""
    kind: int
    window: int
    theta: float
    rot_dim: int
    gate_mode: int = 0  # 0 = sigmoid (the released checkpoints), 1 = silu


# Layered RoPE table (§4) and window (§1) of the Spark-X2.5 architecture page.
FULL_LAYER = Layer(kind=FULL, window=0, theta=5e6, rot_dim=64)
SLIDING_LAYER = Layer(kind=SLIDING, window=512, theta=1e4, rot_dim=256)

# layer_types of the 4B model: (sliding, sliding, sliding, full) x 9 (§1, §2).
LAYER_TYPES_4B = tuple(([SLIDING_LAYER] * 3 + [FULL_LAYER]) * 9)


@dataclass(frozen=True)
class PrefillCase:
    name: str
    B: int
    T: int
    H: int
    Hkv: int
    layer: Layer
    seed: int
    gate_std: float = 1.0
    k_scale: float = 1.0

    @property
    def width(self) -> int:
        return (self.H + 2 * self.Hkv) * HEAD_DIM


@dataclass(frozen=True)
class DecodeCase:
    name: str
    B: int
    H: int
    Hkv: int
    layer: Layer
    seed: int
    cap: int            # cache slots per (b, kv head): contiguous length or ring size
    len_lo: int         # cached tokens per sequence drawn uniformly in [len_lo, len_hi]
    len_hi: int
    gate_std: float = 1.0

    @property
    def width(self) -> int:
        return (self.H + 2 * self.Hkv) * HEAD_DIM


# The workloads the path is measured and checked on.
PREFILL_SLIDING_1P7B_T1024 = PrefillCase(
    "prefill_sliding_1.7b_T1024", B=1, T=1024, H=8, Hkv=2, layer=SLIDING_LAYER, seed=0)
PREFILL_FULL_4B_B2_T8192 = PrefillCase(
    "prefill_full_4b_B2_T8192", B=2, T=8192, H=16, Hkv=4, layer=FULL_LAYER, seed=1,
    gate_std=1.5)
PREFILL_FULL_4B_T65536 = PrefillCase(
    "prefill_full_4b_T65536", B=1, T=65536, H=16, Hkv=4, layer=FULL_LAYER, seed=2,
    k_scale=0.5)
PREFILL_SLIDING_4B_T65536 = PrefillCase(
    "prefill_sliding_4b_T65536", B=1, T=65536, H=16, Hkv=4, layer=SLIDING_LAYER, seed=2,
    k_scale=0.5)
DECODE_FULL_4B_B64 = DecodeCase(
    "decode_full_4b_B64", B=64, H=16, Hkv=4, layer=FULL_LAYER, seed=3,
    cap=131073, len_lo=4096, len_hi=131072)
DECODE_SLIDING_4B_B64 = DecodeCase(
    "decode_sliding_4b_B64", B=64, H=16, Hkv=4, layer=SLIDING_LAYER, seed=3,
    cap=512, len_lo=4096, len_hi=131072)
# 1M-token context: 1,048,575 cached tokens, new token at position 1,048,575.
DECODE_FULL_4B_1M = DecodeCase(
    "decode_full_4b_1M", B=1, H=16, Hkv=4, layer=FULL_LAYER, seed=4,
    cap=1048576, len_lo=1048575, len_hi=1048575)
DECODE_SLIDING_4B_1M = DecodeCase(
    "decode_sliding_4b_1M", B=1, H=16, Hkv=4, layer=SLIDING_LAYER, seed=4,
    cap=512, len_lo=1048575, len_hi=1048575)


def scaled(case, **changes):
    """A copy of a case with some fields replaced (smaller parity variants)."""
    return dataclasses.replace(case, **changes)


def make_prefill_inputs(case: PrefillCase, positions: torch.Tensor | None = None):
    """Seeded CPU inputs: qkv bf16 [B,T,W], gate fp32 [B,T,H], pos int32 [B,T]."""
    g = torch.Generator("cpu").manual_seed(case.seed)
    qkv = torch.randn((case.B, case.T, case.width), generator=g, dtype=torch.float32)
    if case.k_scale != 1.0:
        k0 = case.H * HEAD_DIM
        qkv[:, :, k0:k0 + case.Hkv * HEAD_DIM] *= case.k_scale
    qkv = qkv.to(torch.bfloat16)
    gate = torch.randn((case.B, case.T, case.H), generator=g, dtype=torch.float32)
    gate = gate * case.gate_std
    if positions is None:
        pos = torch.arange(case.T, dtype=torch.int32).repeat(case.B, 1)
    else:
        pos = positions.to(torch.int32).reshape(case.B, case.T).clone()
    return {"qkv": qkv, "gate": gate.contiguous(), "pos": pos.contiguous()}


def make_decode_lengths(case: DecodeCase) -> torch.Tensor:
    """Cached tokens per sequence (= position of the new token), int32 [B]."""
    g = torch.Generator("cpu").manual_seed(case.seed)
    return torch.randint(case.len_lo, case.len_hi + 1, (case.B,), generator=g,
                         dtype=torch.int64).to(torch.int32)


def make_decode_step_inputs(case: DecodeCase):
    """Seeded CPU inputs of the new token: qkv bf16 [B,W], gate fp32 [B,H], pos [B]."""
    pos = make_decode_lengths(case)
    g = torch.Generator("cpu").manual_seed(case.seed + 1000)
    qkv = torch.randn((case.B, case.width), generator=g, dtype=torch.float32)
    qkv = qkv.to(torch.bfloat16)
    gate = torch.randn((case.B, case.H), generator=g, dtype=torch.float32) * case.gate_std
    return {"qkv": qkv, "gate": gate.contiguous(), "pos": pos}


def fill_cache_(cache: torch.Tensor, seed: int) -> torch.Tensor:
    """Fill a [B, Hkv, cap, 256] bf16 cache with N(0,1), seeded, chunk by chunk.

    Works on CPU or CUDA tensors; the chunk order is fixed (one (b, kv head)
    block after the other) so the content depends only on the seed and device.
    """
    B, Hkv, cap, D = cache.shape
    g = torch.Generator(cache.device).manual_seed(seed)
    for b in range(B):
        for h in range(Hkv):
            blk = torch.randn((cap, D), generator=g, device=cache.device,
                              dtype=torch.float32)
            cache[b, h].copy_(blk.to(torch.bfloat16))
    return cache


def bf16_bits(t: torch.Tensor):
    """Raw 16-bit patterns of a bf16 tensor as a numpy uint16 array (host copy)."""
    import numpy as np
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
