"""GPU checks against closed forms of the attention core (through the C ABI).

Each case has an answer that follows from the mathematics alone, with no
oracle run (Spark-X2.5 architecture page: §3 Eq. 1 for the gated softmax
attention, §2 for the masks, §4 for RoPE):

- Zero queries score every key 0, so softmax weighs the visible keys equally
  and each output row is sigmoid(g) times the mean of its visible values.  With
  values that are small integers the sums are exact in fp32, so the result is
  the fp64 mean to within one bf16 rounding: the mask's visible set and the
  softmax normalisation are pinned together.
- RoPE at position 0 is the identity (cos 0 = 1, sin 0 = 0), so a cache filled
  at position 0 holds the input keys bit for bit.
- RoPE makes a score depend only on the difference of the two positions, so
  shifting every position by the same amount leaves the attention unchanged
  (up to the rounding of the rotated bf16 operands).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import full_gqa_attention_gb300 as fga
import oracle
import workloads as wl
from parity import check_close

pytestmark = pytest.mark.gpu

FULL, SLIDING = wl.FULL, wl.SLIDING


@pytest.mark.parametrize("kind,W,H,Hkv", [(FULL, 0, 8, 2), (SLIDING, 512, 8, 2),
                                          (SLIDING, 100, 16, 4), (FULL, 0, 8, 8)])
def test_zero_queries_average_the_visible_values(cuda, kind, W, H, Hkv):
    T = 700
    g = torch.Generator().manual_seed(21 + W + H)
    qkv = torch.zeros((1, T, (H + 2 * Hkv) * 256), dtype=torch.float32)
    qkv[0, :, H * 256:(H + Hkv) * 256] = torch.randn((T, Hkv * 256), generator=g)  # any keys
    j = torch.arange(T)
    for gi in range(Hkv):
        v0 = (H + Hkv + gi) * 256
        qkv[0, :, v0] = (j & 63).float()
        qkv[0, :, v0 + 1] = (j >> 6).float()
        qkv[0, :, v0 + 2] = 1.0
        qkv[0, :, v0 + 3] = ((j * (gi + 3)) % 17).float()
    gate = torch.full((1, T, H), 40.0)          # sigmoid(40) == 1.0 in fp32
    pos = torch.arange(T, dtype=torch.int32)[None]
    layer = wl.Layer(kind=kind, window=max(W, 1), theta=1e4, rot_dim=256 if kind else 64)
    out = fga.spark_attn_prefill(qkv.to(torch.bfloat16).to(cuda), gate.to(cuda), pos.to(cuda),
                                 layer)
    got = out.float().cpu().reshape(T, H, 256)[:, :, :4].double().numpy()
    want = np.zeros((T, Hkv, 4))
    for i in range(T):
        lo = max(0, i - W + 1) if kind == SLIDING else 0
        vis = np.arange(lo, i + 1)
        for gi in range(Hkv):
            want[i, gi] = [np.mean(vis & 63), np.mean(vis >> 6), 1.0,
                           np.mean((vis * (gi + 3)) % 17)]
    want = np.repeat(want, H // Hkv, axis=1)    # head h reads KV head h // G
    # one bf16 rounding (at most 2^-8 relative) of an fp32 value a few fp32 ulps
    # (2^-22 relative) from the mean
    tol = (2.0 ** -8 + 2.0 ** -20) * np.abs(want) + 1e-7
    assert np.all(np.abs(got - want) <= tol), np.abs(got - want).max()
    # the other dims of V are 0, so are the outputs there
    assert float(out.float().reshape(T, H, 256)[:, :, 4:].abs().max()) == 0.0


@pytest.mark.parametrize("layer", [wl.FULL_LAYER, wl.SLIDING_LAYER], ids=["full", "sliding"])
def test_position_zero_rotation_is_the_identity(cuda, layer):
    H, Hkv, T = 16, 4, 300
    x = wl.make_prefill_inputs(wl.PrefillCase("p0", B=1, T=T, H=H, Hkv=Hkv, layer=layer, seed=4),
                               positions=torch.zeros(T, dtype=torch.int32))
    cap = T if layer.kind == FULL else 512
    kc = torch.full((1, Hkv, cap, 256), 7.0, dtype=torch.bfloat16, device=cuda)
    vc = torch.full_like(kc, 7.0)
    fga.spark_attn_prefill_cache(x["qkv"].to(cuda), x["gate"].to(cuda), x["pos"].to(cuda), kc, vc,
                                 layer)
    torch.cuda.synchronize()
    k_in = x["qkv"][0, :, H * 256:(H + Hkv) * 256].reshape(T, Hkv, 256).permute(1, 0, 2)
    assert torch.equal(kc[0, :, :T].cpu(), k_in)


@pytest.mark.parametrize("layer", [wl.FULL_LAYER, wl.SLIDING_LAYER], ids=["full", "sliding"])
def test_shifted_positions_give_the_same_attention(cuda, layer):
    H, Hkv, T, shift = 8, 2, 600, 123_457
    case = wl.PrefillCase("sh", B=1, T=T, H=H, Hkv=Hkv, layer=layer, seed=6)
    base = wl.make_prefill_inputs(case)
    moved = wl.make_prefill_inputs(case, positions=torch.arange(T, dtype=torch.int32) + shift)
    outs = [fga.spark_attn_prefill(x["qkv"].to(cuda), x["gate"].to(cuda), x["pos"].to(cuda),
                                   layer).reshape(T, -1) for x in (base, moved)]
    # the same attention in exact arithmetic (the oracle's fp64 at the original positions)
    want = oracle.prefill(wl.bf16_bits(base["qkv"]), base["gate"].numpy(), base["pos"].numpy(),
                          layer.kind, layer.window, layer.theta, layer.rot_dim, H, Hkv)
    for o, name in zip(outs, ("positions 0..T-1", f"positions shifted by {shift}")):
        check_close(o, want.reshape(T, -1), name)


def _v_row(j: int, gi: int) -> list[float]:
    """Small integers carried by token j's value (exact in bf16 and in fp32 sums)."""
    return [float(j & 63), float(j >> 6), 1.0, float((j * (gi + 3)) % 17)]


@pytest.mark.parametrize("kind,W,cap,positions", [
    (FULL, 0, 2048, [0, 1, 700, 2047]),
    (SLIDING, 512, 512, [5, 511, 512, 1000, 1023]),
    (SLIDING, 100, 512, [0, 99, 100, 513, 2000]),
], ids=["full", "ring-512", "window-100-in-ring-512"])
def test_zero_query_decode_averages_the_visible_slots(cuda, kind, W, cap, positions):
    """Decode with a zero query: every visible slot (the new token included)
    scores 0, so the output is the mean of the visible values.  This pins
    which slots a step sees: all past tokens of a full layer, the latest
    `window` tokens of a ring.  Slots no token has written hold NaN, which a
    correct step never reads."""
    H, Hkv = 16, 4
    B = len(positions)
    layer = wl.Layer(kind=kind, window=max(W, 1), theta=1e4 if kind else 5e6,
                     rot_dim=256 if kind else 64)
    g = torch.Generator().manual_seed(31 + cap + W)
    kc = torch.randn((B, Hkv, cap, 256), generator=g).to(torch.bfloat16)
    vc = torch.full((B, Hkv, cap, 256), float("nan"), dtype=torch.bfloat16)
    qkv = torch.zeros((B, (H + 2 * Hkv) * 256), dtype=torch.float32)
    qkv[:, H * 256:(H + Hkv) * 256] = torch.randn((B, Hkv * 256), generator=g)
    for b, p in enumerate(positions):
        # past tokens: slot s holds the latest token j < p with j = s (mod cap)
        n = min(p, cap)
        s = np.arange(n)
        j = s if kind == FULL else s + cap * ((p - 1 - s) // cap)
        for gi in range(Hkv):
            rows = torch.zeros((n, 256))
            rows[:, :4] = torch.tensor(np.array([_v_row(int(t), gi) for t in j]).reshape(n, 4))
            vc[b, gi, :n] = rows.to(torch.bfloat16)
            v0 = (H + Hkv + gi) * 256            # the new token's value
            qkv[b, v0:v0 + 4] = torch.tensor(_v_row(p, gi))
    gate = torch.full((B, H), 40.0)              # sigmoid(40) == 1.0 in fp32
    pos = torch.tensor(positions, dtype=torch.int32)
    out = fga.spark_attn_decode(qkv.to(torch.bfloat16).to(cuda), gate.to(cuda), pos.to(cuda),
                                kc.to(cuda), vc.to(cuda), layer)
    got = out.float().cpu().reshape(B, H, 256)
    assert not torch.isnan(got).any()
    assert float(got[:, :, 4:].abs().max()) == 0.0
    want = np.zeros((B, Hkv, 4))
    for b, p in enumerate(positions):
        lo = 0 if kind == FULL else max(0, p - W + 1)
        vis = range(lo, p + 1)
        for gi in range(Hkv):
            want[b, gi] = np.mean([_v_row(j, gi) for j in vis], axis=0)
    want = np.repeat(want, H // Hkv, axis=1)
    tol = (2.0 ** -8 + 2.0 ** -20) * np.abs(want) + 1e-7
    diff = np.abs(got[:, :, :4].double().numpy() - want)
    assert np.all(diff <= tol), diff.max()
