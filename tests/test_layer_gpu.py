"""GPU parity of the attention block (projections around the core) against the
fp64 oracle, through the C ABI.

Spark-X2.5 architecture page, §3 Eq. 1 and Fig. 1: q_k_v_proj and g_proj on
the normed hidden state, the core, out_proj.  Weights are seeded random
(N(0, 1/fan_in), so activations stay O(1)); the bar is the core's: max-abs
<= 2e-2 and rel-L2 <= 1e-2 against fp64.
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
D = 256


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().astype(np.uint16)


def weights(hidden: int, H: int, Hkv: int, seed: int, gate_scale: float = 1.0):
    g = torch.Generator().manual_seed(seed)
    w_qkv = (torch.randn(((H + 2 * Hkv) * D, hidden), generator=g) / hidden ** 0.5)
    w_g = (torch.randn((H, hidden), generator=g) * gate_scale / hidden ** 0.5)
    w_o = (torch.randn((hidden, H * D), generator=g) / (H * D) ** 0.5)
    return [w.to(torch.bfloat16) for w in (w_qkv, w_g, w_o)]


def hidden_states(shape, seed: int) -> torch.Tensor:
    return torch.randn(shape, generator=torch.Generator().manual_seed(seed)).to(torch.bfloat16)


def run_prefill(cuda, B, T, hidden, H, Hkv, layer, seed, rows=None, gate_scale=1.0):
    x = hidden_states((B, T, hidden), seed)
    w = weights(hidden, H, Hkv, seed + 1, gate_scale)
    pos = torch.arange(T, dtype=torch.int32).repeat(B, 1)
    ws = fga.new_workspace(fga.spark_attn_layer_prefill_workspace_size(B, T, hidden, H, Hkv,
                                                                       layer))
    y = fga.spark_attn_layer_prefill(x.to(cuda), *[t.to(cuda) for t in w], pos.to(cuda), layer,
                                     workspace=ws)
    assert fga.spark_attn_read_status(ws) == 0
    want = oracle.layer_prefill(bits(x), *[bits(t) for t in w], pos.numpy(), layer.kind,
                                layer.window, layer.theta, layer.rot_dim, H, Hkv, rows=rows,
                                gate_mode=layer.gate_mode)
    got = y.reshape(B * T, hidden)
    if rows is not None:
        got = got[torch.as_tensor(rows, device=got.device)]
    else:
        want = want.reshape(B * T, hidden)
    check_close(got, want, f"layer prefill B={B} T={T} hidden={hidden} H={H} Hkv={Hkv} "
                           f"kind={layer.kind} W={layer.window}")
    return y


@pytest.mark.parametrize("layer", [wl.FULL_LAYER, wl.SLIDING_LAYER,
                                   wl.Layer(kind=SLIDING, window=100, theta=1e4, rot_dim=256,
                                            gate_mode=0)],
                         ids=["full", "sliding512", "sliding100"])
@pytest.mark.parametrize("B,T,hidden,H,Hkv", [(2, 300, 512, 4, 1), (1, 129, 264, 8, 2)])
def test_layer_prefill_small(cuda, layer, B, T, hidden, H, Hkv):
    run_prefill(cuda, B, T, hidden, H, Hkv, layer, seed=31)


@pytest.mark.parametrize("kind", [FULL, SLIDING], ids=["full", "sliding"])
def test_layer_prefill_silu_gate(cuda, kind):
    # gate_attn_act_mode = silu (Spark §3); logits kept O(1) so that the
    # gate's factor (up to |g|) does not scale the bf16 rounding past the bar
    layer = wl.Layer(kind=kind, window=64, theta=1e4, rot_dim=256, gate_mode=1)
    run_prefill(cuda, 2, 150, 512, 4, 1, layer, seed=44, gate_scale=0.3)


def test_layer_prefill_1p7b_sliding_whole(cuda):
    # 1.7B shapes (hidden 2048, H 8, Hkv 2), every row
    run_prefill(cuda, 1, 1024, 2048, 8, 2, wl.SLIDING_LAYER, seed=32)


def test_layer_prefill_4b_full_sampled(cuda):
    # 4B shapes (hidden 2560, H 16, Hkv 4): sampled rows across the sequence
    T = 4096
    rows = np.unique(np.concatenate([np.arange(0, 40), np.arange(T - 40, T),
                                     np.random.default_rng(33).integers(0, T, 120)]))
    run_prefill(cuda, 1, T, 2560, 16, 4, wl.FULL_LAYER, seed=34, rows=rows)


def test_layer_prefill_fills_the_cache(cuda):
    """With caches, the block stores its own rotated keys and values; a decode
    step through the block then matches the oracle's decode over the oracle's
    own caches (built from the oracle's projections, never the GPU's)."""
    B, T, hidden, H, Hkv, cap = 2, 200, 512, 4, 1, 256
    layer = wl.FULL_LAYER
    x = hidden_states((B, T, hidden), 35)
    w = weights(hidden, H, Hkv, 36)
    wd = [t.to(cuda) for t in w]
    pos = torch.arange(T, dtype=torch.int32).repeat(B, 1)
    kc = torch.zeros((B, Hkv, cap, D), dtype=torch.bfloat16, device=cuda)
    vc = torch.zeros_like(kc)
    fga.spark_attn_layer_prefill(x.to(cuda), *wd, pos.to(cuda), layer, k_cache=kc, v_cache=vc)
    xq = oracle.bits_to_f64(bits(x))
    qkv_bits = oracle.bf16_round_bits(xq @ oracle.bits_to_f64(bits(w[0])).T)
    ko = np.zeros((B, Hkv, cap, D), np.uint16)
    vo = np.zeros((B, Hkv, cap, D), np.uint16)
    for b in range(B):
        for t in range(T):
            k = oracle.bits_to_f64(qkv_bits[b, t, H * D:(H + Hkv) * D]).reshape(Hkv, D)
            ko[b, :, t] = oracle.bf16_round_bits(oracle.rope(k, np.full(Hkv, t), layer.rot_dim,
                                                             layer.theta))
            vo[b, :, t] = qkv_bits[b, t, (H + Hkv) * D:].reshape(Hkv, D)
    # the same tokens: values within one bf16 ulp, plus 2^-12 for the fp32
    # accumulation of the GPU projection (it decides the rounding of values
    # near zero); rotated keys within two ulps of the head's largest element
    # (a one-ulp difference in a projected key moves both members of its pair,
    # and a rotated element can be much smaller than its pair)
    g64, w64 = oracle.bits_to_f64(bits(vc.cpu())), oracle.bits_to_f64(vo)
    assert np.all(np.abs(g64 - w64) <= 2.0 ** -7 * np.abs(w64) + 2.0 ** -12)
    g64, w64 = oracle.bits_to_f64(bits(kc.cpu())), oracle.bits_to_f64(ko)
    assert np.all(np.abs(g64 - w64) <= 2.0 ** -6 * np.abs(w64).max(axis=-1, keepdims=True) + 1e-30)
    # one decode step at pos = T through the block
    xn = hidden_states((B, hidden), 37)
    pn = torch.full((B,), T, dtype=torch.int32)
    y = fga.spark_attn_layer_decode(xn.to(cuda), *wd, pn.to(cuda), kc, vc, layer)
    want, _, _ = oracle.layer_decode(bits(xn), *[bits(t) for t in w], pn.numpy(), ko, vo,
                                     layer.kind, layer.window, layer.theta, layer.rot_dim, H, Hkv)
    check_close(y, want, "layer decode after layer prefill")


@pytest.mark.parametrize("layer,cap,positions", [
    (wl.FULL_LAYER, 5000, [0, 17, 4095, 4999]),
    (wl.SLIDING_LAYER, 512, [0, 511, 512, 70000]),
    (wl.SLIDING_LAYER, 512, [1, 3, 100, 300]),
], ids=["full", "sliding", "sliding-ring-filling"])
def test_layer_decode_4b(cuda, layer, cap, positions):
    B, hidden, H, Hkv = len(positions), 2560, 16, 4
    x = hidden_states((B, hidden), 38)
    w = weights(hidden, H, Hkv, 39)
    kc = wl.fill_cache_(torch.empty((B, Hkv, cap, D), dtype=torch.bfloat16), 40)
    vc = wl.fill_cache_(torch.empty_like(kc), 41)
    pos = torch.tensor(positions, dtype=torch.int32)
    kd, vd = kc.to(cuda), vc.to(cuda)
    ws = fga.new_workspace(fga.spark_attn_layer_decode_workspace_size(B, hidden, H, Hkv, cap,
                                                                      layer))
    y = fga.spark_attn_layer_decode(x.to(cuda), *[t.to(cuda) for t in w], pos.to(cuda), kd, vd,
                                    layer, workspace=ws)
    assert fga.spark_attn_read_status(ws) == 0
    want, k_new, v_new = oracle.layer_decode(bits(x), *[bits(t) for t in w], pos.numpy(),
                                             bits(kc), bits(vc), layer.kind, layer.window,
                                             layer.theta, layer.rot_dim, H, Hkv)
    check_close(y, want, f"layer decode kind={layer.kind}")
    vb = oracle.bits_to_f64(bits(vd.cpu()))
    for b, p in enumerate(positions):
        slot = p if layer.kind == FULL else p % cap
        # the new value: the block's own v projection, within one bf16 ulp
        # (plus the fp32-accumulation floor, as above)
        assert np.all(np.abs(vb[b, :, slot] - v_new[b]) <= 2.0 ** -7 * np.abs(v_new[b]) + 2.0 ** -12)


@pytest.mark.parametrize("B", [1, 8, 12], ids=["gemv-1", "gemv-8", "gemm-12"])
def test_layer_decode_batch_sizes(cuda, B):
    # up to 8 sequences the projections are the library's weight-streaming
    # GEMV (g_proj fused with q_k_v_proj); beyond, its tcgen05 GEMM
    layer, cap, hidden, H, Hkv = wl.SLIDING_LAYER, 512, 2560, 16, 4
    x = hidden_states((B, hidden), 45)
    w = weights(hidden, H, Hkv, 46)
    kc = wl.fill_cache_(torch.empty((B, Hkv, cap, D), dtype=torch.bfloat16), 47)
    vc = wl.fill_cache_(torch.empty_like(kc), 48)
    pos = torch.tensor([(97 * b + 5) % 3000 for b in range(B)], dtype=torch.int32)
    y = fga.spark_attn_layer_decode(x.to(cuda), *[t.to(cuda) for t in w], pos.to(cuda),
                                    kc.to(cuda), vc.to(cuda), layer)
    want, _, _ = oracle.layer_decode(bits(x), *[bits(t) for t in w], pos.numpy(), bits(kc),
                                     bits(vc), layer.kind, layer.window, layer.theta,
                                     layer.rot_dim, H, Hkv)
    check_close(y, want, f"layer decode B={B}")


@pytest.mark.parametrize("rot_dim", [64, 128, 192, 256, 16])
@pytest.mark.parametrize("with_cache", [False, True], ids=["nocache", "cache"])
def test_layer_prefill_rope_in_projection_is_exact(cuda, rot_dim, with_cache):
    """The block rotates Q and K in the q_k_v_proj epilogue and runs the core
    without rotating (rotated widths with r/2 a multiple of 32).  That must
    give the same bits as the plain composition: the GEMM alone, the core
    rotating itself, out_proj.  (Gate weights are zero so that both paths
    take sigmoid(0) exactly; the fused gate column is checked against the
    oracle above.)  r = 16 keeps the unfused path and must match too."""
    B, T, hidden, H, Hkv = 2, 300, 512, 8, 2
    kind = SLIDING if rot_dim in (256, 128) else FULL
    layer = wl.Layer(kind=kind, window=100, theta=1e4 if kind == SLIDING else 5e6,
                     rot_dim=rot_dim)
    x = hidden_states((B, T, hidden), 60 + rot_dim).to(cuda)
    w_qkv, _, w_o = [t.to(cuda) for t in weights(hidden, H, Hkv, 61 + rot_dim)]
    w_g = torch.zeros((H, hidden), dtype=torch.bfloat16, device=cuda)
    pos = (torch.arange(T, dtype=torch.int32) * 37 + 5).repeat(B, 1).to(cuda)
    cap = T + 7
    caches = lambda: (torch.zeros((B, Hkv, cap, D), dtype=torch.bfloat16, device=cuda),  # noqa: E731
                      torch.zeros((B, Hkv, cap, D), dtype=torch.bfloat16, device=cuda))
    kc1, vc1 = caches() if with_cache else (None, None)
    kc2, vc2 = caches() if with_cache else (None, None)
    y = fga.spark_attn_layer_prefill(x, w_qkv, w_g, w_o, pos, layer, k_cache=kc1, v_cache=vc1)
    qkv = fga.spark_attn_linear(x, w_qkv)
    gate = fga.spark_attn_linear(x, w_g).float()
    if with_cache:
        attn = fga.spark_attn_prefill_cache(qkv, gate, pos, kc2, vc2, layer)
    else:
        attn = fga.spark_attn_prefill(qkv, gate, pos, layer)
    y2 = fga.spark_attn_linear(attn, w_o)
    torch.cuda.synchronize()
    assert torch.equal(y, y2)
    if with_cache:
        assert torch.equal(kc1, kc2) and torch.equal(vc1, vc2)


def test_layer_prefill_few_rows_uses_gemv(cuda):
    # B*T <= 8 rows: the projections take the GEMV path in prefill too
    run_prefill(cuda, 2, 3, 512, 4, 1, wl.FULL_LAYER, seed=49)


def test_layer_rejects_before_enqueueing(cuda):
    """A cache too small for the core is refused before the projections run."""
    B, T, hidden, H, Hkv = 1, 64, 512, 4, 1
    w = [t.to(cuda) for t in weights(hidden, H, Hkv, 42)]
    x = hidden_states((B, T, hidden), 43).to(cuda)
    pos = torch.arange(T, dtype=torch.int32, device=cuda)[None]
    kc = torch.zeros((B, Hkv, 32, D), dtype=torch.bfloat16, device=cuda)  # FULL needs cap >= T
    y = torch.full((B, T, hidden), 7.0, dtype=torch.bfloat16, device=cuda)
    with pytest.raises(fga.SparkError):
        fga.spark_attn_layer_prefill(x, *w, pos, wl.FULL_LAYER, k_cache=kc, v_cache=kc.clone(),
                                     y=y)
    torch.cuda.synchronize()
    assert bool((y == 7.0).all())
