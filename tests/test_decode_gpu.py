"""GPU parity of one decode step against the fp64 oracle (through the C ABI).

Output: max-abs <= 2e-2 and rel-L2 <= 1e-2.  Cache update: the slot of the
new position is rewritten (value bit-exact, unrotated key dims bit-exact,
rotated key dims within one bf16 ulp plus a 2e-6 floor of the exact fp64
rotation: the GPU rotates in fp32), every other slot is untouched bit for bit.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import full_gqa_attention_gb300 as fga
import oracle
import workloads as wl
from parity import (bits_to_f64, check_close, check_rotated_bf16, f64_to_bf16_bits,
                    silu_gate_unit)

pytestmark = pytest.mark.gpu

FULL, SLIDING = wl.FULL, wl.SLIDING


def run_case(cuda, layer, H, Hkv, cap, positions, seed, check_cache=True):
    B = len(positions)
    case = wl.DecodeCase("t", B=B, H=H, Hkv=Hkv, layer=layer, seed=seed, cap=cap,
                         len_lo=0, len_hi=0)
    step = wl.make_decode_step_inputs(case)
    pos = torch.tensor(positions, dtype=torch.int32)
    kc = wl.fill_cache_(torch.empty((B, Hkv, cap, 256), dtype=torch.bfloat16), seed + 11)
    vc = wl.fill_cache_(torch.empty_like(kc), seed + 12)
    kd, vd = kc.to(cuda), vc.to(cuda)
    ws = fga.new_workspace(fga.spark_attn_decode_workspace_size(B, H, Hkv, cap, layer))
    out = fga.spark_attn_decode(step["qkv"].to(cuda), step["gate"].to(cuda), pos.to(cuda), kd,
                                vd, layer, workspace=ws)
    torch.cuda.synchronize()
    assert fga.spark_attn_read_status(ws) == 0
    want, k_new, v_new = oracle.decode(wl.bf16_bits(step["qkv"]), step["gate"].numpy(),
                                       pos.numpy(), wl.bf16_bits(kc), wl.bf16_bits(vc),
                                       layer.kind, layer.window, layer.theta, layer.rot_dim, H,
                                       Hkv, gate_mode=layer.gate_mode)
    # silu gate: max-abs per unit of gate factor max(1, |silu(g)|), see parity.py
    unit = silu_gate_unit(step["gate"]) if layer.gate_mode == 1 else None
    check_close(out, want, f"decode kind={layer.kind} G={H // Hkv} cap={cap} pos={positions}",
                unit=unit)
    if check_cache:
        kb, vb = wl.bf16_bits(kd), wl.bf16_bits(vd)
        k0, v0 = wl.bf16_bits(kc), wl.bf16_bits(vc)
        for b, p in enumerate(positions):
            slot = p if layer.kind == FULL else p % cap
            kb_slot, vb_slot = kb[b, :, slot].copy(), vb[b, :, slot].copy()
            assert np.array_equal(vb_slot, f64_to_bf16_bits(v_new[b])), "value slot"
            r = layer.rot_dim
            want_k = f64_to_bf16_bits(k_new[b])
            assert np.array_equal(kb_slot[:, r:], want_k[:, r:]), "unrotated key dims"
            k_in = bits_to_f64(wl.bf16_bits(step["qkv"][b, H * 256:(H + Hkv) * 256]))
            check_rotated_bf16(kb_slot[:, :r], k_new[b][:, :r],
                               np.abs(k_in.reshape(Hkv, 256)).max(axis=-1, keepdims=True),
                               "new key")
            kb[b, :, slot] = k0[b, :, slot]
            vb[b, :, slot] = v0[b, :, slot]
        assert np.array_equal(kb, k0) and np.array_equal(vb, v0), "other cache slots changed"
    return out


@pytest.mark.parametrize("positions", [[0, 1, 63, 64], [65, 1000, 4095, 2047]])
def test_full_layer_4b(cuda, positions):
    run_case(cuda, wl.FULL_LAYER, 16, 4, 4096, positions, seed=1)


@pytest.mark.parametrize("positions", [[0, 1, 300, 510], [511, 512, 513, 1023],
                                       [1024, 5000, 131071, 1048575]])
def test_sliding_ring_512(cuda, positions):
    run_case(cuda, wl.SLIDING_LAYER, 16, 4, 512, positions, seed=2)


def test_ring_positions_at_the_limit(cuda):
    """Ring decode at positions up to 2^24 - 1 (the largest accepted): the
    new token's angles turn ~1.7e7 rad and its slot is pos mod 512."""
    top = (1 << 24) - 1
    run_case(cuda, wl.SLIDING_LAYER, 16, 4, 512, [top, top - 1, top - 511, top - 512], seed=31)


def test_ring_larger_than_window(cuda):
    run_case(cuda, wl.SLIDING_LAYER, 16, 4, 600, [100, 599, 600, 601, 1799, 2000], seed=3)


@pytest.mark.parametrize("H,Hkv", [(8, 8), (8, 4), (16, 2), (8, 2)])
def test_group_sizes(cuda, H, Hkv):
    run_case(cuda, wl.FULL_LAYER, H, Hkv, 1500, [7, 640, 1499], seed=4)
    run_case(cuda, wl.SLIDING_LAYER, H, Hkv, 512, [7, 700], seed=5)


@pytest.mark.parametrize("rot", [0, 16, 128])
def test_rotary_widths(cuda, rot):
    layer = wl.Layer(kind=FULL, window=0, theta=5e6, rot_dim=rot)
    run_case(cuda, layer, 16, 4, 2100, [1, 2049, 2099], seed=6)


@pytest.mark.parametrize("kind", [FULL, SLIDING])
def test_silu_gate(cuda, kind):
    """gate_attn_act_mode = silu (Spark-X2.5 architecture, §3)."""
    layer = wl.Layer(kind=kind, window=512, theta=5e6 if kind == FULL else 1e4,
                     rot_dim=64 if kind == FULL else 256, gate_mode=1)
    run_case(cuda, layer, 16, 4, 2048 if kind == FULL else 512, [0, 700, 2047], seed=31)


def test_small_windows(cuda):
    for W in (1, 2, 100):
        layer = wl.Layer(kind=SLIDING, window=W, theta=1e4, rot_dim=256)
        run_case(cuda, layer, 8, 2, max(W, 128), [0, 1, W, 3 * W + 5], seed=7 + W)


def test_split_count_invariance(cuda):
    """The same tokens through differently split caches give one answer."""
    outs = []
    for cap in (1100, 5000, 70000):
        torch.manual_seed(0)
        B, H, Hkv = 1, 16, 4
        case = wl.DecodeCase("t", B=B, H=H, Hkv=Hkv, layer=wl.FULL_LAYER, seed=8, cap=cap,
                             len_lo=0, len_hi=0)
        step = wl.make_decode_step_inputs(case)
        pos = torch.tensor([1050], dtype=torch.int32)
        kc = torch.zeros((B, Hkv, cap, 256), dtype=torch.bfloat16)
        vc = torch.zeros_like(kc)
        base = wl.fill_cache_(torch.empty((B, Hkv, 1100, 256), dtype=torch.bfloat16), 9)
        kc[:, :, :1100] = base
        vc[:, :, :1100] = base.flip(-1)
        out = fga.spark_attn_decode(step["qkv"].to(cuda), step["gate"].to(cuda), pos.to(cuda),
                                    kc.to(cuda), vc.to(cuda), wl.FULL_LAYER)
        outs.append(out.float().cpu())
    for o in outs[1:]:
        assert torch.allclose(o, outs[0], atol=8e-3, rtol=0)


def test_unwritten_slots_may_hold_nan(cuda):
    """Cache slots at and past the new position were never written and may hold
    any bit pattern; NaN there must not reach the output."""
    layer = wl.FULL_LAYER
    B, H, Hkv, cap = 2, 16, 4, 1000
    case = wl.DecodeCase("t", B=B, H=H, Hkv=Hkv, layer=layer, seed=12, cap=cap, len_lo=0,
                         len_hi=0)
    step = wl.make_decode_step_inputs(case)
    pos = torch.tensor([100, 777], dtype=torch.int32)
    kc = wl.fill_cache_(torch.empty((B, Hkv, cap, 256), dtype=torch.bfloat16), 13)
    vc = wl.fill_cache_(torch.empty_like(kc), 14)
    for b, p in enumerate(pos.tolist()):
        kc[b, :, p:] = float("nan")
        vc[b, :, p:] = float("nan")
    kd, vd = kc.to(cuda), vc.to(cuda)
    out = fga.spark_attn_decode(step["qkv"].to(cuda), step["gate"].to(cuda), pos.to(cuda), kd, vd,
                                layer)
    want, _, _ = oracle.decode(wl.bf16_bits(step["qkv"]), step["gate"].numpy(), pos.numpy(),
                               wl.bf16_bits(kc), wl.bf16_bits(vc), layer.kind, layer.window,
                               layer.theta, layer.rot_dim, H, Hkv)
    check_close(out, want, "decode over NaN-poisoned unwritten slots")


def test_bad_position_is_flagged(cuda):
    """A full-layer position at or past the cache end is skipped and flagged;
    the other sequences are still computed."""
    layer = wl.FULL_LAYER
    B, H, Hkv, cap = 2, 16, 4, 256
    case = wl.DecodeCase("t", B=B, H=H, Hkv=Hkv, layer=layer, seed=10, cap=cap, len_lo=0,
                         len_hi=0)
    step = wl.make_decode_step_inputs(case)
    kc = wl.fill_cache_(torch.empty((B, Hkv, cap, 256), dtype=torch.bfloat16), 3).to(cuda)
    vc = wl.fill_cache_(torch.empty((B, Hkv, cap, 256), dtype=torch.bfloat16), 4).to(cuda)
    pos = torch.tensor([100, 256], dtype=torch.int32, device=cuda)
    out = torch.full((B, H * 256), 7.0, dtype=torch.bfloat16, device=cuda)
    ws = fga.new_workspace(fga.spark_attn_decode_workspace_size(B, H, Hkv, cap, layer))
    fga.spark_attn_decode(step["qkv"].to(cuda), step["gate"].to(cuda), pos, kc, vc, layer,
                          out=out, workspace=ws)
    status = fga.spark_attn_read_status(ws, clear=True)
    assert status == fga.SPARK_DEVERR_POSITION
    assert torch.all(out[1] == 7.0), "skipped sequence must be left untouched"
    assert fga.spark_attn_read_status(ws) == 0


def test_fault_in_an_owned_workspace_is_raised(cuda):
    """With check_device_status on (the GPU test session turns it on), a call
    that allocates its own workspace raises the device fault it recorded."""
    layer = wl.FULL_LAYER
    B, H, Hkv, cap = 1, 16, 4, 128
    case = wl.DecodeCase("t", B=B, H=H, Hkv=Hkv, layer=layer, seed=11, cap=cap, len_lo=0,
                         len_hi=0)
    step = wl.make_decode_step_inputs(case)
    kc = torch.zeros((B, Hkv, cap, 256), dtype=torch.bfloat16, device=cuda)
    vc = torch.zeros_like(kc)
    pos = torch.tensor([cap], dtype=torch.int32, device=cuda)
    with pytest.raises(fga.SparkDeviceFault) as err:
        fga.spark_attn_decode(step["qkv"].to(cuda), step["gate"].to(cuda), pos, kc, vc, layer)
    assert err.value.bits == fga.SPARK_DEVERR_POSITION


def _full_size(cuda, dcase, sample_b=None):
    """Full-size decode in the launch configuration the benchmark times; the
    oracle checks every sequence (or the sampled ones), one at a time.

    The step writes only slot(pos) of each sequence, which the oracle
    overwrites with its own new key and value and which no visible past token
    occupies (on a ring it held token pos - cap, outside the window), so each
    sequence's cache is read back after the call: only its slots up to pos
    (full layer) or its ring, one sequence at a time, to bound host memory."""
    step = wl.make_decode_step_inputs(dcase)
    B, H, Hkv, cap = dcase.B, dcase.H, dcase.Hkv, dcase.cap
    kd = torch.empty((B, Hkv, cap, 256), dtype=torch.bfloat16, device=cuda)
    vd = torch.empty_like(kd)
    wl.fill_cache_(kd, dcase.seed + 100)
    wl.fill_cache_(vd, dcase.seed + 200)
    out = fga.spark_attn_decode(step["qkv"].to(cuda), step["gate"].to(cuda),
                                step["pos"].to(cuda), kd, vd, dcase.layer)
    torch.cuda.synchronize()
    out = out.cpu()
    L = dcase.layer
    for b in (range(B) if sample_b is None else sample_b):
        p = int(step["pos"][b])
        n = min(p + 1, cap) if L.kind == FULL else cap
        want, _, _ = oracle.decode(wl.bf16_bits(step["qkv"][b:b + 1]),
                                   step["gate"][b:b + 1].numpy(), step["pos"][b:b + 1].numpy(),
                                   wl.bf16_bits(kd[b:b + 1, :, :n].cpu()),
                                   wl.bf16_bits(vd[b:b + 1, :, :n].cpu()), L.kind, L.window,
                                   L.theta, L.rot_dim, H, Hkv)
        check_close(out[b:b + 1], want, f"{dcase.name} b={b} pos={p}")
    del kd, vd
    torch.cuda.empty_cache()


def test_batched_decode_full_size(cuda):
    """The 4B batched decode workload (64 sequences of 4096..131072 tokens, and
    64 full 512-slot rings): every sequence against the oracle."""
    _full_size(cuda, wl.DECODE_FULL_4B_B64)
    _full_size(cuda, wl.DECODE_SLIDING_4B_B64)


def test_million_token_decode(cuda):
    _full_size(cuda, wl.DECODE_FULL_4B_1M)
    _full_size(cuda, wl.DECODE_SLIDING_4B_1M)


def test_empty_batch(cuda):
    layer = wl.SLIDING_LAYER
    e = torch.empty((0, 24 * 256), dtype=torch.bfloat16, device=cuda)
    out = fga.spark_attn_decode(e, torch.empty((0, 16), device=cuda),
                                torch.empty((0,), dtype=torch.int32, device=cuda),
                                torch.empty((0, 4, 512, 256), dtype=torch.bfloat16, device=cuda),
                                torch.empty((0, 4, 512, 256), dtype=torch.bfloat16, device=cuda),
                                layer)
    assert out.shape == (0, 16 * 256)


@pytest.mark.parametrize("H,Hkv", [(16, 4), (8, 2), (8, 8)])
def test_window_one_passes_v_through_bit_exact(cuda, H, Hkv):
    """Window 1 on a 512-slot ring: every cached slot is outside the window,
    so the output is the new token's V slice of KV head h // (H/Hkv), times
    sigmoid(40) = 1 in fp32, bit for bit (layout pin on the decode path)."""
    G = H // Hkv
    layer = wl.Layer(kind=SLIDING, window=1, theta=1e4, rot_dim=256)
    B, cap = 3, 512
    case = wl.DecodeCase("w1", B=B, H=H, Hkv=Hkv, layer=layer, seed=21, cap=cap, len_lo=0,
                         len_hi=0)
    step = wl.make_decode_step_inputs(case)
    kc = wl.fill_cache_(torch.empty((B, Hkv, cap, 256), dtype=torch.bfloat16), 22).to(cuda)
    vc = wl.fill_cache_(torch.empty((B, Hkv, cap, 256), dtype=torch.bfloat16), 23).to(cuda)
    pos = torch.tensor([0, 700, 511], dtype=torch.int32, device=cuda)
    out = fga.spark_attn_decode(step["qkv"].to(cuda), torch.full((B, H), 40.0, device=cuda),
                                pos, kc, vc, layer)
    v = step["qkv"][:, (H + Hkv) * 256:].reshape(B, Hkv, 256)
    want = v[:, torch.arange(H) // G, :].reshape(B, H * 256)
    assert torch.equal(out.reshape(B, H * 256).cpu(), want)


# Steps whose scans have 2..8 splits per (sequence, KV head): spark_attn_decode
# merges them inside the split kernel, while spark_attn_decode_noalloc keeps the
# separate merge kernel there (its scratch holds no split counters).  The two
# merges run the same arithmetic in the same order.
FUSED_CASES = [
    # layer, H, Hkv, cap, positions (one per sequence)
    (wl.SLIDING_LAYER, 16, 4, 512, [1048575]),                    # the 1M step's rings: 8 splits
    (wl.SLIDING_LAYER, 16, 4, 512, [600, 511, 40]),               # one sequence with one split
    (wl.FULL_LAYER, 16, 4, 300, [299, 0]),                        # nothing cached at pos 0
    (wl.FULL_LAYER, 16, 2, 400, [399, 130]),                      # G = 8: two parts per head
    (wl.SLIDING_LAYER, 8, 8, 512, [700, 300]),                    # G = 1
    (wl.FULL_LAYER, 8, 4, 20000, [19999, 5000, 64, 1, 12345, 6000]),  # long chunks, 6 splits
    (wl.Layer(kind=SLIDING, window=512, theta=1e4, rot_dim=256, gate_mode=1), 16, 4, 512,
     [2000, 900]),                                                # silu gate
]


@pytest.mark.parametrize("layer,H,Hkv,cap,positions", FUSED_CASES)
def test_merge_in_split_kernel_equals_merge_kernel(cuda, layer, H, Hkv, cap, positions):
    B = len(positions)
    g = torch.Generator(cuda).manual_seed(B * 131 + cap)
    qkv = torch.randn((B, (H + 2 * Hkv) * 256), generator=g, device=cuda).to(torch.bfloat16)
    gate = torch.randn((B, H), generator=g, device=cuda)
    pos = torch.tensor(positions, dtype=torch.int32, device=cuda)
    k = torch.randn((B, Hkv, cap, 256), generator=g, device=cuda).to(torch.bfloat16)
    v = torch.randn((B, Hkv, cap, 256), generator=g, device=cuda).to(torch.bfloat16)
    k2, v2 = k.clone(), v.clone()
    ws = fga.new_workspace(fga.spark_attn_decode_workspace_size(B, H, Hkv, cap, layer))
    fused = fga.spark_attn_decode(qkv, gate, pos, k, v, layer, workspace=ws)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    merged = fga.spark_attn_decode_noalloc(qkv, gate, pos, k2, v2, layer, device_status=status)
    torch.cuda.synchronize()
    assert fga.spark_attn_read_status(ws) == 0 and int(status.item()) == 0
    assert torch.equal(fused, merged)
    assert torch.equal(k, k2) and torch.equal(v, v2), "cache updates differ"
    # the split counters (header words after the status word) are back at 0
    assert int(torch.count_nonzero(ws[4:256])) == 0


def test_split_counters_survive_repeated_and_mixed_calls(cuda):
    """One workspace serves calls of different shapes in turn; each call finds
    its counters at 0 and leaves them there, so every result stays right."""
    layer = wl.SLIDING_LAYER
    H, Hkv, cap = 16, 4, 512
    size = max(fga.spark_attn_decode_workspace_size(B, H, Hkv, cap, layer) for B in (1, 2, 5))
    ws = fga.new_workspace(size)
    for i, B in enumerate((1, 5, 2, 1, 5)):
        positions = [3000 + 97 * b + i for b in range(B)]
        out = run_case_with_workspace(cuda, layer, H, Hkv, cap, positions, seed=40 + i, ws=ws)
        del out
        assert int(torch.count_nonzero(ws[4:256])) == 0


def run_case_with_workspace(cuda, layer, H, Hkv, cap, positions, seed, ws):
    B = len(positions)
    case = wl.DecodeCase("t", B=B, H=H, Hkv=Hkv, layer=layer, seed=seed, cap=cap,
                         len_lo=0, len_hi=0)
    step = wl.make_decode_step_inputs(case)
    pos = torch.tensor(positions, dtype=torch.int32)
    kc = wl.fill_cache_(torch.empty((B, Hkv, cap, 256), dtype=torch.bfloat16), seed + 11)
    vc = wl.fill_cache_(torch.empty_like(kc), seed + 12)
    out = fga.spark_attn_decode(step["qkv"].to(cuda), step["gate"].to(cuda), pos.to(cuda),
                                kc.to(cuda), vc.to(cuda), layer, workspace=ws)
    torch.cuda.synchronize()
    assert fga.spark_attn_read_status(ws) == 0
    want, _, _ = oracle.decode(wl.bf16_bits(step["qkv"]), step["gate"].numpy(), pos.numpy(),
                               wl.bf16_bits(kc), wl.bf16_bits(vc), layer.kind, layer.window,
                               layer.theta, layer.rot_dim, H, Hkv)
    check_close(out, want, f"decode B={B} pos={positions} (shared workspace)")
    return out


@pytest.mark.parametrize("B,H,Hkv", [(21, 12, 3), (16, 16, 4)], ids=["63-counters", "64-pairs"])
def test_split_counter_capacity(cuda, B, H, Hkv):
    """The workspace header holds 63 split counters.  With B * Hkv = 63 pairs
    the last header word is used; with 64 the merge kernel runs instead.
    Both give the oracle's result and leave the header words at 0."""
    layer = wl.SLIDING_LAYER
    cap = 512
    ws = fga.new_workspace(fga.spark_attn_decode_workspace_size(B, H, Hkv, cap, layer))
    for rep in range(2):
        positions = [600 + 37 * b + rep for b in range(B)]
        run_case_with_workspace(cuda, layer, H, Hkv, cap, positions, seed=60 + rep, ws=ws)
        assert int(torch.count_nonzero(ws[4:256])) == 0
