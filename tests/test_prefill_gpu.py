"""GPU parity of prefill against the fp64 oracle (through the C ABI).

Bar: max-abs <= 2e-2 and rel-L2 <= 1e-2 against fp64.  Small cases compare
every output element; the full-size workloads compare sampled rows (the
oracle computes rows one by one) in the same launch configuration the
benchmark times.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import full_gqa_attention_gb300 as fga
import oracle
import workloads as wl
from parity import check_close, silu_gate_unit

pytestmark = pytest.mark.gpu

FULL, SLIDING = wl.FULL, wl.SLIDING


def run(cuda, case, rows=None, positions=None):
    """Runs one prefill case through the C ABI and checks it against the oracle.

    With the silu gate the max-abs bar is taken per unit of gate factor
    max(1, |silu(g)|) (see parity.py); rel-L2 is checked on the raw output."""
    x = wl.make_prefill_inputs(case, positions)
    ws = fga.new_workspace(fga.spark_attn_prefill_workspace_size(case.B, case.T, case.H,
                                                                 case.Hkv, case.layer))
    out = fga.spark_attn_prefill(x["qkv"].to(cuda), x["gate"].to(cuda), x["pos"].to(cuda),
                                 case.layer, workspace=ws)
    assert fga.spark_attn_read_status(ws) == 0
    L = case.layer
    want = oracle.prefill(wl.bf16_bits(x["qkv"]), x["gate"].numpy(), x["pos"].numpy(), L.kind,
                          L.window, L.theta, L.rot_dim, case.H, case.Hkv, rows=rows,
                          gate_mode=L.gate_mode)
    got = out.reshape(case.B * case.T, -1)
    if rows is not None:
        got = got[torch.as_tensor(rows, device=got.device)]
    else:
        want = want.reshape(case.B * case.T, -1)
    unit = None
    if L.gate_mode == 1:
        g = x["gate"].reshape(case.B * case.T, case.H).double().numpy()
        unit = silu_gate_unit(g[rows] if rows is not None else g)
    check_close(got, want, f"{case.name} B={case.B} T={case.T} H={case.H} Hkv={case.Hkv} "
                           f"kind={L.kind} W={L.window} r={L.rot_dim}", unit=unit)
    return out, x


SMALL_T = [1, 2, 31, 32, 33, 127, 128, 129, 300, 511, 512, 513, 1000]


@pytest.mark.parametrize("T", SMALL_T)
def test_full_layer_lengths(cuda, T):
    run(cuda, wl.PrefillCase("full", B=2, T=T, H=8, Hkv=2, layer=wl.FULL_LAYER, seed=T))


@pytest.mark.parametrize("T", SMALL_T)
def test_sliding_layer_lengths(cuda, T):
    run(cuda, wl.PrefillCase("sliding", B=1, T=T, H=8, Hkv=2, layer=wl.SLIDING_LAYER,
                             seed=100 + T))


# Grids of one to several waves of CTAs over 152 SMs, with query tiles of 1
# to 10 key tiles and every group size the kernel packs (G = 1, 4): each CTA
# must write its whole output tile, whatever runs beside it.
@pytest.mark.parametrize("kind,B,T,H,Hkv", [(SLIDING, 2, 1300, 16, 4), (FULL, 2, 1300, 16, 4),
                                            (SLIDING, 4, 1216, 8, 2), (FULL, 3, 1000, 8, 8),
                                            (SLIDING, 1, 2600, 16, 4), (FULL, 2, 2432, 8, 2)])
def test_item_lists_per_cta(cuda, kind, B, T, H, Hkv):
    layer = wl.FULL_LAYER if kind == FULL else wl.SLIDING_LAYER
    case = wl.PrefillCase("items", B=B, T=T, H=H, Hkv=Hkv, layer=layer, seed=7 * T + B)
    run(cuda, case)


@pytest.mark.parametrize("W", [1, 2, 63, 511, 513, 600, 4096])
def test_windows(cuda, W):
    layer = wl.Layer(kind=SLIDING, window=W, theta=1e4, rot_dim=256)
    run(cuda, wl.PrefillCase("win", B=1, T=700, H=16, Hkv=4, layer=layer, seed=W))


@pytest.mark.parametrize("H,Hkv", [(8, 8), (8, 4), (16, 2), (16, 4)])
def test_group_sizes(cuda, H, Hkv):
    run(cuda, wl.PrefillCase("g", B=2, T=333, H=H, Hkv=Hkv, layer=wl.FULL_LAYER, seed=H + Hkv))
    run(cuda, wl.PrefillCase("g", B=1, T=777, H=H, Hkv=Hkv, layer=wl.SLIDING_LAYER,
                             seed=H * Hkv))


@pytest.mark.parametrize("rot", [0, 16, 64, 128, 192, 256])
def test_rotary_widths(cuda, rot):
    layer = wl.Layer(kind=FULL, window=0, theta=5e6, rot_dim=rot)
    run(cuda, wl.PrefillCase("rot", B=1, T=257, H=8, Hkv=2, layer=layer, seed=rot))


@pytest.mark.parametrize("kind", [FULL, SLIDING])
def test_silu_gate(cuda, kind):
    """gate_attn_act_mode = silu (Spark-X2.5 architecture, §3)."""
    layer = wl.Layer(kind=kind, window=512, theta=5e6 if kind == FULL else 1e4,
                     rot_dim=64 if kind == FULL else 256, gate_mode=1)
    run(cuda, wl.PrefillCase("silu", B=2, T=600, H=16, Hkv=4, layer=layer, seed=21,
                             gate_std=2.0))


def test_large_positions(cuda):
    """Positions near the 1M context end (RoPE angles up to ~1e6 rad)."""
    case = wl.PrefillCase("pos", B=2, T=200, H=8, Hkv=2, layer=wl.FULL_LAYER, seed=5)
    base = torch.tensor([1048575 - 199, 700000], dtype=torch.int32)
    positions = base[:, None] + torch.arange(200, dtype=torch.int32)[None, :]
    run(cuda, case, positions=positions)
    case = wl.PrefillCase("pos", B=1, T=200, H=8, Hkv=2, layer=wl.SLIDING_LAYER, seed=6)
    rng = np.random.default_rng(0)
    run(cuda, case, positions=torch.tensor(rng.integers(0, 1 << 20, (1, 200)), dtype=torch.int32))


@pytest.mark.parametrize("layer", [wl.FULL_LAYER, wl.SLIDING_LAYER])
def test_positions_at_the_limit(cuda, layer):
    """Positions up to 2^24 - 1, the largest the library accepts: the highest
    frequency turns ~1.7e7 rad, where an fp32 angle would have lost every
    digit; descending and repeated positions are valid too."""
    case = wl.PrefillCase("poslim", B=2, T=160, H=8, Hkv=2, layer=layer, seed=7)
    top = (1 << 24) - 1
    positions = torch.stack([
        top - 159 + torch.arange(160, dtype=torch.int32),        # the last 160 positions
        torch.full((160,), top, dtype=torch.int32) - torch.arange(160, dtype=torch.int32) % 7,
    ])
    run(cuda, case, positions=positions)


@pytest.mark.parametrize("T,W,H,Hkv", [(513, 512, 8, 2), (257, 256, 8, 2), (1025, 512, 16, 4),
                                       (513, 512, 8, 8), (513, 512, 16, 2)])
def test_unmasked_last_tile_repeatable(cuda, T, W, H, Hkv):
    """A query tile holding one token whose window is a whole number of key
    tiles has no masked tile at all, so its softmax finishes early; the result
    must still be complete and identical from run to run."""
    layer = wl.Layer(kind=SLIDING, window=W, theta=1e4, rot_dim=256)
    case = wl.PrefillCase("tail", B=1, T=T, H=H, Hkv=Hkv, layer=layer, seed=T + H)
    out, x = run(cuda, case)
    args = [x["qkv"].to(cuda), x["gate"].to(cuda), x["pos"].to(cuda), layer]
    for _ in range(8):
        assert torch.equal(fga.spark_attn_prefill(*args), out)


def test_window_at_least_T_is_bit_identical_to_causal(cuda):
    x = wl.make_prefill_inputs(wl.PrefillCase("w", B=1, T=400, H=16, Hkv=4,
                                              layer=wl.FULL_LAYER, seed=9))
    args = [x["qkv"].to(cuda), x["gate"].to(cuda), x["pos"].to(cuda)]
    full = fga.spark_attn_prefill(*args, wl.Layer(kind=FULL, window=0, theta=1e4, rot_dim=256))
    for W in (400, 1000):
        sl = fga.spark_attn_prefill(*args, wl.Layer(kind=SLIDING, window=W, theta=1e4,
                                                    rot_dim=256))
        assert torch.equal(sl, full)


def test_gate_zero_halves_exactly(cuda):
    """sigmoid(0) = 1/2: halving is exact in bf16, so the two runs agree bit for bit."""
    case = wl.PrefillCase("g0", B=1, T=300, H=16, Hkv=4, layer=wl.FULL_LAYER, seed=10)
    x = wl.make_prefill_inputs(case)
    q, p = x["qkv"].to(cuda), x["pos"].to(cuda)
    big = fga.spark_attn_prefill(q, torch.full((1, 300, 16), 40.0, device=cuda), p, case.layer)
    half = fga.spark_attn_prefill(q, torch.zeros((1, 300, 16), device=cuda), p, case.layer)
    assert torch.equal(half.float() * 2.0, big.float())


@pytest.mark.parametrize("kind,W", [(FULL, 0), (SLIDING, 1), (SLIDING, 7), (SLIDING, 64),
                                    (SLIDING, 512), (SLIDING, 600)])
def test_band_edges_exact(cuda, kind, W):
    """Pins both edges of every row's visible band.  Without RoPE, keys
    k_j = -(j >> 4, j & 15, 0, ...) and q = (2560, 160, 0, ...) give the exact
    score q.k_j / 16 = -10 j, so softmax puts weight 1 - 5e-5 on the OLDEST
    visible key; with q negated, on the NEWEST.  V carries the key index
    (v_j = (j & 63, j >> 6, 0, ...)), so each output row reads back the index
    of its band edge: lo_i = max(0, i - W + 1) (window) or 0 (causal), and i."""
    T, H, Hkv = 700, 8, 2
    j = torch.arange(T)
    qkv = torch.zeros((1, T, (H + 2 * Hkv) * 256), dtype=torch.float32)
    for g in range(Hkv):
        k0, v0 = (H + g) * 256, (H + Hkv + g) * 256
        qkv[0, :, k0] = -(j >> 4).float()
        qkv[0, :, k0 + 1] = -(j & 15).float()
        qkv[0, :, v0] = (j & 63).float()
        qkv[0, :, v0 + 1] = (j >> 6).float()
    gate = torch.full((1, T, H), 40.0)   # sigmoid(40) == 1.0 in fp32
    pos = torch.arange(T, dtype=torch.int32)[None]
    layer = wl.Layer(kind=kind, window=max(W, 1), theta=1e4, rot_dim=0)
    lo = torch.clamp(j - W + 1, min=0) if kind == SLIDING else torch.zeros_like(j)
    for sign, edge in ((1.0, lo), (-1.0, j)):
        for h in range(H):
            qkv[0, :, h * 256] = 2560.0 * sign
            qkv[0, :, h * 256 + 1] = 160.0 * sign
        out = fga.spark_attn_prefill(qkv.to(torch.bfloat16).to(cuda), gate.to(cuda),
                                     pos.to(cuda), layer)
        got = out.float().cpu().reshape(T, H, 256)
        idx = torch.round(got[:, :, 0]) + 64 * torch.round(got[:, :, 1])
        assert torch.all((got[:, :, :2] - torch.round(got[:, :, :2])).abs() < 0.02)
        assert torch.equal(idx.long(), edge[:, None].expand(T, H)), (kind, W, sign)


def sample_rows(B, T, n_random, seed):
    rng = np.random.default_rng(seed)
    pick = set()
    for b in range(B):
        for t in [0, 1, 2, 31, 32, 33, 127, 128, 129, 511, 512, 513, T // 2, T - 2, T - 1]:
            if 0 <= t < T:
                pick.add(b * T + t)
    pick.update(int(r) for r in rng.integers(0, B * T, n_random))
    return np.array(sorted(pick), dtype=np.int64)


def test_sliding_1p7b_T1024_whole(cuda):
    run(cuda, wl.PREFILL_SLIDING_1P7B_T1024)


def test_full_4b_B2_T8192_sampled(cuda):
    c = wl.PREFILL_FULL_4B_B2_T8192
    run(cuda, c, rows=sample_rows(c.B, c.T, 160, 1))


def test_long_4b_T65536_sampled(cuda):
    for c in (wl.PREFILL_SLIDING_4B_T65536, wl.PREFILL_FULL_4B_T65536):
        run(cuda, c, rows=sample_rows(c.B, c.T, 48, 2))
        torch.cuda.empty_cache()


def test_empty(cuda):
    e = torch.empty((1, 0, 24 * 256), dtype=torch.bfloat16, device=cuda)
    out = fga.spark_attn_prefill(e, torch.empty((1, 0, 16), device=cuda),
                                 torch.empty((1, 0), dtype=torch.int32, device=cuda),
                                 wl.FULL_LAYER)
    assert out.shape == (1, 0, 16 * 256)


@pytest.mark.parametrize("H,Hkv,rot", [(16, 4, 256), (8, 2, 64), (8, 8, 0), (8, 1, 128)])
def test_window_one_passes_v_through_bit_exact(cuda, H, Hkv, rot):
    """Window 1: each row sees only its own token, so p = 1 and the output is
    that token's V slice of KV head h // (H/Hkv), times sigmoid(40) = 1 in
    fp32: bit for bit.  Pins the Q|K|V layout of qkv, the head-to-KV-head map
    and the output layout (Spark §3, Fig. 1) on the GPU."""
    G = H // Hkv
    case = wl.PrefillCase("w1", B=2, T=200, H=H, Hkv=Hkv,
                          layer=wl.Layer(kind=SLIDING, window=1, theta=1e4, rot_dim=rot), seed=13)
    x = wl.make_prefill_inputs(case)
    out = fga.spark_attn_prefill(x["qkv"].to(cuda), torch.full((2, 200, H), 40.0, device=cuda),
                                 x["pos"].to(cuda), case.layer)
    v = x["qkv"][:, :, (H + Hkv) * 256:].reshape(2, 200, Hkv, 256)
    want = v[:, :, torch.arange(H) // G, :].reshape(2, 200, H * 256)
    assert torch.equal(out.cpu(), want)
