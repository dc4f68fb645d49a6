"""Seeded random sweep of the attention core against the fp64 oracle.

The parametrised tests name their cases; this sweep draws the combinations in
between: sequence count and length, group size G, layer kind, window, rotated
width, RoPE base, gate activation, gate scale and (for prefill) positions that
are not 0..T-1.  Every output element is compared with the oracle at the
parity bar of the other tests.  The draws are fixed by the seeds, so a failure
names its case and reproduces.
"""
from __future__ import annotations

import random

import numpy as np
import pytest
import torch

import full_gqa_attention_gb300 as fga
import oracle
import workloads as wl
from parity import check_close, silu_gate_unit
from test_decode_gpu import run_case

pytestmark = pytest.mark.gpu

GROUPS = [(8, 8), (8, 4), (16, 4), (16, 2), (8, 1)]   # (H, Hkv): G = 1, 2, 4, 8, 8


def draw_layer(rng: random.Random):
    kind = rng.choice([wl.FULL, wl.SLIDING])
    window = rng.choice([1, 2, 17, 128, 129, 300, 512, 1000]) if kind == wl.SLIDING else 0
    rot = rng.choice([0, 16, 64, 128, 192, 256])
    theta = rng.choice([1e4, 5e6, 1e6])
    gate_mode = rng.choice([0, 0, 1])
    return wl.Layer(kind=kind, window=max(window, 1), theta=theta, rot_dim=rot,
                    gate_mode=gate_mode)


@pytest.mark.parametrize("seed", range(16))
def test_prefill_sweep(cuda, seed):
    rng = random.Random(1000 + seed)
    H, Hkv = rng.choice(GROUPS)
    B = rng.choice([1, 2, 3])
    T = rng.choice([1, 5, 31, 64, 100, 129, 257, 400])
    layer = draw_layer(rng)
    gate_std = rng.choice([0.5, 1.0, 2.0])
    case = wl.PrefillCase(f"sweep{seed}", B=B, T=T, H=H, Hkv=Hkv, layer=layer,
                          seed=2000 + seed, gate_std=gate_std)
    positions = None
    if rng.random() < 0.5:           # positions that are not the token index
        g = torch.Generator().manual_seed(3000 + seed)
        positions = torch.randint(0, 1 << 20, (B, T), generator=g, dtype=torch.int64)
    x = wl.make_prefill_inputs(case, positions)
    out = fga.spark_attn_prefill(x["qkv"].to(cuda), x["gate"].to(cuda), x["pos"].to(cuda), layer)
    want = oracle.prefill(wl.bf16_bits(x["qkv"]), x["gate"].numpy(), x["pos"].numpy(), layer.kind,
                          layer.window, layer.theta, layer.rot_dim, H, Hkv,
                          gate_mode=layer.gate_mode).reshape(B * T, -1)
    unit = None
    if layer.gate_mode == 1:
        unit = silu_gate_unit(x["gate"].reshape(B * T, H).double().numpy())
    check_close(out.reshape(B * T, -1), want, f"sweep {seed}: B={B} T={T} H={H} Hkv={Hkv} "
                f"{layer} gate_std={gate_std} random_pos={positions is not None}", unit=unit)


@pytest.mark.parametrize("seed", range(12))
def test_decode_sweep(cuda, seed):
    rng = random.Random(5000 + seed)
    H, Hkv = rng.choice(GROUPS)
    layer = draw_layer(rng)
    if layer.kind == wl.SLIDING:
        cap = rng.choice([layer.window, max(layer.window, 512), max(layer.window, 128) + 64])
        positions = [rng.randrange(0, 3 * cap) for _ in range(rng.choice([1, 3, 5]))]
    else:
        cap = rng.choice([64, 300, 2048, 5000])
        positions = [rng.randrange(0, cap) for _ in range(rng.choice([1, 3, 5]))]
    run_case(cuda, layer, H, Hkv, cap, positions, seed=6000 + seed)


@pytest.mark.parametrize("seed", range(10))
def test_chunked_prefill_sweep(cuda, seed):
    """One sequence prefilled as a run of chunks of random sizes (the first at
    start 0) over a cache whose unwritten slots hold NaN, then one decode
    step.  Every chunk row and the decoded token are compared with the
    oracle's prefill of the whole sequence."""
    rng = random.Random(7000 + seed)
    H, Hkv = rng.choice(GROUPS)
    kind = rng.choice([wl.FULL, wl.SLIDING])
    W = rng.choice([17, 128, 300, 512]) if kind == wl.SLIDING else 0
    layer = wl.Layer(kind=kind, window=max(W, 1), theta=rng.choice([1e4, 5e6]),
                     rot_dim=rng.choice([0, 16, 64, 128, 256]))
    sizes = [rng.choice([1, 7, 64, 100, 129, 200, 333]) for _ in range(rng.choice([2, 3, 5]))]
    total = sum(sizes)
    if kind == wl.FULL:
        cap = total + 1 + rng.choice([0, 5, 200])
    else:
        cap = (W + max(sizes) - 1 + 127) // 128 * 128 + rng.choice([0, 128])
    case = wl.PrefillCase(f"cs{seed}", B=1, T=total + 1, H=H, Hkv=Hkv, layer=layer,
                          seed=8000 + seed)
    x = wl.make_prefill_inputs(case)
    kc = torch.full((1, Hkv, cap, 256), float("nan"), dtype=torch.bfloat16, device=cuda)
    vc = torch.full_like(kc, float("nan"))
    outs, s0 = [], 0
    for n in sizes:
        sl = slice(s0, s0 + n)
        outs.append(fga.spark_attn_prefill_chunk(
            x["qkv"][:, sl].contiguous().to(cuda), x["gate"][:, sl].contiguous().to(cuda),
            x["pos"][:, sl].contiguous().to(cuda), kc, vc,
            torch.tensor([s0], dtype=torch.int32, device=cuda), layer))
        s0 += n
    got = torch.cat(outs, dim=1).reshape(total, -1)
    qb = wl.bf16_bits(x["qkv"])
    want = oracle.prefill(qb, x["gate"].numpy(), x["pos"].numpy(), layer.kind, layer.window,
                          layer.theta, layer.rot_dim, H, Hkv)
    want = want.reshape(total + 1, -1)
    check_close(got, want[:total], f"chunks {sizes} cap={cap} H={H} Hkv={Hkv} {layer}")
    y = fga.spark_attn_decode(x["qkv"][:, total].contiguous().to(cuda),
                              x["gate"][:, total].contiguous().to(cuda),
                              torch.tensor([total], dtype=torch.int32, device=cuda), kc, vc, layer)
    check_close(y, want[total:], f"decode after chunks {sizes}")


@pytest.mark.parametrize("seed", range(8))
def test_attention_block_sweep(cuda, seed):
    """The attention block (projections around the core) over random hidden
    sizes, lengths (few rows take the GEMV path, more the tcgen05 GEMM with
    RoPE in its epilogue), group sizes, layer kinds and rotated widths."""
    from test_layer_gpu import run_prefill
    rng = random.Random(9000 + seed)
    H, Hkv = rng.choice(GROUPS)
    B = rng.choice([1, 2])
    T = rng.choice([1, 3, 8, 9, 100, 129, 300])
    hidden = rng.choice([264, 512, 1032, 2048])
    kind = rng.choice([wl.FULL, wl.SLIDING])
    layer = wl.Layer(kind=kind, window=rng.choice([17, 128, 512]) if kind == wl.SLIDING else 1,
                     theta=rng.choice([1e4, 5e6]), rot_dim=rng.choice([0, 16, 64, 128, 256]),
                     gate_mode=rng.choice([0, 0, 1]))
    # with the silu gate the logits are kept O(1), as in the block's silu test, so that
    # the gate factor (up to |g|) does not scale the bf16 rounding past the bar
    run_prefill(cuda, B, T, hidden, H, Hkv, layer, seed=9500 + seed,
                gate_scale=0.3 if layer.gate_mode == 1 else 1.0)
