"""GPU tests of the prefill from and to host memory (spark_attn_prefill_host).

It runs the same kernels as spark_attn_prefill, one sequence at a time, with
the copies of one sequence overlapping the compute of another; its output must
equal the device-memory call's bit for bit, for pinned and pageable buffers,
with odd batch sizes that reuse the two staging areas.
"""
from __future__ import annotations

import pytest
import torch

import full_gqa_attention_gb300 as fga
import oracle
import workloads as wl
from parity import check_close

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("layer", [wl.FULL_LAYER, wl.SLIDING_LAYER], ids=["full", "sliding"])
@pytest.mark.parametrize("B,T", [(1, 129), (3, 300), (5, 64)])
@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
def test_host_prefill_equals_device_prefill(cuda, layer, B, T, pinned):
    case = wl.PrefillCase("h", B=B, T=T, H=16, Hkv=4, layer=layer, seed=50 + B)
    x = wl.make_prefill_inputs(case)
    host = {k: (v.pin_memory() if pinned else v.clone()) for k, v in x.items()}
    want = fga.spark_attn_prefill(x["qkv"].to(cuda), x["gate"].to(cuda), x["pos"].to(cuda), layer)
    ws = fga.new_workspace(fga.spark_attn_prefill_host_workspace_size(B, T, 16, 4, layer))
    got = fga.spark_attn_prefill_host(host["qkv"], host["gate"], host["pos"], layer, workspace=ws)
    torch.cuda.synchronize()
    assert fga.spark_attn_read_status(ws) == 0
    assert torch.equal(got, want.cpu())


def test_host_prefill_silu_gate(cuda):
    layer = wl.Layer(kind=wl.SLIDING, window=100, theta=1e4, rot_dim=256, gate_mode=1)
    case = wl.PrefillCase("h", B=3, T=160, H=16, Hkv=4, layer=layer, seed=62)
    x = wl.make_prefill_inputs(case)
    want = fga.spark_attn_prefill(x["qkv"].to(cuda), x["gate"].to(cuda), x["pos"].to(cuda), layer)
    got = fga.spark_attn_prefill_host(x["qkv"].pin_memory(), x["gate"].pin_memory(),
                                      x["pos"].pin_memory(), layer)
    torch.cuda.synchronize()
    assert torch.equal(got, want.cpu())


def test_host_prefill_matches_the_oracle(cuda):
    case = wl.PrefillCase("h", B=2, T=200, H=8, Hkv=2, layer=wl.SLIDING_LAYER, seed=61)
    x = wl.make_prefill_inputs(case)
    got = fga.spark_attn_prefill_host(x["qkv"].pin_memory(), x["gate"].pin_memory(),
                                      x["pos"].pin_memory(), case.layer)
    torch.cuda.synchronize()
    L = case.layer
    want = oracle.prefill(wl.bf16_bits(x["qkv"]), x["gate"].numpy(), x["pos"].numpy(), L.kind,
                          L.window, L.theta, L.rot_dim, 8, 2)
    check_close(got.reshape(400, -1), want.reshape(400, -1), "host prefill")


def test_host_prefill_empty_and_rejects(cuda):
    layer = wl.FULL_LAYER
    e = torch.empty((0, 4, 6144), dtype=torch.bfloat16)
    out = fga.spark_attn_prefill_host(e, torch.empty((0, 4, 16)), torch.empty((0, 4),
                                      dtype=torch.int32), layer)
    assert out.shape == (0, 4, 4096)
    with pytest.raises(TypeError):
        fga.spark_attn_prefill_host(e.to(cuda), torch.empty((0, 4, 16)),
                                    torch.empty((0, 4), dtype=torch.int32), layer)


def test_host_prefill_long_sequences_full_layer_bit_exact(cuda):
    """Sequences longer than one host chunk (2048 tokens on a full layer) go through in chunks
    over a device KV cache; on a full layer the chunks' query and key tiles
    fall where the one-shot prefill puts them, so the output is identical."""
    case = wl.PrefillCase("hl", B=2, T=4500, H=16, Hkv=4, layer=wl.FULL_LAYER, seed=63)
    x = wl.make_prefill_inputs(case)
    want = fga.spark_attn_prefill(x["qkv"].to(cuda), x["gate"].to(cuda), x["pos"].to(cuda),
                                  case.layer)
    ws = fga.new_workspace(fga.spark_attn_prefill_host_workspace_size(2, 4500, 16, 4, case.layer))
    got = fga.spark_attn_prefill_host(x["qkv"].pin_memory(), x["gate"].pin_memory(),
                                      x["pos"].pin_memory(), case.layer, workspace=ws)
    torch.cuda.synchronize()
    assert fga.spark_attn_read_status(ws) == 0
    assert torch.equal(got, want.cpu())


def test_host_prefill_long_sequences_sliding_layer(cuda):
    """On a sliding layer the chunks read a ring in 128-aligned key tiles, so
    the rounding order differs from the one-shot prefill: checked against the
    oracle on rows around every chunk edge and the window edge."""
    case = wl.PrefillCase("hs", B=2, T=4500, H=16, Hkv=4, layer=wl.SLIDING_LAYER, seed=64)
    x = wl.make_prefill_inputs(case)
    got = fga.spark_attn_prefill_host(x["qkv"].pin_memory(), x["gate"].pin_memory(),
                                      x["pos"].pin_memory(), case.layer)
    torch.cuda.synchronize()
    import numpy as np
    edges = [0, 511, 512, 2047, 2048, 2049, 2559, 2560, 3071, 3072, 3073, 3583, 3584, 4095,
             4096, 4499]
    rows = np.array(sorted({b * 4500 + t for b in (0, 1) for e in edges
                            for t in range(max(0, e - 2), min(4500, e + 3))}))
    L = case.layer
    want = oracle.prefill(wl.bf16_bits(x["qkv"]), x["gate"].numpy(), x["pos"].numpy(), L.kind,
                          L.window, L.theta, L.rot_dim, 16, 4, rows=rows)
    check_close(got.reshape(9000, -1)[torch.as_tensor(rows)], want, "host prefill sliding chunks")


@pytest.mark.parametrize("kind,T", [(wl.FULL, 2049), (wl.FULL, 4097), (wl.SLIDING, 3072),
                                    (wl.SLIDING, 3073), (wl.SLIDING, 6200)])
def test_host_prefill_piece_boundaries(cuda, kind, T):
    """Lengths at the host pieces' edges: one token over a chunk (a one-token
    last piece), exactly one sliding chunk (one piece, no cache), and several
    sliding chunks whose ring wraps.  Rows around every piece edge and the
    window edge are checked against the oracle."""
    layer = wl.FULL_LAYER if kind == wl.FULL else wl.SLIDING_LAYER
    chunk = 2048 if kind == wl.FULL else 3072
    case = wl.PrefillCase("hb", B=1, T=T, H=16, Hkv=4, layer=layer, seed=70 + T)
    x = wl.make_prefill_inputs(case)
    ws = fga.new_workspace(fga.spark_attn_prefill_host_workspace_size(1, T, 16, 4, layer))
    got = fga.spark_attn_prefill_host(x["qkv"].pin_memory(), x["gate"].pin_memory(),
                                      x["pos"].pin_memory(), layer, workspace=ws)
    torch.cuda.synchronize()
    assert fga.spark_attn_read_status(ws) == 0
    import numpy as np
    edges = {0, 511, 512, T - 1} | {c for c in range(chunk, T, chunk)}
    rows = np.array(sorted({t for e in edges for t in range(max(0, e - 2), min(T, e + 3))}))
    L = case.layer
    want = oracle.prefill(wl.bf16_bits(x["qkv"]), x["gate"].numpy(), x["pos"].numpy(), L.kind,
                          L.window, L.theta, L.rot_dim, 16, 4, rows=rows)
    check_close(got.reshape(T, -1)[torch.as_tensor(rows)], want, f"host prefill T={T}")
    if kind == wl.FULL:
        # full-layer chunks put their tiles where the one-shot prefill does
        one = fga.spark_attn_prefill(x["qkv"].to(cuda), x["gate"].to(cuda), x["pos"].to(cuda),
                                     layer)
        assert torch.equal(got, one.cpu())
