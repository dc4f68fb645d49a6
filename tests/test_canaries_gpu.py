"""Out-of-bounds writes, caught with guard canaries (compute-sanitizer is not
available on this pool).

Every buffer a call writes -- outputs, KV caches, workspaces -- sits between
two 4 KB guard regions filled with a known byte pattern, 256-byte alignment
kept.  After the call the guards must be intact: no kernel, including the TMA
stores at ragged tensor ends, may write past the buffer it was given.  The
outputs are also checked against the fp64 oracle, so a guard cannot pass on a
call that did not run.
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

PAD = 4096          # bytes of guard on each side (a multiple of 256)
FILL = 0xA5


class Guarded:
    """A tensor of `shape` and `dtype` inside a byte buffer with guards."""

    def __init__(self, shape, dtype, device, init=None):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.n = n
        self.buf = torch.full((PAD + n + PAD,), FILL, dtype=torch.uint8, device=device)
        self.t = self.buf[PAD:PAD + n].view(dtype).reshape(shape)
        if init is not None:
            self.t.copy_(init)

    def intact(self) -> bool:
        return bool((self.buf[:PAD] == FILL).all()) and bool((self.buf[PAD + self.n:] == FILL).all())


def guarded_host(shape, dtype):
    g = Guarded(shape, dtype, "cpu")
    g.buf = g.buf.pin_memory()
    g.t = g.buf[PAD:PAD + g.n].view(dtype).reshape(shape)
    return g


def workspace(nbytes, cuda):
    g = Guarded((nbytes,), torch.uint8, cuda)
    g.t.zero_()
    return g


def oracle_prefill(x, layer, H, Hkv):
    L = layer
    return oracle.prefill(wl.bf16_bits(x["qkv"]), x["gate"].numpy(), x["pos"].numpy(), L.kind,
                          L.window, L.theta, L.rot_dim, H, Hkv)


@pytest.mark.parametrize("T", [1, 33, 129, 300])
@pytest.mark.parametrize("layer", [wl.FULL_LAYER, wl.SLIDING_LAYER], ids=["full", "sliding"])
def test_prefill_writes_only_its_output_and_workspace(cuda, layer, T):
    B, H, Hkv = 2, 16, 4
    x = wl.make_prefill_inputs(wl.PrefillCase("g", B=B, T=T, H=H, Hkv=Hkv, layer=layer, seed=T))
    out = Guarded((B, T, H * 256), torch.bfloat16, cuda)
    ws = workspace(fga.spark_attn_prefill_workspace_size(B, T, H, Hkv, layer), cuda)
    fga.spark_attn_prefill(x["qkv"].to(cuda), x["gate"].to(cuda), x["pos"].to(cuda), layer,
                           out=out.t, workspace=ws.t)
    torch.cuda.synchronize()
    assert out.intact() and ws.intact()
    check_close(out.t.reshape(B * T, -1), oracle_prefill(x, layer, H, Hkv).reshape(B * T, -1),
                f"guarded prefill T={T}")


# the ring holds the window plus one 100-token chunk, in whole 128-slot tiles
@pytest.mark.parametrize("layer,cap", [(wl.FULL_LAYER, 300), (wl.SLIDING_LAYER, 640)],
                         ids=["full", "ring"])
def test_cache_fill_chunk_and_decode_stay_inside_their_buffers(cuda, layer, cap):
    B, H, Hkv, T0, T1 = 2, 16, 4, 150, 100
    x = wl.make_prefill_inputs(wl.PrefillCase("g", B=B, T=T0 + T1 + 1, H=H, Hkv=Hkv,
                                              layer=layer, seed=5 + cap))
    kc = Guarded((B, Hkv, cap, 256), torch.bfloat16, cuda)
    vc = Guarded((B, Hkv, cap, 256), torch.bfloat16, cuda)
    kc.t.zero_()
    vc.t.zero_()
    sl = lambda a, b: {k: v[:, a:b].contiguous().to(cuda) for k, v in x.items()}  # noqa: E731
    p0, p1 = sl(0, T0), sl(T0, T0 + T1)
    o0 = Guarded((B, T0, H * 256), torch.bfloat16, cuda)
    ws0 = workspace(fga.spark_attn_prefill_workspace_size(B, T0, H, Hkv, layer), cuda)
    fga.spark_attn_prefill_cache(p0["qkv"], p0["gate"], p0["pos"], kc.t, vc.t, layer, out=o0.t,
                                 workspace=ws0.t)
    o1 = Guarded((B, T1, H * 256), torch.bfloat16, cuda)
    ws1 = workspace(fga.spark_attn_prefill_workspace_size(B, T1, H, Hkv, layer), cuda)
    start = torch.full((B,), T0, dtype=torch.int32, device=cuda)
    fga.spark_attn_prefill_chunk(p1["qkv"], p1["gate"], p1["pos"], kc.t, vc.t, start, layer,
                                 out=o1.t, workspace=ws1.t)
    y = Guarded((B, H * 256), torch.bfloat16, cuda)
    wsd = workspace(fga.spark_attn_decode_workspace_size(B, H, Hkv, cap, layer), cuda)
    t = T0 + T1
    fga.spark_attn_decode(x["qkv"][:, t].contiguous().to(cuda),
                          x["gate"][:, t].contiguous().to(cuda),
                          torch.full((B,), t, dtype=torch.int32, device=cuda), kc.t, vc.t, layer,
                          out=y.t, workspace=wsd.t)
    torch.cuda.synchronize()
    for name, g in (("k cache", kc), ("v cache", vc), ("prefill out", o0), ("chunk out", o1),
                    ("decode out", y), ("prefill ws", ws0), ("chunk ws", ws1), ("decode ws", wsd)):
        assert g.intact(), name
    want = oracle_prefill(x, layer, H, Hkv)          # [B, T0+T1+1, H*256]
    check_close(o1.t, want[:, T0:t], "guarded chunk")
    check_close(y.t, want[:, t], "guarded decode")


def test_block_and_linear_stay_inside_their_buffers(cuda):
    from test_layer_gpu import bits, hidden_states, weights
    B, T, hidden, H, Hkv = 1, 129, 264, 8, 2
    layer = wl.SLIDING_LAYER
    x = hidden_states((B, T, hidden), 51)
    w = weights(hidden, H, Hkv, 52)
    pos = torch.arange(T, dtype=torch.int32)[None]
    y = Guarded((B, T, hidden), torch.bfloat16, cuda)
    ws = workspace(fga.spark_attn_layer_prefill_workspace_size(B, T, hidden, H, Hkv, layer), cuda)
    fga.spark_attn_layer_prefill(x.to(cuda), *[t.to(cuda) for t in w], pos.to(cuda), layer,
                                 y=y.t, workspace=ws.t)
    # a ragged GEMM: M and N not multiples of the 128 x 256 tile
    a = hidden_states((300, 264), 53).to(cuda)
    wt = (torch.randn((200, 264), generator=torch.Generator().manual_seed(54)) / 16).to(
        torch.bfloat16).to(cuda)
    lin = Guarded((300, 200), torch.bfloat16, cuda)
    fga.spark_attn_linear(a, wt, y=lin.t)
    torch.cuda.synchronize()
    assert y.intact() and ws.intact() and lin.intact()
    want = oracle.layer_prefill(bits(x), *[bits(t) for t in w], pos.numpy(), layer.kind,
                                layer.window, layer.theta, layer.rot_dim, H, Hkv)
    check_close(y.t.reshape(B * T, hidden), want.reshape(B * T, hidden), "guarded block")
    ref = (a.float() @ wt.float().T)
    assert float((lin.t.float() - ref).abs().max()) <= 2.0 ** -6 * float(ref.abs().max()) + 1e-3


def test_host_prefill_stays_inside_its_host_buffer(cuda):
    B, T, H, Hkv = 2, 2100, 16, 4            # chunked: 2048 + 52 tokens per sequence
    layer = wl.FULL_LAYER
    x = wl.make_prefill_inputs(wl.PrefillCase("gh", B=B, T=T, H=H, Hkv=Hkv, layer=layer, seed=9))
    out = guarded_host((B, T, H * 256), torch.bfloat16)
    ws = workspace(fga.spark_attn_prefill_host_workspace_size(B, T, H, Hkv, layer), cuda)
    fga.spark_attn_prefill_host(x["qkv"].pin_memory(), x["gate"].pin_memory(),
                                x["pos"].pin_memory(), layer, out=out.t, workspace=ws.t)
    torch.cuda.synchronize()
    assert out.intact() and ws.intact()
    want = fga.spark_attn_prefill(x["qkv"].to(cuda), x["gate"].to(cuda), x["pos"].to(cuda), layer)
    assert torch.equal(out.t, want.cpu())
