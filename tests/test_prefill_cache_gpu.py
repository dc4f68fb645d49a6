"""Prefill that fills the decode cache, then decode continues the sequence
(the prefill -> decode hand-off of past_key_values.update; Spark-X2.5-4B
hybrid-attention explainer, lshu.cn).

A prefill of tokens 0..T-1 with spark_attn_prefill_cache followed by a decode
of token T on the same caches must equal row T of the oracle's prefill over
tokens 0..T.  The cache holds each token's rotated key (within one bf16 ulp
of the fp64 rotation; unrotated dims bit-exact) and its value bit-exact, at
slot t (full layer) or t mod cap (ring, last cap tokens only).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import full_gqa_attention_gb300 as fga
import oracle
import workloads as wl
from parity import bits_to_f64, check_close, check_rotated_bf16

pytestmark = pytest.mark.gpu

FULL, SLIDING = wl.FULL, wl.SLIDING


@pytest.mark.parametrize("kind,T,cap", [(FULL, 300, 301), (FULL, 1000, 4096),
                                        (SLIDING, 300, 512), (SLIDING, 700, 512),
                                        (SLIDING, 1300, 600)])
def test_prefill_then_decode(cuda, kind, T, cap):
    layer = wl.FULL_LAYER if kind == FULL else wl.SLIDING_LAYER
    H, Hkv, B = 16, 4, 2
    case = wl.PrefillCase("pc", B=B, T=T + 1, H=H, Hkv=Hkv, layer=layer, seed=T + cap)
    x = wl.make_prefill_inputs(case)                 # tokens 0..T
    qkv, gate, pos = x["qkv"], x["gate"], x["pos"]
    kc = torch.full((B, Hkv, cap, 256), 5.0, dtype=torch.bfloat16, device=cuda)
    vc = torch.full_like(kc, 5.0)
    pre_in = [qkv[:, :T].contiguous().to(cuda), gate[:, :T].contiguous().to(cuda),
              pos[:, :T].contiguous().to(cuda)]
    out = fga.spark_attn_prefill_cache(*pre_in, kc, vc, layer)
    # the attention output is the plain prefill's, bit for bit
    assert torch.equal(out, fga.spark_attn_prefill(*pre_in, layer))
    # cache contents
    kbits, vbits = wl.bf16_bits(kc), wl.bf16_bits(vc)
    qb = wl.bf16_bits(qkv)
    r = layer.rot_dim
    toks = range(T) if kind == FULL else range(max(0, T - cap), T)
    kx = qb[:, :, H * 256:(H + Hkv) * 256].reshape(B, T + 1, Hkv, 256)
    for t in toks:
        slot = t if kind == FULL else t % cap
        v_want = qb[:, t, (H + Hkv) * 256:].reshape(B, Hkv, 256)
        assert np.array_equal(vbits[:, :, slot], v_want), t
        x64 = bits_to_f64(kx[:, t])
        kd = oracle.rope(x64.reshape(-1, 256), np.full(B * Hkv, int(pos[0, t]), np.int32), r,
                         layer.theta).reshape(B, Hkv, 256)
        assert np.array_equal(kbits[:, :, slot, r:], kx[:, t, :, r:]), t   # unrotated dims
        check_rotated_bf16(kbits[:, :, slot, :r], kd[:, :, :r],
                           np.abs(x64).max(axis=-1, keepdims=True), f"token {t}")
    # decode of token T continues the sequence
    dout = fga.spark_attn_decode(qkv[:, T].contiguous().to(cuda), gate[:, T].contiguous().to(cuda),
                                 pos[:, T].contiguous().to(cuda), kc, vc, layer)
    L = layer
    rows = np.array([b * (T + 1) + T for b in range(B)], np.int64)
    want = oracle.prefill(qb, gate.numpy(), pos.numpy(), L.kind, L.window, L.theta, L.rot_dim, H,
                          Hkv, rows=rows)
    check_close(dout, want, f"prefill_cache -> decode kind={kind} T={T} cap={cap}")


def test_prefill_cache_rejects_small_cache(cuda):
    layer = wl.FULL_LAYER
    q = torch.zeros((1, 64, 24 * 256), dtype=torch.bfloat16, device=cuda)
    g = torch.zeros((1, 64, 16), device=cuda)
    p = torch.zeros((1, 64), dtype=torch.int32, device=cuda)
    kc = torch.zeros((1, 4, 32, 256), dtype=torch.bfloat16, device=cuda)
    with pytest.raises(fga.SparkError) as e:
        fga.spark_attn_prefill_cache(q, g, p, kc, kc.clone(), layer)
    assert e.value.status == 5  # SPARK_ERR_CAPACITY: a full layer needs cap >= T


@pytest.mark.parametrize("kind,T,cap,poison", [(FULL, 200, 2048, False), (FULL, 333, 1100, True),
                                               (SLIDING, 200, 768, False),
                                               (SLIDING, 129, 768, True)])
def test_chunked_prefill(cuda, kind, T, cap, poison):
    """Two sequences with 300 and 700 tokens already cached take a chunk of T
    more tokens in one call (ragged start); the chunk's rows equal the oracle's
    rows of a prefill over the whole sequence, and a decode of the next token
    continues it.  With `poison`, slots never written hold NaN."""
    _chunked(cuda, kind, T, cap, poison, 16, 4)


@pytest.mark.parametrize("kind,cap", [(FULL, 2048), (SLIDING, 768)])
@pytest.mark.parametrize("H,Hkv", [(8, 8), (16, 2)])
def test_chunked_prefill_group_sizes(cuda, kind, cap, H, Hkv):
    """The chunked prefill with groups of 1 and 8 query heads per KV head (the
    kernels built for other group sizes than the models' 4)."""
    _chunked(cuda, kind, 200, cap, False, H, Hkv)


def _chunked(cuda, kind, T, cap, poison, H, Hkv):
    layer = wl.FULL_LAYER if kind == FULL else wl.SLIDING_LAYER
    starts = [300, 700]
    total = max(starts) + T + 1
    case = wl.PrefillCase("chunk", B=2, T=total, H=H, Hkv=Hkv, layer=layer, seed=T + cap)
    x = wl.make_prefill_inputs(case)
    qkv, gate, pos = x["qkv"], x["gate"], x["pos"]
    fill = float("nan") if poison else 0.0
    kc = torch.full((2, Hkv, cap, 256), fill, dtype=torch.bfloat16, device=cuda)
    vc = torch.full_like(kc, fill)
    # cache the first start[b] tokens of each sequence
    for b, s0 in enumerate(starts):
        fga.spark_attn_prefill_cache(qkv[b:b + 1, :s0].contiguous().to(cuda),
                                     gate[b:b + 1, :s0].contiguous().to(cuda),
                                     pos[b:b + 1, :s0].contiguous().to(cuda),
                                     kc[b:b + 1], vc[b:b + 1], layer)
    # one chunk of T tokens for both sequences, at their own offsets
    cq = torch.stack([qkv[b, s0:s0 + T] for b, s0 in enumerate(starts)]).contiguous()
    cg = torch.stack([gate[b, s0:s0 + T] for b, s0 in enumerate(starts)]).contiguous()
    cp = torch.stack([pos[b, s0:s0 + T] for b, s0 in enumerate(starts)]).contiguous()
    start = torch.tensor(starts, dtype=torch.int32, device=cuda)
    ws = fga.new_workspace(fga.spark_attn_prefill_workspace_size(2, T, H, Hkv, layer))
    out = fga.spark_attn_prefill_chunk(cq.to(cuda), cg.to(cuda), cp.to(cuda), kc, vc, start,
                                       layer, workspace=ws)
    assert fga.spark_attn_read_status(ws) == 0
    qb = wl.bf16_bits(qkv)
    L = layer
    for b, s0 in enumerate(starts):
        rows = np.arange(s0, s0 + T, dtype=np.int64)
        want = oracle.prefill(qb[b:b + 1, :s0 + T], gate[b:b + 1, :s0 + T].numpy(),
                              pos[b:b + 1, :s0 + T].numpy(), L.kind, L.window, L.theta,
                              L.rot_dim, H, Hkv, rows=rows)
        check_close(out[b], want, f"chunk b={b} start={s0} kind={kind} T={T} cap={cap}")
    # decode of the next token continues each sequence
    nq = torch.stack([qkv[b, s0 + T] for b, s0 in enumerate(starts)]).contiguous()
    ng = torch.stack([gate[b, s0 + T] for b, s0 in enumerate(starts)]).contiguous()
    npos = torch.tensor([s0 + T for s0 in starts], dtype=torch.int32)
    dout = fga.spark_attn_decode(nq.to(cuda), ng.to(cuda), npos.to(cuda), kc, vc, layer)
    for b, s0 in enumerate(starts):
        want = oracle.prefill(qb[b:b + 1, :s0 + T + 1], gate[b:b + 1, :s0 + T + 1].numpy(),
                              pos[b:b + 1, :s0 + T + 1].numpy(), L.kind, L.window, L.theta,
                              L.rot_dim, H, Hkv, rows=np.array([s0 + T], np.int64))
        check_close(dout[b:b + 1], want, f"decode after chunk b={b} kind={kind}")


def test_chunked_prefill_ring_rules(cuda):
    layer = wl.SLIDING_LAYER
    q = torch.zeros((1, 64, 24 * 256), dtype=torch.bfloat16, device=cuda)
    g = torch.zeros((1, 64, 16), device=cuda)
    p = torch.zeros((1, 64), dtype=torch.int32, device=cuda)
    st = torch.zeros((1,), dtype=torch.int32, device=cuda)
    for cap, code in ((512, 5), (600, 3)):   # too small for the chunk; not a multiple of 128
        kc = torch.zeros((1, 4, cap, 256), dtype=torch.bfloat16, device=cuda)
        with pytest.raises(fga.SparkError) as e:
            fga.spark_attn_prefill_chunk(q, g, p, kc, kc.clone(), st, layer)
        assert e.value.status == code
