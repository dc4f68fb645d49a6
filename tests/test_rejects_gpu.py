"""Rejected calls change nothing on the device (through the C ABI).

The CPU tests (test_abi.py) check the status each invalid argument returns.
Here the same kinds of calls get real device buffers, each pre-filled with a
byte pattern: a rejected call must return its status and leave the output,
the KV caches and the workspace exactly as they were, so nothing was
enqueued.  A valid call on the same buffers then does change them.
"""
from __future__ import annotations

import ctypes

import pytest
import torch

import full_gqa_attention_gb300 as fga
from full_gqa_attention_gb300 import _binding as bnd

pytestmark = pytest.mark.gpu

B, T, H, Hkv, CAP = 2, 64, 16, 4, 512
P = ctypes.c_void_p


def desc(kind=1, window=512, theta=1e4, rot=256, gate=0):
    return fga.layer_desc(kind, window, theta, rot, gate)


@pytest.fixture
def bufs(cuda):
    g = torch.Generator(device=cuda).manual_seed(3)
    b = {
        "qkv": torch.randn((B, T, (H + 2 * Hkv) * 256), generator=g, device=cuda).to(
            torch.bfloat16),
        "gate": torch.randn((B, T, H), generator=g, device=cuda),
        "pos": torch.arange(T, dtype=torch.int32, device=cuda).repeat(B, 1).contiguous(),
        "out": torch.full((B, T, H * 256), 3.0, dtype=torch.bfloat16, device=cuda),
        "k": torch.full((B, Hkv, CAP, 256), 5.0, dtype=torch.bfloat16, device=cuda),
        "v": torch.full((B, Hkv, CAP, 256), 6.0, dtype=torch.bfloat16, device=cuda),
        "ws": torch.full((1 << 24,), 0x5A, dtype=torch.uint8, device=cuda),
    }
    b["snap"] = {k: v.clone() for k, v in b.items()}
    return b


def unchanged(b) -> bool:
    torch.cuda.synchronize()
    return all(torch.equal(b[k], b["snap"][k]) for k in ("out", "k", "v", "ws"))


def ptr(t, offset=0):
    return P(t.data_ptr() + offset)


def prefill(b, d, h=H, hkv=Hkv, out_off=0, ws_off=0, ws_bytes=None):
    return fga.lib.spark_attn_prefill(ptr(b["qkv"]), ptr(b["gate"]), ptr(b["pos"]),
                                      ctypes.byref(d), B, T, h, hkv, ptr(b["out"], out_off),
                                      ptr(b["ws"], ws_off),
                                      b["ws"].numel() - ws_off if ws_bytes is None else ws_bytes,
                                      None)


def prefill_cache(b, d, cap=CAP, k_off=0):
    return fga.lib.spark_attn_prefill_cache(ptr(b["qkv"]), ptr(b["gate"]), ptr(b["pos"]),
                                            ptr(b["k"], k_off), ptr(b["v"]), cap, ctypes.byref(d),
                                            B, T, H, Hkv, ptr(b["out"]), ptr(b["ws"]),
                                            b["ws"].numel(), None)


def decode(b, d, cap=CAP, v_off=0, ws_bytes=None):
    qkv1 = b["qkv"][:, 0].contiguous()
    gate1 = b["gate"][:, 0].contiguous()
    pos1 = torch.full((B,), T, dtype=torch.int32, device=b["qkv"].device)
    st = fga.lib.spark_attn_decode(ptr(qkv1), ptr(gate1), ptr(pos1), ptr(b["k"]),
                                   ptr(b["v"], v_off), cap, ctypes.byref(d), B, H, Hkv,
                                   ptr(b["out"]), ptr(b["ws"]),
                                   b["ws"].numel() if ws_bytes is None else ws_bytes, None)
    return st


CASES = [
    ("prefill: H % Hkv != 0", lambda b: prefill(b, desc(), hkv=3), bnd.SPARK_ERR_SHAPE),
    ("prefill: group of 3", lambda b: prefill(b, desc(), h=12), bnd.SPARK_ERR_UNSUPPORTED),
    ("prefill: window 0", lambda b: prefill(b, desc(window=0)), bnd.SPARK_ERR_SHAPE),
    ("prefill: rot_dim 40", lambda b: prefill(b, desc(rot=40)), bnd.SPARK_ERR_UNSUPPORTED),
    ("prefill: gate mode 2", lambda b: prefill(b, desc(gate=2)), bnd.SPARK_ERR_UNSUPPORTED),
    ("prefill: output not 16-byte aligned", lambda b: prefill(b, desc(), out_off=2),
     bnd.SPARK_ERR_ALIGN),
    ("prefill: workspace not 256-byte aligned", lambda b: prefill(b, desc(), ws_off=16),
     bnd.SPARK_ERR_ALIGN),
    ("prefill: workspace too small", lambda b: prefill(b, desc(), ws_bytes=1024),
     bnd.SPARK_ERR_WORKSPACE),
    ("prefill_cache: ring smaller than its window", lambda b: prefill_cache(b, desc(), cap=256),
     bnd.SPARK_ERR_CAPACITY),
    ("prefill_cache: key cache not aligned", lambda b: prefill_cache(b, desc(), k_off=8),
     bnd.SPARK_ERR_ALIGN),
    ("decode: ring smaller than its window", lambda b: decode(b, desc(), cap=100),
     bnd.SPARK_ERR_CAPACITY),
    ("decode: value cache not aligned", lambda b: decode(b, desc(), v_off=4), bnd.SPARK_ERR_ALIGN),
    ("decode: workspace too small", lambda b: decode(b, desc(), ws_bytes=256),
     bnd.SPARK_ERR_WORKSPACE),
    ("decode: theta 0", lambda b: decode(b, desc(theta=0.0)), bnd.SPARK_ERR_SHAPE),
]


@pytest.mark.parametrize("name,call,code", CASES, ids=[c[0] for c in CASES])
def test_rejected_call_changes_nothing(bufs, name, call, code):
    assert call(bufs) == code
    assert unchanged(bufs), name


def test_a_valid_call_on_the_same_buffers_does_write(bufs):
    bufs["ws"].zero_()
    bufs["snap"]["ws"] = bufs["ws"].clone()
    assert prefill_cache(bufs, desc()) == bnd.SPARK_OK
    torch.cuda.synchronize()
    assert not torch.equal(bufs["out"], bufs["snap"]["out"])
    assert not torch.equal(bufs["k"], bufs["snap"]["k"])
    assert fga.spark_attn_read_status(bufs["ws"]) == 0
