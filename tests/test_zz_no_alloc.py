"""spark_attn_decode_noalloc: decode for callers that cannot allocate a
workspace (their device memory belongs to a runtime or plugin host that
passes them only inputs and outputs, or cudaMalloc would synchronize a path
that must not stall).  The call keeps its split-KV scratch in a fixed buffer
inside the library.

This file is collected last on purpose: the buffer is shared by every call,
so the test also shows that results stay right after all other tests ran.
It must pass alone in a fresh process as well.
"""
from __future__ import annotations

import ctypes

import pytest
import torch

import full_gqa_attention_gb300 as fga
import oracle
import workloads as wl
from full_gqa_attention_gb300 import _binding as bnd
from parity import check_close

pytestmark = pytest.mark.gpu


def make_case(cuda, layer, B, H, Hkv, cap, positions, seed):
    case = wl.DecodeCase("t", B=B, H=H, Hkv=Hkv, layer=layer, seed=seed, cap=cap, len_lo=0,
                         len_hi=0)
    step = wl.make_decode_step_inputs(case)
    kc = torch.empty((B, Hkv, cap, 256), dtype=torch.bfloat16, device=cuda)
    vc = torch.empty_like(kc)
    g = torch.Generator(cuda).manual_seed(seed)
    kc.normal_(generator=g)
    vc.normal_(generator=g)
    return {"qkv": step["qkv"].to(cuda), "gate": step["gate"].to(cuda),
            "pos": torch.tensor(positions, dtype=torch.int32, device=cuda),
            "k": kc, "v": vc, "layer": layer}


def oracle_want(c, k_before, v_before):
    """The fp64 oracle's output for a case, from its caches before the call."""
    L = c["layer"]
    H = c["gate"].shape[1]
    Hkv = k_before.shape[1]
    want, _, _ = oracle.decode(wl.bf16_bits(c["qkv"].cpu()), c["gate"].cpu().numpy(),
                               c["pos"].cpu().numpy(), wl.bf16_bits(k_before),
                               wl.bf16_bits(v_before), L.kind, L.window, L.theta, L.rot_dim,
                               H, Hkv, gate_mode=L.gate_mode)
    return want


def test_noalloc_decode_matches_workspace_decode(cuda):
    cases = [
        # 18 splits per (sequence, KV head): the separate merge kernel
        make_case(cuda, wl.FULL_LAYER, 2, 16, 4, 20000, [19999, 7000], seed=1),
        # 8 splits per ring at B=3: the separate merge kernel
        make_case(cuda, wl.SLIDING_LAYER, 3, 16, 4, 512, [600, 511, 40], seed=2),
        # 64 rings: one split each, merged inside the split kernel
        make_case(cuda, wl.SLIDING_LAYER, 64, 16, 4, 512,
                  [513 + 37 * b for b in range(64)], seed=3),
    ]
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    # calls in a row, on different shapes, each against the workspace path and
    # the fp64 oracle
    for c in cases:
        k_before, v_before = c["k"].cpu(), c["v"].cpu()
        k_ref, v_ref = c["k"].clone(), c["v"].clone()
        want = fga.spark_attn_decode(c["qkv"], c["gate"], c["pos"], k_ref, v_ref, c["layer"])
        got = fga.spark_attn_decode_noalloc(c["qkv"], c["gate"], c["pos"], c["k"], c["v"],
                                            c["layer"], device_status=status)
        torch.cuda.synchronize()
        what = f"no-alloc decode kind={c['layer'].kind} B={c['qkv'].shape[0]}"
        check_close(got, want, what + " vs workspace decode")
        check_close(got, oracle_want(c, k_before, v_before), what + " vs oracle")
        assert torch.equal(c["k"], k_ref) and torch.equal(c["v"], v_ref), "cache update differs"
    assert int(status.item()) == 0


def test_noalloc_decode_rejects_work_beyond_its_buffer(cuda):
    """Work whose split-KV state exceeds the fixed buffer is refused up front."""
    layer = wl.FULL_LAYER
    B, H, Hkv, cap = 64, 16, 4, 131073
    need = fga.spark_attn_decode_workspace_size(B, H, Hkv, cap, layer)
    assert need > fga.SPARK_NOALLOC_SCRATCH_BYTES
    qkv = torch.zeros((B, (H + 2 * Hkv) * 256), dtype=torch.bfloat16, device=cuda)
    k = torch.zeros((B, Hkv, 16, 256), dtype=torch.bfloat16, device=cuda)  # never read
    out = torch.full((B, H * 256), 3.0, dtype=torch.bfloat16, device=cuda)
    d = fga.as_desc(layer)
    st = fga.lib.spark_attn_decode_noalloc(
        ctypes.c_void_p(qkv.data_ptr()), ctypes.c_void_p(qkv.data_ptr()),
        ctypes.c_void_p(qkv.data_ptr()), ctypes.c_void_p(k.data_ptr()),
        ctypes.c_void_p(k.data_ptr()), cap, ctypes.byref(d), B, H, Hkv,
        ctypes.c_void_p(out.data_ptr()), None, None)
    assert st == bnd.SPARK_ERR_WORKSPACE
    assert torch.all(out == 3.0)
