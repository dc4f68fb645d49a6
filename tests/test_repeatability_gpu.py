"""Run-to-run repeatability of the kernels on grids of many waves.

Every output element is computed in a fixed order: a query tile visits its
key tiles in ascending order, and the split-KV states of a decode step are
merged in a fixed order.  So the result must not depend on how the hardware
schedules CTAs.  A copy running on a second stream takes SMs and memory
bandwidth away at unpredictable moments and reorders the CTAs of the grid;
the output must stay bit-identical, run after run.
"""
from __future__ import annotations

import pytest
import torch

import full_gqa_attention_gb300 as fga
import workloads as wl

pytestmark = pytest.mark.gpu

RUNS_PLAIN, RUNS_CONTENDED = 2, 3


class Contention:
    """Back-to-back 256 MB copies on a side stream, enqueued just before the
    call under test so that both run at the same time."""

    def __init__(self, cuda):
        self.stream = torch.cuda.Stream(cuda)
        self.a = torch.empty(128 << 20, dtype=torch.bfloat16, device=cuda).normal_()
        self.b = torch.empty_like(self.a)

    def start(self, n=6):
        self.stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(self.stream):
            for _ in range(n):
                self.b.copy_(self.a)

    def finish(self):
        torch.cuda.current_stream().wait_stream(self.stream)


def repeat_and_compare(cuda, call):
    first = call().clone()
    torch.cuda.synchronize()
    load = Contention(cuda)
    for i in range(RUNS_PLAIN + RUNS_CONTENDED):
        contended = i >= RUNS_PLAIN
        if contended:
            load.start()
        out = call()
        if contended:
            load.finish()
        torch.cuda.synchronize()
        assert torch.equal(out, first), f"run {i + 1} differs (contended={contended})"


def prefill_inputs(cuda, B, T, H, Hkv, seed):
    g = torch.Generator(cuda).manual_seed(seed)
    qkv = torch.randn((B, T, (H + 2 * Hkv) * 256), generator=g, device=cuda).to(torch.bfloat16)
    gate = torch.randn((B, T, H), generator=g, device=cuda)
    pos = torch.arange(T, dtype=torch.int32, device=cuda).repeat(B, 1).contiguous()
    return qkv, gate, pos


@pytest.mark.parametrize("layer", [wl.FULL_LAYER, wl.SLIDING_LAYER], ids=["full", "sliding"])
def test_prefill_4b_B2_T8192_repeatable_under_contention(cuda, layer):
    """2048 CTAs (256 query tiles x 4 KV heads x 2 sequences): about 13 waves."""
    B, T, H, Hkv = 2, 8192, 16, 4
    qkv, gate, pos = prefill_inputs(cuda, B, T, H, Hkv, seed=21)
    ws = fga.new_workspace(fga.spark_attn_prefill_workspace_size(B, T, H, Hkv, layer))
    out = torch.empty((B, T, H * 256), dtype=torch.bfloat16, device=cuda)
    repeat_and_compare(cuda, lambda: fga.spark_attn_prefill(qkv, gate, pos, layer, out=out,
                                                            workspace=ws))
    assert fga.spark_attn_read_status(ws) == 0


@pytest.mark.parametrize("layer,cap", [(wl.FULL_LAYER, 40000), (wl.SLIDING_LAYER, 512)],
                         ids=["full", "ring"])
def test_decode_split_kv_repeatable_under_contention(cuda, layer, cap):
    """Split-KV decode of 6 sequences: the full layer splits each (sequence,
    KV head) into several chunks whose states the merge combines."""
    B, H, Hkv = 6, 16, 4
    g = torch.Generator(cuda).manual_seed(22)
    qkv = torch.randn((B, (H + 2 * Hkv) * 256), generator=g, device=cuda).to(torch.bfloat16)
    gate = torch.randn((B, H), generator=g, device=cuda)
    k = torch.randn((B, Hkv, cap, 256), generator=g, device=cuda).to(torch.bfloat16)
    v = torch.randn((B, Hkv, cap, 256), generator=g, device=cuda).to(torch.bfloat16)
    hi = cap - 1 if layer.kind == wl.FULL else 5000
    pos = torch.tensor([hi, 17, hi // 2, 4095, 4096, 511], dtype=torch.int32, device=cuda)
    ws = fga.new_workspace(fga.spark_attn_decode_workspace_size(B, H, Hkv, cap, layer))
    out = torch.empty((B, H * 256), dtype=torch.bfloat16, device=cuda)
    # the step writes the new token's K/V at slot(pos); repeating it rewrites
    # the same values, so every run sees the same cache
    repeat_and_compare(cuda, lambda: fga.spark_attn_decode(qkv, gate, pos, k, v, layer, out=out,
                                                           workspace=ws))
    assert fga.spark_attn_read_status(ws) == 0
