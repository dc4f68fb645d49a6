"""GPU parity of the projection GEMM (spark_attn_linear, tcgen05) against a
plain PyTorch fp32 product of the same bf16 operands.

y = bf16(x W^T): the kernel accumulates in fp32 in another order than the
reference, so a value whose fp32 sum lies next to a bf16 rounding boundary
may round the other way: the bar is one bf16 ulp, element by element, plus
an absolute floor for results that cancel to near zero.
Shapes: the attention block's projections (Spark-X2.5 architecture §6:
2560 -> 6144, 4096 -> 2560; 1.7B: 2048 -> 3072), row counts that leave a
ragged last tile, and N / K that are not multiples of the tile.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import full_gqa_attention_gb300 as fga
from parity import bf16_ulp_diff

pytestmark = pytest.mark.gpu


def ref_product(x, w):
    return x.float() @ w.float().T


def check_gemm(got, ref, what):
    want = ref.to(torch.bfloat16)
    gb = got.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    wb = want.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    ulp = bf16_ulp_diff(gb, wb)
    err = (got.float() - ref).abs()
    # one ulp, or an absolute floor of 2^-14 of the row's largest magnitude
    floor = ref.abs().amax(dim=-1, keepdim=True) * 2.0 ** -14
    bad = (torch.as_tensor(ulp > 1, device=err.device)) & (err > floor)
    assert not bool(bad.any()), f"{what}: {int(bad.sum())} elements off by more than 1 ulp"


def run(cuda, M, N, K, seed, scale=1.0):
    g = torch.Generator(cuda).manual_seed(seed)
    x = torch.randn((M, K), generator=g, device=cuda).to(torch.bfloat16)
    w = (torch.randn((N, K), generator=g, device=cuda) * scale / K ** 0.5).to(torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    y = fga.spark_attn_linear(x, w, device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return x, w, y


@pytest.mark.parametrize("M", [1, 9, 127, 128, 129, 300, 1000])
@pytest.mark.parametrize("N,K", [(6144, 2560), (2560, 4096), (3072, 2048), (264, 72)])
def test_linear_shapes(cuda, M, N, K):
    x, w, y = run(cuda, M, N, K, seed=M * 7 + N + K)
    check_gemm(y, ref_product(x, w), f"M={M} N={N} K={K}")


def test_linear_full_size(cuda):
    """The benchmark's q_k_v_proj (16384 x 2560 -> 6144) and out_proj
    (16384 x 4096 -> 2560), every element."""
    for (M, N, K) in ((16384, 6144, 2560), (16384, 2560, 4096)):
        x, w, y = run(cuda, M, N, K, seed=N)
        for r0 in range(0, M, 4096):
            check_gemm(y[r0:r0 + 4096], ref_product(x[r0:r0 + 4096], w),
                       f"M={M} N={N} K={K} rows {r0}..")


def test_linear_repeatable_and_tiles_independent(cuda):
    """The same product twice gives the same bits; and rows computed in a
    larger call equal the same rows computed alone (each output tile depends
    only on its own rows and columns)."""
    x, w, y1 = run(cuda, 700, 2560, 4096, seed=3)
    y2 = fga.spark_attn_linear(x, w)
    y3 = fga.spark_attn_linear(x[128:256].contiguous(), w)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
    assert torch.equal(y1[128:256], y3)


def test_linear_empty_and_rejections(cuda):
    x = torch.empty((0, 64), dtype=torch.bfloat16, device=cuda)
    w = torch.zeros((16, 64), dtype=torch.bfloat16, device=cuda)
    assert fga.spark_attn_linear(x, w).shape == (0, 16)
    # N not a multiple of 8
    with pytest.raises(fga.SparkError):
        fga.spark_attn_linear(torch.zeros((4, 64), dtype=torch.bfloat16, device=cuda),
                              torch.zeros((12, 64), dtype=torch.bfloat16, device=cuda))
