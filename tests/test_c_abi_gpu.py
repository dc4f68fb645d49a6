"""The C ABI used from C++ alone (tests/c_abi_example.cpp), without Python.

The program allocates its own device buffers, runs a sliding-layer prefill
that fills a 512-slot ring and one decode step over it, checks that an invalid
head count is refused on the host, and reads the status word.  Its outputs
must equal, bit for bit, those of the same calls made through the Python
binding on the same inputs.
"""
from __future__ import annotations

import os
import subprocess

import numpy as np
import pytest
import torch

import full_gqa_attention_gb300 as fga
import workloads as wl
from full_gqa_attention_gb300 import build as lib_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def compile_example(out_dir) -> str:
    exe = os.path.join(str(out_dir), "c_abi_example")
    lib_dir = os.path.dirname(lib_build.build())
    subprocess.run([lib_build._nvcc(), "-O2", "-std=c++17", "-I", lib_build.INCLUDE,
                    os.path.join(ROOT, "tests", "c_abi_example.cpp"), "-o", exe,
                    "-L", lib_dir, "-lspark_attn", "-Xlinker", "-rpath=" + lib_dir], check=True)
    return exe


def test_example_builds_against_the_header(tmp_path):
    """Host-side check: the program compiles and links against the library."""
    assert os.path.exists(compile_example(tmp_path))


@pytest.mark.gpu
@pytest.mark.parametrize("B,T", [(1, 700), (3, 300)])
def test_c_program_matches_the_binding(cuda, tmp_path, B, T):
    H, Hkv = 16, 4
    layer = wl.SLIDING_LAYER
    x = wl.make_prefill_inputs(wl.PrefillCase("c", B=B, T=T, H=H, Hkv=Hkv, layer=layer,
                                              seed=80 + T))
    g = torch.Generator().manual_seed(81 + T)
    qkv1 = torch.randn((B, (H + 2 * Hkv) * 256), generator=g).to(torch.bfloat16)
    gate1 = torch.randn((B, H), generator=g)
    pos1 = torch.full((B,), T, dtype=torch.int32)
    for name, t in (("qkv", x["qkv"]), ("gate", x["gate"]), ("pos", x["pos"]),
                    ("qkv1", qkv1), ("gate1", gate1), ("pos1", pos1)):
        raw = t.contiguous().view(torch.int16) if t.dtype == torch.bfloat16 else t.contiguous()
        raw.numpy().tofile(str(tmp_path / f"{name}.bin"))
    exe = compile_example(tmp_path)
    run = subprocess.run([exe, str(tmp_path), str(B), str(T), str(H), str(Hkv)],
                         capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, run.stderr + run.stdout
    assert run.stdout.startswith("ok status=0")
    out_c = np.fromfile(str(tmp_path / "out.bin"), dtype=np.int16).reshape(B, T, H * 256)
    y_c = np.fromfile(str(tmp_path / "y.bin"), dtype=np.int16).reshape(B, H * 256)
    # the same calls through the binding
    kc = torch.empty((B, Hkv, 512, 256), dtype=torch.bfloat16, device=cuda)
    vc = torch.empty_like(kc)
    out = fga.spark_attn_prefill_cache(x["qkv"].to(cuda), x["gate"].to(cuda), x["pos"].to(cuda),
                                       kc, vc, layer)
    y = fga.spark_attn_decode(qkv1.to(cuda), gate1.to(cuda), pos1.to(cuda), kc, vc, layer)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().view(torch.int16).numpy(), out_c)
    assert np.array_equal(y.cpu().view(torch.int16).numpy(), y_c)
