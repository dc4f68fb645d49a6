"""The library's bounded on-chip waits, driven to their limit on the GPU.

Every pipeline wait in the library's kernels goes through mbar_wait
(csrc/ptx.cuh): it gives up after a time limit instead of hanging, sets
SPARK_DEVERR_TIMEOUT in the workspace status word and lets the kernel drain
and return.  tests/wait_probe.cu runs that helper on a barrier that nothing
completes (a flag that nothing sets), so the wait must run out; the test
checks the status bit, that every waiting thread returned, that the limit was
respected, and that the context still runs the library correctly afterwards.
No GPU fault is involved: the wait ends by itself.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import time

import pytest
import torch

import full_gqa_attention_gb300 as fga
from full_gqa_attention_gb300 import build as lib_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROBE = os.path.join(ROOT, "tests", "wait_probe.cu")


def compile_probe(out_dir) -> str:
    out = os.path.join(str(out_dir), "wait_probe.so")
    subprocess.run([lib_build._nvcc(), *lib_build.ARCH, *lib_build.NVCC_FLAGS, "-shared",
                    PROBE, "-o", out], check=True)
    return out


def test_probe_compiles(tmp_path):
    """Host-side check: the probe builds against the library's headers."""
    assert os.path.exists(compile_probe(tmp_path))


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    lib = ctypes.CDLL(compile_probe(tmp_path_factory.mktemp("probe")))
    lib.wait_probe.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
    lib.wait_probe.restype = ctypes.c_int
    return lib


def run_probe(probe, cuda, arrive):
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    result = torch.zeros(3, dtype=torch.int32, device=cuda)
    torch.cuda.synchronize()
    t0 = time.monotonic()
    rc = probe.wait_probe(ctypes.c_void_p(status.data_ptr()), ctypes.c_void_p(result.data_ptr()),
                          arrive, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return rc, int(status.item()), result.tolist(), time.monotonic() - t0


@pytest.mark.gpu
def test_wait_that_nothing_completes_gives_up_and_reports(cuda, probe):
    rc, status, (done, gave_up, longest_us), wall = run_probe(probe, cuda, arrive=0)
    assert rc == 0
    assert status == fga.SPARK_DEVERR_TIMEOUT
    assert (done, gave_up) == (0, 32), "every waiting thread must return, none completed"
    # the limit is 2 s of %globaltimer; the first thread to give up releases the others
    assert 1.9e6 <= longest_us <= 2.5e6, longest_us
    assert wall < 30.0
    # the context is intact: a library call right after runs and reports no fault
    from test_prefill_gpu import run  # noqa: E402  (the prefill parity helper)
    import workloads as wl
    run(cuda, wl.PrefillCase("after-timeout", B=1, T=200, H=8, Hkv=2,
                             layer=wl.SLIDING_LAYER, seed=3))


@pytest.mark.gpu
def test_wait_whose_phase_completes_returns_at_once(cuda, probe):
    rc, status, (done, gave_up, longest_us), _ = run_probe(probe, cuda, arrive=1)
    assert rc == 0
    assert status == 0
    assert (done, gave_up) == (32, 0)
    assert longest_us < 100_000
