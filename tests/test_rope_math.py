"""The kernels' RoPE angle reduction, checked on the CPU.

full_gqa_attention_gb300/csrc/rope_math.cuh holds the reduction of the RoPE
angle pos * theta^(-2k/r) (Spark-X2.5 architecture page, §4) to [-1/2, 1/2]
turns that every kernel runs before sincospif.  tests/rope_check.cpp compiles
that same header with the host compiler and compares it with the angle
evaluated in long double, at the model's two (theta, rotated width) settings
and positions up to 2^24.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "full_gqa_attention_gb300", "csrc")

# The two roundings left after the exact steps are ~2^-25 turns (~2e-7 rad);
# measured 1.96e-7 rad up to 2^24.  A plain fp32 product pos * inv_freq is off
# by up to 0.03 rad at 1M positions.
ROPE_TOL = 2.5e-7


def _build(dirpath: str, out: str):
    subprocess.run(["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-I", dirpath,
                    os.path.join(ROOT, "tests", "rope_check.cpp"), "-o", out], check=True)
    lib = ctypes.CDLL(out)
    lib.rope_max_err.argtypes = [ctypes.c_double, ctypes.c_int, ctypes.c_int, ctypes.c_int]
    lib.rope_max_err.restype = ctypes.c_double
    return lib


@pytest.fixture(scope="module")
def checker(tmp_path_factory):
    return _build(CSRC, str(tmp_path_factory.mktemp("rope") / "rope_check.so"))


@pytest.mark.parametrize("theta,r", [(5e6, 64), (1e4, 256), (1e4, 64), (5e6, 256)])
def test_rope_angles_to_1m(checker, theta, r):
    # every position of the first 4096, then a stride through 1M context
    assert checker.rope_max_err(theta, r, 4096, 1) <= ROPE_TOL
    assert checker.rope_max_err(theta, r, 1 << 20, 997) <= ROPE_TOL


@pytest.mark.parametrize("theta,r", [(5e6, 64), (1e4, 256)])
def test_rope_angles_to_2_24(checker, theta, r):
    assert checker.rope_max_err(theta, r, (1 << 24) - 1, 65521) <= ROPE_TOL


# Mistakes planted in a copy of rope_math.cuh that the checks must catch.
MUTANTS = {
    "low part of the frequency dropped": ("rm_fma(fp, u_lo, e)", "e"),
    "rounding error of the product dropped": ("rm_fma(fp, u_lo, e)", "rm_mul(fp, u_lo)"),
    "rounding error with the wrong sign": ("rm_fma(fp, u_hi, -p)", "rm_fma(fp, u_hi, p)"),
    "whole turns not removed": ("rm_add(p, -rm_rint(p))", "p"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_checks_catch_planted_mistakes(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(os.path.join(CSRC, "rope_math.cuh")).read()
    assert src.count(old) == 1, name
    (tmp_path / "rope_math.cuh").write_text(src.replace(old, new))
    lib = _build(str(tmp_path), str(tmp_path / "mutant.so"))
    worst = max(lib.rope_max_err(5e6, 64, 1 << 20, 9973), lib.rope_max_err(1e4, 256, 1 << 20, 9973))
    assert not worst <= ROPE_TOL, f"planted mistake not caught: {name}"
