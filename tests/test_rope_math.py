"""The kernels' RoPE angle arithmetic, checked on the CPU.

full_gqa_attention_gb300/csrc/rope_math.cuh holds the cos/sin of the RoPE
angle pos * theta^(-2k/r) (Spark-X2.5 architecture page, §4) that every kernel
uses: an exact reduction of the angle in turns, then sin and cos from a
quadrant split and their Taylor series on |x| <= pi/4.  tests/rope_check.cpp
compiles that same header with the host compiler and compares it with the
angle evaluated in long double, at the model's two (theta, rotated width)
settings and positions up to 2^24.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "full_gqa_attention_gb300", "csrc")

# fp32 evaluation leaves ~1.5 ulps of 1 (measured 8.7e-8); the reduction adds
# ~2^-25 turns (measured 2.0e-7 up to 2^24).  Both sit far inside a bf16 ulp
# (2^-8 relative), and tight enough that dropping the x^9 term of sin
# (3e-7 at pi/4) fails.
SINCOS_TOL = 1.5e-7
ROPE_TOL = 3e-7


def _build(dirpath: str, out: str):
    subprocess.run(["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-I", dirpath,
                    os.path.join(ROOT, "tests", "rope_check.cpp"), "-o", out], check=True)
    lib = ctypes.CDLL(out)
    lib.sincos_turns_max_err.argtypes = [ctypes.c_int]
    lib.sincos_turns_max_err.restype = ctypes.c_double
    lib.rope_max_err.argtypes = [ctypes.c_double, ctypes.c_int, ctypes.c_int, ctypes.c_int]
    lib.rope_max_err.restype = ctypes.c_double
    return lib


@pytest.fixture(scope="module")
def checker(tmp_path_factory):
    return _build(CSRC, str(tmp_path_factory.mktemp("rope") / "rope_check.so"))


def test_sincos_turns(checker):
    err = checker.sincos_turns_max_err(200000)
    assert err <= SINCOS_TOL, err


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
    "cos sign in the odd quadrants": ("c = ((iq + 1) & 2) ? -b : b;", "c = (iq & 2) ? -b : b;"),
    "x^9 term of sin dropped": ("float sp = rm::S9;", "float sp = 0.0f;"),
    "x^8 term of cos dropped": ("cp = rm_fma(cp, r2, rm::C8);", "cp = rm_fma(cp, r2, 0.0f);"),
    "low part of the frequency dropped": ("rm_fma(fp, u_lo, e)", "e"),
    "rounding error of the product dropped": ("rm_fma(fp, u_lo, e)", "rm_mul(fp, u_lo)"),
    "quarter-turn step": ("rm_fma(q, -0.25f, t)", "rm_fma(q, -0.5f, t)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_checks_catch_planted_mistakes(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(os.path.join(CSRC, "rope_math.cuh")).read()
    assert src.count(old) == 1, name
    (tmp_path / "rope_math.cuh").write_text(src.replace(old, new))
    lib = _build(str(tmp_path), str(tmp_path / "mutant.so"))
    sincos = lib.sincos_turns_max_err(20000)
    rope = max(lib.rope_max_err(5e6, 64, 1 << 20, 9973), lib.rope_max_err(1e4, 256, 1 << 20, 9973))
    assert not (sincos <= SINCOS_TOL and rope <= ROPE_TOL), f"planted mistake not caught: {name}"
