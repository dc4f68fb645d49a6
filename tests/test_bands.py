"""The kernels' integer band logic, checked exhaustively on the CPU.

full_gqa_attention_gb300/csrc/bands.cuh holds the functions the prefill and
decode kernels use to pick key tiles, decide which tiles need a per-element
mask, and which ring slots a decode step sees.  tests/band_check.cpp compiles
that same header with the host compiler and checks it against the mask
definition (Spark-X2.5 architecture page, §2: causal, and 0 <= i - j < window
on sliding layers; ring semantics after the lshu.cn explainer's cache
truncation) for every query tile of every length up to 70k tokens.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "full_gqa_attention_gb300", "csrc")
FULL, SLIDING = 0, 1


@pytest.fixture(scope="module")
def checker(tmp_path_factory):
    out = str(tmp_path_factory.mktemp("bands") / "band_check.so")
    subprocess.run(["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-I", CSRC,
                    os.path.join(ROOT, "tests", "band_check.cpp"), "-o", out], check=True)
    lib = ctypes.CDLL(out)
    for fn in (lib.check_key_tiles, lib.check_tile_masks):
        fn.argtypes = [ctypes.c_int] * 6
        fn.restype = ctypes.c_longlong
    lib.check_ring.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_longlong]
    lib.check_ring.restype = ctypes.c_longlong
    return lib


# (kind, window): the two layer types of the model and the windows the
# parity tests use, including ones smaller and larger than a key tile
LAYERS = [(FULL, 0), (SLIDING, 512), (SLIDING, 1), (SLIDING, 7), (SLIDING, 127),
          (SLIDING, 128), (SLIDING, 129), (SLIDING, 513), (SLIDING, 4096)]
TQ = [16, 32, 64, 128]          # tokens per query tile for G = 8, 4, 2, 1


@pytest.mark.parametrize("kind,window", LAYERS)
@pytest.mark.parametrize("tq", TQ)
def test_key_tiles_every_length_to_70k(checker, kind, window, tq):
    assert checker.check_key_tiles(kind, window, tq, 70000, 0, 0) == 0


@pytest.mark.parametrize("kind,window", LAYERS)
@pytest.mark.parametrize("start", [1, 300, 511, 4096])
def test_key_tiles_chunked(checker, kind, window, start):
    # chunked prefill: queries at start + t; ring reads use 128-aligned tiles
    aligned = 1 if kind == SLIDING else 0
    assert checker.check_key_tiles(kind, window, 32, 6000, start, aligned) == 0


@pytest.mark.parametrize("kind,window", LAYERS)
@pytest.mark.parametrize("tq", TQ)
def test_tile_masks(checker, kind, window, tq):
    assert checker.check_tile_masks(kind, window, tq, 1300, 0, 0) == 0


# chunk offsets that put a tile edge one key past a query tile's first query
# (start = 94: 94 + 32 = 126 = 128 - 2) and ring-aligned tiles that start
# exactly `window` keys before a query tile's last query
CHUNKED = [(94, 0), (30, 0), (300, 0), (700, 1), (1000, 1), (833, 1)]


@pytest.mark.parametrize("kind,window", [(FULL, 0), (SLIDING, 512), (SLIDING, 7),
                                         (SLIDING, 130)])
@pytest.mark.parametrize("start,aligned", CHUNKED)
def test_tile_masks_chunked(checker, kind, window, start, aligned):
    assert checker.check_tile_masks(kind, window, 32, 900, start, aligned) == 0


@pytest.mark.parametrize("cap,window", [(512, 512), (600, 512), (512, 7), (1024, 1), (128, 100)])
def test_ring_slots(checker, cap, window):
    assert checker.check_ring(cap, window, 3 * cap + 5) == 0


# Mistakes planted in a copy of bands.cuh that the checks above must catch.
MUTANTS = {
    "window edge of the first tile": ("a0 - window + 1 > 0 ? a0 - window + 1 : 0",
                                      "a0 - window + 2 > 0 ? a0 - window + 2 : 0"),
    "mask skipped at the window edge": ("a_last - key0 >= window", "a_last - key0 > window"),
    "mask skipped on the diagonal": ("key0 + tile - 1 > a0", "key0 + tile - 1 > a0 + 1"),
    "ring slot one token too old": ("return pos - j < static_cast<long long>(window);",
                                    "return pos - j <= static_cast<long long>(window);"),
    "full cache scans the new slot": ("return (kind == kLayerFull) ? pos :",
                                      "return (kind == kLayerFull) ? pos + 1 :"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_checks_catch_planted_mistakes(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(os.path.join(CSRC, "bands.cuh")).read()
    assert src.count(old) == 1, name
    (tmp_path / "bands.cuh").write_text(src.replace(old, new))
    out = str(tmp_path / "mutant.so")
    subprocess.run(["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-I", str(tmp_path),
                    os.path.join(ROOT, "tests", "band_check.cpp"), "-o", out], check=True)
    lib = ctypes.CDLL(out)
    for fn in (lib.check_key_tiles, lib.check_tile_masks):
        fn.argtypes = [ctypes.c_int] * 6
        fn.restype = ctypes.c_longlong
    lib.check_ring.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_longlong]
    lib.check_ring.restype = ctypes.c_longlong
    failures = (lib.check_key_tiles(SLIDING, 512, 32, 3000, 0, 0)
                + lib.check_tile_masks(SLIDING, 512, 32, 1300, 0, 0)
                + lib.check_tile_masks(FULL, 0, 32, 600, 0, 0)
                + lib.check_ring(512, 512, 1600))
    for kind, window in ((FULL, 0), (SLIDING, 512), (SLIDING, 130)):
        for start, aligned in CHUNKED:
            failures += lib.check_tile_masks(kind, window, 32, 900, start, aligned)
    assert failures > 0, f"planted mistake not caught: {name}"
