"""CPU tests of the C ABI: the library loads, exports what the header
declares, and rejects bad arguments on the host before any launch.

No call here reaches the device: every call carries an argument that the
host-side checks refuse first (or is an empty call, which launches nothing).
"""
from __future__ import annotations

import ctypes
import os
import re

import pytest

import full_gqa_attention_gb300 as fga
from full_gqa_attention_gb300 import _binding as bnd

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "spark_attn.h")

FAKE = 0x10000  # an aligned address that is never dereferenced: each call below
                # is refused on the host before any pointer is used


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spark_\w+)\s*\(", text)))


def test_library_exports_every_declared_function():
    names = declared_functions()
    assert "spark_attn_prefill" in names and "spark_attn_decode" in names
    for n in names:
        assert hasattr(fga.lib, n), f"{n} declared in the header but not exported"


def test_status_strings_and_version():
    seen = set()
    for s in range(9):
        msg = fga.spark_status_str(s)
        assert msg and msg not in seen
        seen.add(msg)
    assert re.fullmatch(r"\d+\.\d+\.\d+", fga.spark_attn_version())


def desc(kind=1, window=512, theta=1e4, rot=256, gate=0):
    return bnd.spark_layer_desc(kind, window, theta, rot, gate)


def decode_call(d=None, B=2, H=16, Hkv=4, cap=512, ptrs=None, ws_bytes=1 << 30, null_desc=False):
    p = [FAKE] * 7 if ptrs is None else ptrs
    dd = None if null_desc else ctypes.byref(d or desc())
    return fga.lib.spark_attn_decode(p[0], p[1], p[2], p[3], p[4], cap, dd, B, H, Hkv, p[5],
                                     p[6], ws_bytes, None)


def prefill_call(d=None, B=1, T=64, H=16, Hkv=4, ptrs=None, ws_bytes=1 << 30, null_desc=False):
    p = [FAKE] * 5 if ptrs is None else ptrs
    dd = None if null_desc else ctypes.byref(d or desc(kind=0, window=0, theta=5e6, rot=64))
    return fga.lib.spark_attn_prefill(p[0], p[1], p[2], dd, B, T, H, Hkv, p[3], p[4],
                                      ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(null_desc=True), bnd.SPARK_ERR_NULL),
    (dict(H=16, Hkv=3), bnd.SPARK_ERR_SHAPE),
    (dict(H=12, Hkv=4), bnd.SPARK_ERR_UNSUPPORTED),          # G = 3
    (dict(H=32, Hkv=2), bnd.SPARK_ERR_UNSUPPORTED),          # G = 16
    (dict(B=-1), bnd.SPARK_ERR_SHAPE),
    (dict(d=desc(window=0)), bnd.SPARK_ERR_SHAPE),
    (dict(d=desc(rot=63)), bnd.SPARK_ERR_SHAPE),
    (dict(d=desc(rot=258)), bnd.SPARK_ERR_SHAPE),
    (dict(d=desc(rot=8)), bnd.SPARK_ERR_UNSUPPORTED),
    (dict(d=desc(theta=0.0)), bnd.SPARK_ERR_SHAPE),
    (dict(d=desc(gate=2)), bnd.SPARK_ERR_UNSUPPORTED),
    (dict(d=desc(kind=2)), bnd.SPARK_ERR_SHAPE),
    (dict(cap=511), bnd.SPARK_ERR_CAPACITY),                 # ring smaller than the window
    (dict(cap=0, d=desc(kind=0, window=0, theta=5e6, rot=64)), bnd.SPARK_ERR_CAPACITY),
    (dict(ptrs=[FAKE, 0, FAKE, FAKE, FAKE, FAKE, FAKE]), bnd.SPARK_ERR_NULL),
    (dict(ptrs=[FAKE] * 6 + [0]), bnd.SPARK_ERR_NULL),
    (dict(ptrs=[FAKE + 2] + [FAKE] * 6), bnd.SPARK_ERR_ALIGN),
    (dict(ptrs=[FAKE] * 3 + [FAKE + 8] + [FAKE] * 3), bnd.SPARK_ERR_ALIGN),
    (dict(ptrs=[FAKE] * 6 + [FAKE + 16]), bnd.SPARK_ERR_ALIGN),   # workspace needs 256
    (dict(ws_bytes=100), bnd.SPARK_ERR_WORKSPACE),
])
def test_decode_rejects(kw, code):
    assert decode_call(**kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(null_desc=True), bnd.SPARK_ERR_NULL),
    (dict(T=-3), bnd.SPARK_ERR_SHAPE),
    (dict(H=16, Hkv=5), bnd.SPARK_ERR_SHAPE),
    (dict(H=6, Hkv=2), bnd.SPARK_ERR_UNSUPPORTED),
    (dict(d=desc(kind=1, window=-1)), bnd.SPARK_ERR_SHAPE),
    (dict(d=desc(kind=0, rot=40)), bnd.SPARK_ERR_UNSUPPORTED),
    (dict(ptrs=[0] + [FAKE] * 4), bnd.SPARK_ERR_NULL),
    (dict(ptrs=[FAKE] * 3 + [FAKE + 4, FAKE]), bnd.SPARK_ERR_ALIGN),
    (dict(ptrs=[FAKE, FAKE + 1, FAKE, FAKE, FAKE]), bnd.SPARK_ERR_ALIGN),
    (dict(ws_bytes=255), bnd.SPARK_ERR_WORKSPACE),
])
def test_prefill_rejects(kw, code):
    assert prefill_call(**kw) == code


def test_empty_calls_launch_nothing():
    # B == 0 or T == 0 is a valid empty call, even with NULL data pointers
    assert decode_call(B=0, ptrs=[0] * 7) == bnd.SPARK_OK
    assert prefill_call(B=0, ptrs=[0] * 5) == bnd.SPARK_OK
    assert prefill_call(T=0, ptrs=[0] * 5) == bnd.SPARK_OK


def test_workspace_queries():
    full = desc(kind=0, window=0, theta=5e6, rot=64)
    sl = desc()
    # prefill: header + rotated leading K dims (rot_dim rounded up to 64)
    n = fga.lib.spark_attn_prefill_workspace_size(2, 8192, 16, 4, ctypes.byref(full))
    assert n >= 256 + 2 * 4 * 8192 * 64 * 2
    n = fga.lib.spark_attn_prefill_workspace_size(1, 100, 16, 4, ctypes.byref(sl))
    assert n >= 256 + 1 * 4 * 100 * 256 * 2
    assert fga.lib.spark_attn_prefill_workspace_size(1, 100, 16, 3, ctypes.byref(sl)) == 0
    # decode: partial softmax states per (b, h, split)
    n = fga.lib.spark_attn_decode_workspace_size(64, 16, 4, 131073, ctypes.byref(full))
    assert n > 64 * 16 * 258 * 4
    assert fga.lib.spark_attn_decode_workspace_size(1, 16, 4, 100, ctypes.byref(sl)) == 0
    assert fga.lib.spark_attn_decode_workspace_size(0, 16, 4, 512, ctypes.byref(sl)) >= 256


def test_binding_refuses_cpu_tensors():
    import torch
    x = torch.zeros((1, 4, 6 * 256), dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        fga.spark_attn_prefill(x, torch.zeros((1, 4, 4)), torch.zeros((1, 4), dtype=torch.int32),
                               fga.layer_desc(0, 0, 5e6, 64))


def test_layer_calls_check_before_enqueueing():
    """The attention-block calls refuse bad arguments on the host (no GPU is
    needed to reach these answers)."""
    full = fga.layer_desc(fga.SPARK_LAYER_FULL, 0, 5e6, 64)
    d = ctypes.byref(full)
    L = fga.lib
    # hidden not a multiple of 8, or not positive
    assert L.spark_attn_layer_prefill(None, None, None, None, None, None, None, 0, d, 1, 4, 2561,
                                      16, 4, None, None, 0, None) == 3
    assert L.spark_attn_layer_prefill(None, None, None, None, None, None, None, 0, d, 1, 4, 0,
                                      16, 4, None, None, 0, None) == 2
    # the core's own shape rule (H % Hkv)
    assert L.spark_attn_layer_prefill(None, None, None, None, None, None, None, 0, d, 1, 4, 2560,
                                      16, 3, None, None, 0, None) == 2
    assert L.spark_attn_layer_decode(None, None, None, None, None, None, None, 100, d, 1, 2560,
                                     16, 3, None, None, 0, None) == 2
    # empty batch: nothing to do
    assert L.spark_attn_layer_prefill(None, None, None, None, None, None, None, 0, d, 0, 4, 2560,
                                      16, 4, None, None, 0, None) == 0
    assert L.spark_attn_layer_decode(None, None, None, None, None, None, None, 100, d, 0, 2560,
                                     16, 4, None, None, 0, None) == 0
    # missing pointers
    assert L.spark_attn_layer_prefill(None, None, None, None, None, None, None, 0, d, 1, 4, 2560,
                                      16, 4, None, None, 0, None) == 1
    # workspace sizes: the core's plus the projections' buffers
    core = L.spark_attn_prefill_workspace_size(2, 8192, 16, 4, d)
    n = L.spark_attn_layer_prefill_workspace_size(2, 8192, 2560, 16, 4, d)
    rows = 2 * 8192
    assert n >= core + rows * (6144 * 2 + 16 * 4 + 4096 * 2)
    assert L.spark_attn_layer_prefill_workspace_size(2, 8192, 2561, 16, 4, d) == 0
    assert L.spark_attn_layer_decode_workspace_size(1, 2560, 16, 4, 1 << 20, d) > \
        L.spark_attn_decode_workspace_size(1, 16, 4, 1 << 20, d)


def test_decode_launch_count():
    """1 launch where the split kernel merges itself, 2 where the merge kernel
    follows it, 0 for invalid arguments or an empty batch (plan for the
    152-SM GB300 when no device is visible)."""
    full = desc(kind=0, window=0, theta=5e6, rot=64)
    ring = desc()
    count = fga.lib.spark_attn_decode_launch_count
    assert count(1, 16, 4, 512, ctypes.byref(ring)) == 1          # 8 splits, 4 counters
    assert count(64, 16, 4, 512, ctypes.byref(ring)) == 1         # one split each
    assert count(1, 16, 4, 1 << 20, ctypes.byref(full)) == 2      # 38 splits
    assert count(21, 12, 3, 512, ctypes.byref(ring)) == 1         # 63 counters: the last word
    assert count(16, 16, 4, 512, ctypes.byref(ring)) == 2         # 64 pairs, 2 splits each
    assert count(0, 16, 4, 512, ctypes.byref(ring)) == 0
    assert count(1, 16, 5, 512, ctypes.byref(ring)) == 0          # H % Hkv != 0
    assert count(1, 16, 4, 512, None) == 0
