"""CPU pins of the oracle's attention block (projections around the core).

Spark-X2.5 architecture page, §3 Eq. 1 and Fig. 1: q_k_v_proj and g_proj read
the normed hidden state, the core attends, out_proj maps the gated output back
to the hidden size; §1 / §3: tensors are bf16, the gated output is cast back
to the weight dtype.  The pins choose weights that are permutations and
selections (possibly scaled by 1.5), so every projection reduces to a gather
of known values; the expected block output is then built from gathers, the
core oracle (pinned on its own in test_oracle.py) and torch's fp32 -> bf16
conversion, never from the projection code under test.  Planted mistakes in a
copy of the oracle's block code must each fail a pin.
"""
from __future__ import annotations

import importlib.util
import os
import sys

import numpy as np
import pytest
import torch

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
D = 256


def bf16_bits_of(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)


def f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_exact_bits(v: np.ndarray) -> np.ndarray:
    """fp64 -> bf16 patterns, round to nearest even, through the fp32 image:
    where fp32 rounding landed exactly on a bf16 midpoint, the fp64 value
    decides (a formulation independent of the oracle's frexp / rint one)."""
    v = np.asarray(v, np.float64)
    f = v.astype(np.float32)
    b = f.view(np.uint32)
    low, hi = b & 0xFFFF, b >> 16
    up = (low > 0x8000) | ((low == 0x8000) & ((hi & 1) == 1))
    mid = low == 0x8000
    m = np.abs(f.astype(np.float64))
    up = np.where(mid & (np.abs(v) > m), True, up)
    up = np.where(mid & (np.abs(v) < m), False, up)
    return (hi + up).astype(np.uint16)


def perm_matrix(perm: np.ndarray, scale: float = 1.0) -> np.ndarray:
    """Rows i select column perm[i]: (x W^T)[:, i] = scale * x[:, perm[i]]."""
    n = perm.shape[0]
    w = np.zeros((n, n), np.float32)
    w[np.arange(n), perm] = scale
    return bf16_bits_of(torch.from_numpy(w))


def selection(rows: int, cols: int, pick: np.ndarray, scale: float = 1.0) -> np.ndarray:
    """[rows, cols] with W[r, pick[r]] = scale: (x W^T)[:, r] = scale * x[:, pick[r]]."""
    w = np.zeros((rows, cols), np.float32)
    w[np.arange(rows), pick] = scale
    return bf16_bits_of(torch.from_numpy(w))


def setup(seed: int, B: int, T: int, H: int, Hkv: int, scale: float):
    """A block whose hidden size equals the qkv width, with permutation /
    selection weights, and the expected output built by gathers."""
    rng = np.random.default_rng(seed)
    width = (H + 2 * Hkv) * D
    hidden = width
    x = torch.randn((B, T, hidden), generator=torch.Generator().manual_seed(seed))
    x_bits = bf16_bits_of(x)
    xf = f64(x_bits)
    perm = rng.permutation(width)
    assert np.any(perm[perm] != np.arange(width))  # not an involution
    gpick = rng.integers(0, hidden, H)
    opick = rng.integers(0, H * D, hidden)
    w_qkv = perm_matrix(perm, scale)
    w_g = selection(H, hidden, gpick, scale)
    w_o = selection(hidden, H * D, opick)
    # expected: gathers, then torch's RNE conversion of the exact fp32 products
    qkv_bits = bf16_bits_of(torch.from_numpy((xf[:, :, perm] * scale).astype(np.float32)))
    g = f64(bf16_bits_of(torch.from_numpy((xf[:, :, gpick] * scale).astype(np.float32))))
    pos = np.tile(np.arange(T, dtype=np.int32), (B, 1))
    return dict(x_bits=x_bits, w_qkv=w_qkv, w_g=w_g, w_o=w_o, qkv_bits=qkv_bits, g=g,
                pos=pos, opick=opick, hidden=hidden)


LAYERS = [(oracle.SLIDING, 7, 1e4, 256), (oracle.FULL, 0, 5e6, 64)]


def pin_prefill_permutation_weights(orc_mod, scale):
    for kind, W, theta, r in LAYERS:
        s = setup(3, B=2, T=9, H=2, Hkv=1, scale=scale)
        y = orc_mod.layer_prefill(s["x_bits"], s["w_qkv"], s["w_g"], s["w_o"], s["pos"], kind,
                                  W, theta, r, 2, 1)
        a = oracle.prefill(s["qkv_bits"], s["g"].astype(np.float32), s["pos"], kind, W, theta,
                           r, 2, 1)
        want = f64(bf16_exact_bits(a))[:, :, s["opick"]]
        assert np.array_equal(y, want), np.abs(y - want).max()


def pin_prefill_rows_subset(orc_mod):
    s = setup(5, B=1, T=11, H=1, Hkv=1, scale=1.0)
    full = orc_mod.layer_prefill(s["x_bits"], s["w_qkv"], s["w_g"], s["w_o"], s["pos"],
                                 oracle.SLIDING, 4, 1e4, 256, 1, 1)
    rows = np.array([0, 5, 10])
    part = orc_mod.layer_prefill(s["x_bits"], s["w_qkv"], s["w_g"], s["w_o"], s["pos"],
                                 oracle.SLIDING, 4, 1e4, 256, 1, 1, rows=rows)
    assert np.array_equal(part, full.reshape(11, -1)[rows])


def pin_decode_permutation_weights(orc_mod, scale):
    H, Hkv, B, cap = 2, 1, 3, 16
    s = setup(7, B=B, T=1, H=H, Hkv=Hkv, scale=scale)
    gen = torch.Generator().manual_seed(8)
    kc = bf16_bits_of(torch.randn((B, Hkv, cap, D), generator=gen))
    vc = bf16_bits_of(torch.randn((B, Hkv, cap, D), generator=gen))
    pos = np.array([0, 5, 15], np.int32)
    for kind, W, theta, r in LAYERS:
        y, kn, vn = orc_mod.layer_decode(s["x_bits"].reshape(B, -1), s["w_qkv"], s["w_g"],
                                         s["w_o"], pos, kc, vc, kind, W, theta, r, H, Hkv)
        a, kn2, vn2 = oracle.decode(s["qkv_bits"].reshape(B, -1), s["g"].reshape(B, H)
                                    .astype(np.float32), pos, kc, vc, kind, W, theta, r, H,
                                    Hkv)
        assert np.array_equal(y, f64(bf16_exact_bits(a))[:, s["opick"]])
        assert np.array_equal(kn, kn2) and np.array_equal(vn, vn2)


def pin_out_proj_is_linear(orc_mod):
    s = setup(9, B=1, T=5, H=1, Hkv=1, scale=1.0)
    rng = np.random.default_rng(10)
    w_o = bf16_bits_of(torch.from_numpy(rng.standard_normal((s["hidden"], D)).astype(np.float32)))
    w_o2 = bf16_bits_of(torch.from_numpy(2.0 * f64(w_o).astype(np.float32)))
    args = (s["x_bits"], s["w_qkv"], s["w_g"])
    y1 = orc_mod.layer_prefill(*args, w_o, s["pos"], oracle.FULL, 0, 5e6, 64, 1, 1)
    y2 = orc_mod.layer_prefill(*args, w_o2, s["pos"], oracle.FULL, 0, 5e6, 64, 1, 1)
    assert np.array_equal(2.0 * y1, y2)


PINS = [
    ("prefill permutation weights", lambda m: pin_prefill_permutation_weights(m, 1.0)),
    ("prefill weights x1.5 (bf16 rounding of qkv and gate)",
     lambda m: pin_prefill_permutation_weights(m, 1.5)),
    ("prefill rows subset", pin_prefill_rows_subset),
    ("decode permutation weights", lambda m: pin_decode_permutation_weights(m, 1.0)),
    ("decode weights x1.5", lambda m: pin_decode_permutation_weights(m, 1.5)),
    ("out_proj linear", pin_out_proj_is_linear),
]


@pytest.mark.parametrize("name,pin", PINS, ids=[p[0] for p in PINS])
def test_layer_pin(name, pin):
    pin(oracle)


# Mistakes planted one at a time in a copy of the oracle's block code.
MUTANTS = [
    ("q_k_v_proj not transposed",
     "qkv_bits = bf16_round_bits(x @ bits_to_f64(w_qkv_bits).T)          # q_k_v_proj",
     "qkv_bits = bf16_round_bits(x @ bits_to_f64(w_qkv_bits))"),
    ("g_proj from the wrong side",
     "g = bits_to_f64(bf16_round_bits(x @ bits_to_f64(w_g_bits).T))      # g_proj",
     "g = bits_to_f64(bf16_round_bits(x[..., ::-1] @ bits_to_f64(w_g_bits).T))"),
    ("decode q_k_v_proj not transposed",
     "    qkv_bits = bf16_round_bits(x @ bits_to_f64(w_qkv_bits).T)\n    g = bits_to_f64(bf16_round_bits(x @ bits_to_f64(w_g_bits).T))\n    a, k_new",
     "    qkv_bits = bf16_round_bits(x @ bits_to_f64(w_qkv_bits))\n    g = bits_to_f64(bf16_round_bits(x @ bits_to_f64(w_g_bits).T))\n    a, k_new"),
    ("gated output not cast to bf16", "    a = bits_to_f64(bf16_round_bits(a))                                # cast to bf16\n",
     "\n"),
    ("rounding by truncation", "q = np.rint(m * 256.0) / 256.0", "q = np.trunc(m * 256.0) / 256.0"),
    ("ties rounded away from zero", "q = np.rint(m * 256.0) / 256.0",
     "q = np.sign(m) * np.floor(np.abs(m) * 256.0 + 0.5) / 256.0"),
    ("out_proj transposed input", "    return a @ bits_to_f64(w_o_bits).T                                 # out_proj",
     "    return a @ bits_to_f64(w_o_bits)[::-1].T"),
    ("decode gate not rounded",
     "    g = bits_to_f64(bf16_round_bits(x @ bits_to_f64(w_g_bits).T))\n    a, k_new",
     "    g = x @ bits_to_f64(w_g_bits).T\n    a, k_new"),
]


def load_mutant(tmp_path, old, new):
    src = open(os.path.join(ROOT, "oracle", "__init__.py")).read()
    assert src.count(old) == 1, old
    pkg = tmp_path / "oracle_mutant"
    pkg.mkdir()
    (pkg / "__init__.py").write_text(src.replace(old, new))
    # the mutant reuses the pinned core oracle's compiled library
    spec = importlib.util.spec_from_file_location("oracle_mutant", str(pkg / "__init__.py"))
    mod = importlib.util.module_from_spec(spec)
    sys.modules["oracle_mutant"] = mod
    spec.loader.exec_module(mod)
    mod._default = oracle.default()
    return mod


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_layer_mutants_are_caught(tmp_path, name, old, new):
    mod = load_mutant(tmp_path, old, new)
    failed = 0
    for _, pin in PINS:
        try:
            pin(mod)
        except (AssertionError, ValueError, IndexError):
            failed += 1
    sys.modules.pop("oracle_mutant", None)
    assert failed > 0, f"planted mistake not caught: {name}"
