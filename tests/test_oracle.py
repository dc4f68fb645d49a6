"""CPU tests of the fp64 oracle: its pins, planted mistakes, page constants."""
from __future__ import annotations

import json
import os
import tempfile

import numpy as np
import pytest

import oracle
import oracle_pins
import workloads

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(orc, pin):
    pin(orc)


# Plausible mistakes, planted one at a time in a copy of the oracle source.
# Every one of them must make at least one pin fail.
MUTANTS = [
    ("rope_sign_first_half", "y[k] = x1 * c - x2 * s;", "y[k] = x1 * c + x2 * s;"),
    ("rope_sign_second_half", "y[k + half] = x2 * c + x1 * s;", "y[k + half] = x2 * c - x1 * s;"),
    ("rope_freq_over_head_dim", "-2.0 * (double)k / (double)rot_dim",
     "-2.0 * (double)k / (double)ORACLE_HEAD_DIM"),
    ("rope_pairs_adjacent", "double x1 = x[k], x2 = x[k + half];",
     "double x1 = x[k], x2 = x[(k + 1) % rot_dim];"),
    ("window_off_by_one", "int64_t lo = i - (int64_t)window + 1;",
     "int64_t lo = i - (int64_t)window;"),
    ("scale_one_over_d", "1.0 / sqrt((double)ORACLE_HEAD_DIM)", "1.0 / (double)ORACLE_HEAD_DIM"),
    ("gate_dropped_prefill", "out[d] *= gsig;", "out[d] *= 1.0;"),
    ("gate_dropped_decode", "dst[d] = o[d] * gsig;", "dst[d] = o[d];"),
    ("sigmoid_sign", "1.0 / (1.0 + exp(-x))", "1.0 / (1.0 + exp(x))"),
    ("silu_without_x", "mode == ORACLE_GATE_SILU ? x * sigmoid(x) : sigmoid(x)",
     "mode == ORACLE_GATE_SILU ? sigmoid(x) : sigmoid(x)"),
    ("group_map_modulo", "int g = h / G;", "int g = h % Hkv;"),
    ("v_from_k_slot", "(int64_t)(H + Hkv + g) * D", "(int64_t)(H + g) * D"),
    ("softmax_sign", "exp(s_scratch[j] - m)", "exp(m - s_scratch[j])"),
    ("self_not_visible", "int64_t nvis = i - lo + 1;", "int64_t nvis = i - lo;"),
    ("ring_slot_mod_window", "? tok % cap : tok", "? tok % window : tok"),
    ("decode_query_position", "rope_head(qx, (double)p, rot_dim, theta, q);",
     "rope_head(qx, (double)(p + 1), rot_dim, theta, q);"),
    ("decode_new_token_misplaced", "if (tok == p) {", "if (tok == p - 1) {"),
    ("decode_window_off_by_one", "int64_t nvis = p - lo + 1;", "int64_t nvis = p - lo;"),
    ("q_from_k_slot", "qkv + row * width + (int64_t)h * D;",
     "qkv + row * width + (int64_t)(h / G) * D;"),
]


def test_mutants_are_caught():
    src = open(oracle._SRC).read()
    escaped = []
    with tempfile.TemporaryDirectory() as tmp:
        for name, old, new in MUTANTS:
            assert old in src, f"mutant {name}: pattern not found in the oracle source"
            msrc = os.path.join(tmp, f"{name}.c")
            with open(msrc, "w") as f:
                f.write(src.replace(old, new))
            lib = oracle.OracleLib(oracle.build(force=True, src=msrc,
                                                out=os.path.join(tmp, f"{name}.so")))
            caught = []
            for pin in oracle_pins.ALL_PINS:
                try:
                    pin(lib)
                except (AssertionError, ValueError, FloatingPointError):
                    caught.append(pin.__name__)
            if not caught:
                escaped.append(name)
    assert not escaped, f"planted mistakes no pin catches: {escaped}"


def test_config_constants_match_pages():
    """The workload presets carry the page's config values (§1, §4)."""
    cfg = json.load(open(os.path.join(GOLDEN, "spark_x25_config.json")))
    m4, m17, rope = cfg["4B"], cfg["1.7B"], cfg["rope"]
    c2 = workloads.PREFILL_FULL_4B_B2_T8192
    assert (c2.H, c2.Hkv) == (m4["num_attention_heads"], m4["num_key_value_heads"])
    assert c2.width == m4["qkv_width"] == (16 + 2 * 4) * 256
    c1 = workloads.PREFILL_SLIDING_1P7B_T1024
    assert (c1.H, c1.Hkv) == (m17["num_attention_heads"], m17["num_key_value_heads"])
    assert c1.width == m17["qkv_width"]
    fl, sl = workloads.FULL_LAYER, workloads.SLIDING_LAYER
    assert fl.theta == rope["full_attention"]["rope_theta"]
    assert fl.rot_dim == rope["full_attention"]["rotated_dims"]
    assert fl.rot_dim == int(256 * rope["full_attention"]["partial_rotary_factor"])
    assert sl.theta == rope["sliding_attention"]["rope_theta"]
    assert sl.rot_dim == rope["sliding_attention"]["rotated_dims"]
    assert sl.window == m4["sliding_window"]
    lt = workloads.LAYER_TYPES_4B
    assert len(lt) == m4["num_hidden_layers"]
    full_1based = [i + 1 for i, l in enumerate(lt) if l.kind == workloads.FULL]
    assert full_1based == m4["full_layers_1based"]
    # 1M-context decode: the new token sits at the last position the model
    # supports (max_position_embeddings - 1).
    d5 = workloads.DECODE_FULL_4B_1M
    assert d5.len_hi == m4["max_position_embeddings"] - 1
    assert d5.cap == m4["max_position_embeddings"]


def test_kv_bytes_match_pages():
    """KV-cache arithmetic of §6: 2 (K,V) x Hkv x 256 x 2 B per token per layer."""
    kv = json.load(open(os.path.join(GOLDEN, "kv_cache_bytes.json")))
    import torch
    for case, want in ((workloads.DECODE_FULL_4B_B64, kv["bytes_per_token_per_layer_4B"]),):
        one_token = torch.empty((1, case.Hkv, 1, 256), dtype=torch.bfloat16)
        assert 2 * one_token.numel() * one_token.element_size() == want
    assert 2 * 2 * 256 * 2 == kv["bytes_per_token_per_layer_1p7B"]
    per_tok = kv["bytes_per_token_per_layer_4B"]
    full = kv["full_layers_4B"] * 10**6 * per_tok
    assert abs(full / 1e9 - kv["page_full_9_layers_1M_GB"]) < 0.05
    sliding = kv["sliding_layers_4B"] * kv["sliding_cache_tokens"] * per_tok
    assert sliding == 56_623_104 and abs(sliding / 1e6 - kv["page_sliding_27_layers_MB"]) < 0.05
    allfull = 36 * 10**6 * per_tok
    assert abs(allfull / 1e9 - kv["page_all_full_36_layers_1M_GB"]) < 0.5
    assert abs(full / allfull - kv["page_ratio"]) < 1e-12
    assert abs(7 * 10**6 * kv["bytes_per_token_per_layer_1p7B"] / 1e9
               - kv["page_1p7B_7_full_layers_1M_GB"]) < 0.5
    # the 1M decode workload reads exactly 9 x 2^20 x 4096 B of full-layer KV
    assert 9 * workloads.DECODE_FULL_4B_1M.cap * per_tok == 38_654_705_664


def test_oracle_rejects_bad_arguments(orc):
    bits = np.zeros((1, 2, 6 * 256), np.uint16)
    g = np.zeros((1, 2, 4), np.float32)
    pos = np.zeros((1, 2), np.int32)
    with pytest.raises(ValueError):
        orc.prefill(bits, g, pos, 1, 0, 1e4, 256, 4, 1)  # sliding window 0
    with pytest.raises(ValueError):
        orc.prefill(bits, g, pos, 0, 0, 1e4, 63, 4, 1)  # odd rot_dim
