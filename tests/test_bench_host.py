"""bench.py host logic that needs no GPU: the packing of the decode step's
host transfers (every layer's new-token inputs in one buffer, every output in
one buffer)."""
from __future__ import annotations

import torch

import bench


def _layers(n):
    dec = []
    g = torch.Generator().manual_seed(5)
    for i in range(n):
        H, Hkv, B = (16, 4, 1) if i % 2 else (8, 2, 3)
        dec.append({
            "host": {
                "qkv": torch.randn((B, (H + 2 * Hkv) * 256), generator=g).to(torch.bfloat16),
                "gate": torch.randn((B, H), generator=g),
                "pos": torch.arange(B, dtype=torch.int32) + 7 * i,
            },
            "dev": {},
            "out": torch.empty((B, H * 256), dtype=torch.bfloat16),
        })
    return dec


def test_pack_decode_io_keeps_values_shapes_and_alignment(monkeypatch):
    monkeypatch.setattr(torch.Tensor, "pin_memory", lambda self: self)  # no CUDA here
    dec = _layers(5)
    want = [{k: v.clone() for k, v in L["host"].items()} for L in dec]
    out_shapes = [L["out"].shape for L in dec]
    io = bench.pack_decode_io(dec, torch.device("cpu"))
    base_in, base_out = io["dev_in"].data_ptr(), io["dev_out"].data_ptr()
    n_in = 0
    for L, w, shape in zip(dec, want, out_shapes):
        for k, t in w.items():
            v = L["dev"][k]
            assert v.dtype == t.dtype and v.shape == t.shape and torch.equal(v, t)
            # sections start on 256-byte boundaries of the packed buffer
            assert (v.data_ptr() - base_in) % 256 == 0
            n_in += t.numel() * t.element_size()
        assert L["out"].shape == shape and L["out"].dtype == torch.bfloat16
        assert (L["out"].data_ptr() - base_out) % 256 == 0
    # the host buffer holds the same bytes the device buffer was filled with
    assert torch.equal(io["host_in"], io["dev_in"])
    # one transfer each way: the packed sizes are the tensors plus section padding
    assert n_in <= io["host_in"].numel() < n_in + 256 * 3 * len(dec)
    n_out = sum(L["out"].numel() * 2 for L in dec)
    assert n_out <= io["host_out"].numel() < n_out + 256 * len(dec)


def test_pack_decode_io_outputs_do_not_overlap(monkeypatch):
    monkeypatch.setattr(torch.Tensor, "pin_memory", lambda self: self)
    dec = _layers(4)
    bench.pack_decode_io(dec, torch.device("cpu"))
    for i, L in enumerate(dec):
        L["out"].fill_(float(i + 1))
    for i, L in enumerate(dec):
        assert torch.all(L["out"] == float(i + 1))


def test_decode_step_launch_count_of_the_1m_step():
    """The 1M-context step: 9 full layers (38 splits each: split + merge kernel)
    and 27 rings (8 splits, B * Hkv = 4: the split kernel merges itself)."""
    dec = [{"case": bench.DECODE_FULL if layer.kind == bench.wl.FULL else bench.DECODE_SLIDING,
            "layer": layer} for layer in bench.decode_layers(36)]
    assert bench.decode_step_launches(dec) == 9 * 2 + 27 * 1
