"""Benchmark of the Spark-X2.5 attention core on GB300.

One step is one pass of the whole hot path over one batch of synthetic input:
  * prefill of a 4B-shaped full_attention layer, B=2, T=8192, H=16, Hkv=4
    (causal, RoPE theta 5e6 on 64 dims, sigmoid gate): 1.0996 TFLOP;
  * one 1M-context decode step of all 36 attention cores of the 4B model in
    layer order (9 full layers with 1,048,575 cached tokens each, 27 sliding
    layers with full 512-slot rings): 38.71 GB of KV read.
The JSON line's value is the prefill throughput (TFLOP/s); the decode KV-read
bandwidth is reported beside it.  Outside the timed step the line also carries
the 1.7B sliding prefill (B=1, T=1024) per call and in a CUDA graph, the whole
attention block of the prefill layer (projections + core), and the decode step
through all 36 attention blocks.  Inputs are seeded synthetic tensors of the
model's shapes (no dataset or weights exist for this path).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl {ours,reference}]
                  [--only {all,prefill,decode}] [--decode-layers L]

Under torchrun every rank runs its own replica (the attention core needs no
exchange between GPUs); value is the work of all ranks over the slowest rank.
--impl reference times the fp64 CPU oracle on a bounded sample instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

PREFILL = wl.PREFILL_FULL_4B_B2_T8192
# the same shapes as a sliding_attention layer, for profiling (--prefill-layer sliding)
PREFILL_SLIDING_B2_T8192 = wl.scaled(wl.PREFILL_FULL_4B_B2_T8192,
                                     name="prefill_sliding_4b_B2_T8192", layer=wl.SLIDING_LAYER)
DECODE_FULL = wl.DECODE_FULL_4B_1M
DECODE_SLIDING = wl.DECODE_SLIDING_4B_1M
METRIC = "prefill attn TFLOP/s & % bf16 peak; decode KV-read GB/s & % HBM peak (1 GB300)"
KV_BYTES_PER_TOKEN = 2 * 4 * 256 * 2  # K and V, 4 KV heads, 256 dims, bf16


def visible_pairs(T: int, kind: int, window: int) -> int:
    """Sum over queries of the number of visible keys (mask definition)."""
    if kind == wl.FULL:
        return T * (T + 1) // 2
    W = window
    if T <= W:
        return T * (T + 1) // 2
    return W * (W + 1) // 2 + (T - W) * W


def prefill_flops(case) -> float:
    return 4.0 * 256 * case.B * case.H * visible_pairs(case.T, case.layer.kind,
                                                        case.layer.window)


def decode_layers(n_layers: int):
    return list(wl.LAYER_TYPES_4B[:n_layers])


def pack_decode_io(dec, dev):
    """Lay every layer's new-token inputs (qkv, gate, pos) and outputs out in one
    pinned host buffer and one device buffer each, so that a decode step moves its
    inputs in one host-to-device copy and its outputs in one read.  Each layer's
    device tensors become views into the packed buffers (same values)."""
    import torch

    def sections(tensors):
        offs, off = [], 0
        for t in tensors:
            off = (off + 255) // 256 * 256
            offs.append(off)
            off += t.numel() * t.element_size()
        return offs, (off + 255) // 256 * 256
    ins = [L["host"][k] for L in dec for k in ("qkv", "gate", "pos")]
    in_offs, in_bytes = sections(ins)
    host_in = torch.zeros(in_bytes, dtype=torch.uint8).pin_memory()
    dev_in = torch.zeros(in_bytes, dtype=torch.uint8, device=dev)
    for t, off in zip(ins, in_offs):
        n = t.numel() * t.element_size()
        host_in[off:off + n].copy_(t.contiguous().view(-1).view(torch.uint8))
    dev_in.copy_(host_in)
    outs = [L["out"] for L in dec]
    out_offs, out_bytes = sections(outs)
    dev_out = torch.zeros(out_bytes, dtype=torch.uint8, device=dev)
    host_out = torch.zeros(out_bytes, dtype=torch.uint8).pin_memory()
    i = 0
    for L in dec:
        for k in ("qkv", "gate", "pos"):
            t = L["host"][k]
            n = t.numel() * t.element_size()
            L["dev"][k] = dev_in[in_offs[i]:in_offs[i] + n].view(t.dtype).view(t.shape)
            i += 1
    for L, off in zip(dec, out_offs):
        o = L["out"]
        n = o.numel() * o.element_size()
        L["out"] = dev_out[off:off + n].view(o.dtype).view(o.shape)
    return {"host_in": host_in, "dev_in": dev_in, "host_out": host_out, "dev_out": dev_out}


def decode_kv_bytes(layers) -> tuple[int, int]:
    """(bytes of all layers, bytes of one full layer) of visible K/V per step."""
    p = DECODE_FULL.len_hi
    full = (p + 1) * KV_BYTES_PER_TOKEN
    sliding = min(p + 1, wl.SLIDING_LAYER.window) * KV_BYTES_PER_TOKEN
    total = sum(full if l.kind == wl.FULL else sliding for l in layers)
    return total, full


def decode_step_launches(dec) -> int:
    """Kernels one decode step enqueues, as the library reports them: per layer
    1 (the split kernel merges itself) or 2 (split kernel, then merge kernel)."""
    import full_gqa_attention_gb300 as fga
    return sum(fga.spark_attn_decode_launch_count(L["case"].B, L["case"].H, L["case"].Hkv,
                                                  L["case"].cap, L["layer"]) for L in dec)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained"), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# ---------------------------------------------------------------- distributed

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("gloo", rank=rank, world_size=world)
    return rank, world, local


def dist_barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def dist_max(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_sum(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs.

    Each sample carries nvidia-smi's timestamp, so that the samples taken
    inside the timed region (between mark_start and mark_end) are told apart
    from those of the untimed repeat of the same step that follows it."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    INTERVAL_MS = 100

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.t_start = self.t_end = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.INTERVAL_MS)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def mark_start(self):
        self.t_start = time.time()

    def mark_end(self):
        self.t_end = time.time()

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    @staticmethod
    def _when(stamp: str):
        import datetime
        try:
            return datetime.datetime.strptime(stamp, "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def summary(self):
        sm, mx, reasons, in_timed = [], [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 10:
                continue
            try:
                sm.append(float(f[2]))
                mx.append(float(f[3]))
            except ValueError:
                continue
            t = self._when(f[0])
            if (t is not None and self.t_start is not None and self.t_end is not None
                    and self.t_start <= t <= self.t_end):
                in_timed += 1
            for name, v in zip(names, f[6:10]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "sm_mhz_min": min(sm), "reasons": sorted(reasons), "samples": len(sm),
                "samples_in_timed_region": in_timed, "interval_ms": self.INTERVAL_MS,
                "window": "the timed steps, then the same step repeated untimed for "
                          f"{CLOCK_SOAK_S:.1f} s so that the load is sampled often enough"}


# After the timed steps the same step runs on, untimed, this long while the
# clock sampler keeps going: the timed region alone is too short for the
# sampler's interval.
CLOCK_SOAK_S = 2.5


# ---------------------------------------------------------------- our arm

def run_ours(args, rank, world, local):
    import torch
    import full_gqa_attention_gb300 as fga

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    hbm_peak, bf16_peak, bf16_sust, peak_src = load_peaks()
    do_prefill = args.only in ("all", "prefill")
    do_decode = args.only in ("all", "decode")
    layers = decode_layers(args.decode_layers) if do_decode else []

    # ---- prefill inputs (resident) and their pinned host copies (for e2e)
    pre = None
    if do_prefill:
        x = wl.make_prefill_inputs(PREFILL)
        pre = {
            "host": {k: v.pin_memory() for k, v in x.items()},
            "dev": {k: v.to(dev) for k, v in x.items()},
        }
        c = PREFILL
        pre["out"] = torch.empty((c.B, c.T, c.H * 256), dtype=torch.bfloat16, device=dev)
        pre["host_out"] = torch.empty_like(pre["out"], device="cpu").pin_memory()
        pre["ws_host"] = fga.new_workspace(
            fga.spark_attn_prefill_host_workspace_size(c.B, c.T, c.H, c.Hkv, c.layer), dev)
        pre["ws"] = fga.new_workspace(fga.spark_attn_prefill_workspace_size(
            c.B, c.T, c.H, c.Hkv, c.layer), dev)

    # ---- decode state: one cache per layer, new-token inputs per layer
    dec = []
    for i, layer in enumerate(layers):
        case = DECODE_FULL if layer.kind == wl.FULL else DECODE_SLIDING
        step = wl.make_decode_step_inputs(wl.scaled(case, seed=case.seed + 7 * i))
        kc = torch.empty((case.B, case.Hkv, case.cap, 256), dtype=torch.bfloat16, device=dev)
        vc = torch.empty_like(kc)
        g = torch.Generator(dev).manual_seed(1000 + i)
        kc.normal_(generator=g)
        vc.normal_(generator=g)
        dec.append({
            "case": case, "layer": layer, "k": kc, "v": vc,
            "host": {k: v.pin_memory() for k, v in step.items()},
            "dev": {k: v.to(dev) for k, v in step.items()},
            "out": torch.empty((case.B, case.H * 256), dtype=torch.bfloat16, device=dev),
            "ws": fga.new_workspace(fga.spark_attn_decode_workspace_size(
                case.B, case.H, case.Hkv, case.cap, layer), dev),
        })
    dec_io = pack_decode_io(dec, dev) if dec else None
    torch.cuda.synchronize()

    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    def step(timing=None):
        if pre is not None:
            d = pre["dev"]
            if timing is not None:
                timing["p0"].append(ev()); timing["p0"][-1].record(stream)
            fga.spark_attn_prefill(d["qkv"], d["gate"], d["pos"], PREFILL.layer,
                                   out=pre["out"], workspace=pre["ws"], stream=stream)
            if timing is not None:
                timing["p1"].append(ev()); timing["p1"][-1].record(stream)
        if dec:
            if timing is not None:
                timing["d0"].append(ev()); timing["d0"][-1].record(stream)
            for L in dec:
                d = L["dev"]
                full = L["layer"].kind == wl.FULL
                if timing is not None and full:
                    e = ev(); e.record(stream); timing["f0"].append(e)
                fga.spark_attn_decode(d["qkv"], d["gate"], d["pos"], L["k"], L["v"], L["layer"],
                                      out=L["out"], workspace=L["ws"], stream=stream)
                if timing is not None and full:
                    e = ev(); e.record(stream); timing["f1"].append(e)
            if timing is not None:
                timing["d1"].append(ev()); timing["d1"][-1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    timing = {k: [] for k in ("p0", "p1", "d0", "d1", "f0", "f1")}
    start, stop = ev(), ev()
    with ClockSampler(local) as clocks:
        dist_barrier(world)
        torch.cuda.synchronize()
        clocks.mark_start()
        start.record(stream)
        for _ in range(args.steps):
            step(timing)
        stop.record(stream)
        torch.cuda.synchronize()
        clocks.mark_end()
        dist_barrier(world)
        # the same load, untimed, while the sampler keeps sampling
        t_soak = time.time() + CLOCK_SOAK_S
        while time.time() < t_soak:
            for _ in range(4):
                step()
            torch.cuda.synchronize()
    total_ms = start.elapsed_time(stop) / args.steps

    def mean_ms(a, b):
        ts = [x.elapsed_time(y) for x, y in zip(timing[a], timing[b])]
        return sum(ts) / len(ts) if ts else None

    prefill_ms = mean_ms("p0", "p1")
    decode_ms = mean_ms("d0", "d1")
    full_call_ms = mean_ms("f0", "f1")

    # ---- end to end through the public API with host buffers
    h2d = d2h = 0
    if pre is not None:
        h2d += sum(t.numel() * t.element_size() for t in pre["host"].values())
        d2h += pre["host_out"].numel() * pre["host_out"].element_size()
    if dec_io is not None:
        h2d += dec_io["host_in"].numel()
        d2h += dec_io["host_out"].numel()

    def e2e_step(timing):
        if pre is not None:
            # host buffers in and out through the C ABI's host-memory prefill:
            # the copies of one sequence overlap the compute of the other
            h = pre["host"]
            timing["p0"].append(ev()); timing["p0"][-1].record(stream)
            fga.spark_attn_prefill_host(h["qkv"], h["gate"], h["pos"], PREFILL.layer,
                                        out=pre["host_out"], workspace=pre["ws_host"],
                                        stream=stream)
            timing["p1"].append(ev()); timing["p1"][-1].record(stream)
        if dec:
            # every layer's new-token inputs in one copy, every output in one read
            timing["d0"].append(ev()); timing["d0"][-1].record(stream)
            dec_io["dev_in"].copy_(dec_io["host_in"], non_blocking=True)
            for L in dec:
                d = L["dev"]
                fga.spark_attn_decode(d["qkv"], d["gate"], d["pos"], L["k"], L["v"],
                                      L["layer"], out=L["out"], workspace=L["ws"],
                                      stream=stream)
            dec_io["host_out"].copy_(dec_io["dev_out"], non_blocking=True)
            timing["d1"].append(ev()); timing["d1"][-1].record(stream)

    e2e_t = {k: [] for k in ("p0", "p1", "d0", "d1")}
    e2e_step({k: [] for k in e2e_t})
    torch.cuda.synchronize()
    dist_barrier(world)
    for _ in range(args.steps):
        e2e_step(e2e_t)
    torch.cuda.synchronize()
    dist_barrier(world)

    def mean_e2e(a, b):
        ts = [x.elapsed_time(y) for x, y in zip(e2e_t[a], e2e_t[b])]
        return sum(ts) / len(ts) if ts else 0.0

    e2e_prefill_ms = mean_e2e("p0", "p1")
    e2e_decode_ms = mean_e2e("d0", "d1")

    # device status words must be clean
    status = 0
    if pre is not None:
        status |= fga.spark_attn_read_status(pre["ws"])
    if pre is not None:
        status |= fga.spark_attn_read_status(pre["ws_host"])
    for L in dec:
        status |= fga.spark_attn_read_status(L["ws"])

    # ---- aggregate over ranks (replicas: work adds up, time is the slowest rank)
    total_ms_max = dist_max(total_ms, world)
    pf = prefill_flops(PREFILL) if pre is not None else 0.0
    kv_total, kv_full = decode_kv_bytes(layers)
    n_full = sum(1 for l in layers if l.kind == wl.FULL)
    prefill_ms_max = dist_max(prefill_ms or 0.0, world)
    decode_ms_max = dist_max(decode_ms or 0.0, world)
    full_ms_max = dist_max(full_call_ms or 0.0, world)
    e2e_prefill_max = dist_max(e2e_prefill_ms, world)
    e2e_decode_max = dist_max(e2e_decode_ms, world)
    status = int(dist_max(float(status), world))
    launches = args.steps * ((2 if pre is not None else 0) + decode_step_launches(dec))
    launches_all = int(dist_sum(float(launches), world))
    if rank != 0:
        return None

    prefill_tflops = world * pf / (prefill_ms_max * 1e9) if pre is not None else None
    decode_gbs = world * kv_total / (decode_ms_max * 1e6) if dec else None
    full_gbs = kv_full / (full_ms_max * 1e6) if n_full else None
    e2e_prefill_tflops = world * pf / (e2e_prefill_max * 1e9) if pre is not None else None
    e2e_decode_gbs = world * kv_total / (e2e_decode_max * 1e6) if dec else None

    if pre is not None:
        value, unit = prefill_tflops, "TFLOP/s"
        e2e_value = e2e_prefill_tflops
    else:
        value, unit = decode_gbs, "GB/s"
        e2e_value = e2e_decode_gbs

    rooflines = []
    if dec and n_full:
        rooflines.append({
            "kernel": "decode_split_kernel (+ decode_merge_kernel in the timed call)",
            "bound": "hbm", "achieved": full_gbs, "peak": hbm_peak, "unit": "GB/s",
            "frac": full_gbs / hbm_peak,
            "traffic": TRAFFIC.get("decode_split_kernel"),
            "algorithmic_per_launch": kv_full,
            "peak_source": f"{peak_src} hbm_gbs (copy)"})
    if pre is not None:
        achieved = pf / (prefill_ms_max * 1e9)
        rooflines.append({
            "kernel": "prefill_attn_kernel (+ prefill_rope_k_kernel in the timed call)",
            "bound": "tensor", "achieved": achieved, "peak": bf16_peak, "unit": "TFLOP/s",
            "frac": achieved / bf16_peak,
            "traffic": TRAFFIC.get("prefill_attn_kernel"),
            "algorithmic_per_launch": pf,
            "peak_source": f"{peak_src} bf16_tflops (burst)"})
    # the dominant kernel of the step by time
    if dec and pre is not None:
        dominant = rooflines[0] if (decode_ms_max > prefill_ms_max) else rooflines[1]
    else:
        dominant = rooflines[0]

    line = {
        "metric": METRIC,
        "value": value,
        "unit": unit,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": total_ms_max,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded normal activations and KV caches at the 4B model shapes)",
        "config": {
            "workload": (f"prefill 4B {'full' if PREFILL.layer.kind == wl.FULL else 'sliding'}"
                         "_attention B=2 T=8192 H=16 Hkv=4 + 1M-context "
                         "36-layer 4B decode step (9 full, 27 sliding)"
                         if (pre is not None and dec) else args.only),
            "prefill": {"B": PREFILL.B, "T": PREFILL.T, "H": PREFILL.H, "Hkv": PREFILL.Hkv,
                        "kind": "full" if PREFILL.layer.kind == wl.FULL else "sliding",
                        "window": PREFILL.layer.window if PREFILL.layer.kind == wl.SLIDING
                        else None,
                        "rope_theta": PREFILL.layer.theta, "rot_dim": PREFILL.layer.rot_dim}
            if pre else None,
            "decode": {"B": 1, "layers": len(dec), "full_layers": n_full,
                       "cached_tokens": DECODE_FULL.len_hi, "ring_slots": 512} if dec else None,
            "parallelism": f"replicas x{world}",
            "l2": "inputs larger than L2 (prefill qkv 201 MB; each full-layer cache 4 GiB)",
        },
        "prefill": {"ms": prefill_ms_max, "tflops": prefill_tflops,
                    "frac_bf16_peak": (prefill_tflops / world / bf16_peak) if pre else None,
                    "flops": pf} if pre is not None else None,
        "decode": {"ms": decode_ms_max, "kv_gbs": decode_gbs,
                   "frac_hbm_peak": (decode_gbs / world / hbm_peak) if dec else None,
                   "kv_bytes": kv_total, "full_layer_call_ms": full_ms_max,
                   "full_layer_kv_gbs": full_gbs} if dec else None,
        "roofline": dominant,
        "rooflines": rooflines,
        "e2e": {"value": e2e_value, "unit": unit, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "prefill_ms": e2e_prefill_max,
                "decode_ms": e2e_decode_max, "decode_kv_gbs": e2e_decode_gbs,
                "api": "prefill: spark_attn_prefill_host (C ABI with pinned host buffers; "
                       "per-sequence copies overlap the compute); decode: spark_attn_decode "
                       "for every layer, all layers' new-token inputs copied from pinned host "
                       "memory in one transfer and all outputs read back in one, every step"},
        "gpu_launches": launches_all,
        "clocks": clocks.summary(),
        "device_status": status,
    }
    if pre is not None and rank == 0:
        line["small_prefill"] = time_small_prefill(fga, dev, bf16_peak)
        line["layer_prefill"] = time_layer_prefill(fga, dev, bf16_peak)
        line["layer_prefill_sliding"] = time_layer_prefill(fga, dev, bf16_peak,
                                                           case=PREFILL_SLIDING_B2_T8192,
                                                           compare_gemms=False)
    if dec and rank == 0:
        line["layer_decode"] = time_layer_decode(fga, dev, dec, hbm_peak)
    if pre is not None and dec and rank == 0 and not args.no_other_configs:
        line["other_configs"] = time_other_configs(fga, dev, bf16_peak, hbm_peak)
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args, dec)
    return line


def time_small_prefill(fga, dev, bf16_peak, calls=50):
    """The 1.7B sliding_attention prefill (B=1, T=1024): 64 query tiles, far
    fewer than the SMs, so launch latency is a large part of a call.  Timed
    per call back to back, and as `calls` calls captured in one CUDA graph.
    Its 6 MB of inputs stay in L2 between calls."""
    import torch
    c = wl.PREFILL_SLIDING_1P7B_T1024
    x = wl.make_prefill_inputs(c)
    q, g, p = (x[k].to(dev) for k in ("qkv", "gate", "pos"))
    out = torch.empty((c.B, c.T, c.H * 256), dtype=torch.bfloat16, device=dev)
    ws = fga.new_workspace(fga.spark_attn_prefill_workspace_size(c.B, c.T, c.H, c.Hkv, c.layer),
                           dev)

    def call(stream):
        fga.spark_attn_prefill(q, g, p, c.layer, out=out, workspace=ws, stream=stream)

    side = torch.cuda.Stream(device=dev)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(5):
            call(side)
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(side)
        for _ in range(calls):
            call(side)
        s1.record(side)
    torch.cuda.synchronize()
    eager_ms = s0.elapsed_time(s1) / calls

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(calls):
            call(torch.cuda.current_stream())
    stream = torch.cuda.current_stream()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    graph.replay()
    g1.record(stream)
    torch.cuda.synchronize()
    graph_ms = g0.elapsed_time(g1) / calls
    status = fga.spark_attn_read_status(ws)
    flops = prefill_flops(c)
    return {
        "workload": "prefill 1.7B sliding_attention B=1 T=1024 H=8 Hkv=2 W=512",
        "flops": flops, "calls": calls, "l2": "resident (6 MB of inputs)",
        "eager_us_per_call": 1000.0 * eager_ms,
        "graph_us_per_call": 1000.0 * graph_ms,
        "tflops_eager": flops / eager_ms / 1e9,
        "tflops_graph": flops / graph_ms / 1e9,
        "frac_bf16_peak_graph": flops / graph_ms / 1e9 / bf16_peak,
        "device_status": status,
    }


def time_layer_prefill(fga, dev, bf16_peak, calls=10, case=None, compare_gemms=True):
    """The whole attention block of the benchmark's prefill layer (4B
    full_attention, B=2, T=8192, hidden 2560): q_k_v_proj and g_proj (one
    launch of the library's tcgen05 GEMM), the core, out_proj (the same GEMM),
    with seeded random weights of the model's shapes.  Work = the three
    projections' flops plus the core's algorithmic flops.  Beside it, the two
    projection GEMMs alone, through spark_attn_linear and through torch.matmul
    (cuBLAS) as a comparison that is not on the library's path."""
    import torch
    c = PREFILL if case is None else case
    hidden = 2560
    g = torch.Generator().manual_seed(11)
    x = torch.randn((c.B, c.T, hidden), generator=g).to(torch.bfloat16).to(dev)
    width = (c.H + 2 * c.Hkv) * 256
    w_qkv = (torch.randn((width, hidden), generator=g) / hidden ** 0.5).to(torch.bfloat16).to(dev)
    w_g = (torch.randn((c.H, hidden), generator=g) / hidden ** 0.5).to(torch.bfloat16).to(dev)
    w_o = (torch.randn((hidden, c.H * 256), generator=g) / (c.H * 256) ** 0.5).to(
        torch.bfloat16).to(dev)
    pos = torch.arange(c.T, dtype=torch.int32, device=dev).repeat(c.B, 1)
    y = torch.empty((c.B, c.T, hidden), dtype=torch.bfloat16, device=dev)
    ws = fga.new_workspace(fga.spark_attn_layer_prefill_workspace_size(c.B, c.T, hidden, c.H,
                                                                       c.Hkv, c.layer), dev)
    stream = torch.cuda.current_stream()

    def timed(fn, n):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    ms = timed(lambda: fga.spark_attn_layer_prefill(x, w_qkv, w_g, w_o, pos, c.layer, y=y,
                                                    workspace=ws, stream=stream), calls)
    rows = c.B * c.T
    proj = 2.0 * rows * hidden * (width + c.H + c.H * 256)
    flops = proj + prefill_flops(c)
    kind = "full" if c.layer.kind == wl.FULL else "sliding"
    res = {
        "workload": f"attention block of a 4B {kind}_attention prefill layer: q_k_v_proj "
                    f"2560->6144 (RoPE in its epilogue), g_proj 2560->16, core, out_proj "
                    f"4096->2560 (B={c.B} T={c.T}, random weights)",
        "ms": ms, "flops": flops, "projection_flops": proj,
        "tflops": flops / ms / 1e9, "frac_bf16_peak": flops / ms / 1e9 / bf16_peak,
        "calls": calls,
        "projections": "library tcgen05 GEMM (q_k_v_proj and g_proj in one launch; out_proj), "
                       "bf16 operands, fp32 accumulation in TMEM",
        "device_status": fga.spark_attn_read_status(ws),
    }
    if not compare_gemms:
        return res
    # the projection GEMMs alone (inputs resident; x and W stay in L2 between
    # calls, as they would inside the block)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    x2 = x.reshape(rows, hidden)
    a = torch.randn((rows, c.H * 256), generator=g).to(torch.bfloat16).to(dev)
    y_qkv = torch.empty((rows, width), dtype=torch.bfloat16, device=dev)
    gemms = {}
    for name, xx, ww, yy in (("q_k_v_proj", x2, w_qkv, y_qkv), ("out_proj", a, w_o,
                                                                 y.reshape(rows, hidden))):
        f = 2.0 * xx.shape[0] * xx.shape[1] * ww.shape[0]
        t_ours = timed(lambda: fga.spark_attn_linear(xx, ww, yy, device_status=status,
                                                     stream=stream), 20)
        t_ref = timed(lambda: torch.matmul(xx, ww.t(), out=yy), 20)
        gemms[name] = {"M": xx.shape[0], "N": ww.shape[0], "K": xx.shape[1], "flops": f,
                       "ours_ms": t_ours, "ours_tflops": f / t_ours / 1e9,
                       "ours_frac_bf16_peak": f / t_ours / 1e9 / bf16_peak,
                       "torch_cublas_ms": t_ref, "torch_cublas_tflops": f / t_ref / 1e9}
    res["projection_gemms"] = gemms
    res["device_status"] |= int(status.item())
    return res


def time_layer_decode(fga, dev, dec, hbm_peak, steps=5):
    """One decode step through all the attention blocks of the decode
    workload (the 36 layers of the 4B model at 1M context): per layer
    q_k_v_proj and g_proj of one hidden state (the library's GEMV), the core on that
    layer's cache, out_proj.  Seeded random weights of the model's shapes
    (1.9 GB for 36 layers).  Bytes = the core's KV read plus the projection
    weights, the two streams a decode step must read."""
    import torch
    hidden = 2560
    g = torch.Generator().manual_seed(12)
    blocks = []
    for L in dec:
        c = L["case"]
        width = (c.H + 2 * c.Hkv) * 256
        w_qkv = (torch.randn((width, hidden), generator=g) / hidden ** 0.5).to(torch.bfloat16)
        w_g = (torch.randn((c.H, hidden), generator=g) / hidden ** 0.5).to(torch.bfloat16)
        w_o = (torch.randn((hidden, c.H * 256), generator=g) / (c.H * 256) ** 0.5).to(
            torch.bfloat16)
        x = torch.randn((c.B, hidden), generator=g).to(torch.bfloat16)
        blocks.append({
            "w": [w_qkv.to(dev), w_g.to(dev), w_o.to(dev)], "x": x.to(dev),
            "y": torch.empty((c.B, hidden), dtype=torch.bfloat16, device=dev),
            "ws": fga.new_workspace(fga.spark_attn_layer_decode_workspace_size(
                c.B, hidden, c.H, c.Hkv, c.cap, L["layer"]), dev),
        })
    stream = torch.cuda.current_stream()

    def one_step():
        for L, bl in zip(dec, blocks):
            fga.spark_attn_layer_decode(bl["x"], *bl["w"], L["dev"]["pos"], L["k"], L["v"],
                                        L["layer"], y=bl["y"], workspace=bl["ws"], stream=stream)

    for _ in range(3):
        one_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        one_step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    # the same step captured in a CUDA graph, as a serving loop would replay it
    side = torch.cuda.Stream(device=dev)
    side.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph):
            cap_stream = torch.cuda.current_stream()
            for L, bl in zip(dec, blocks):
                fga.spark_attn_layer_decode(bl["x"], *bl["w"], L["dev"]["pos"], L["k"], L["v"],
                                            L["layer"], y=bl["y"], workspace=bl["ws"],
                                            stream=cap_stream)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(steps):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    graph_ms = e0.elapsed_time(e1) / steps
    kv, _ = decode_kv_bytes([L["layer"] for L in dec])
    weights = sum(sum(w.numel() * w.element_size() for w in bl["w"]) for bl in blocks)
    status = 0
    for bl in blocks:
        status |= fga.spark_attn_read_status(bl["ws"])
    gbs = (kv + weights) / ms / 1e6
    return {
        "workload": f"1M-context decode step through all {len(dec)} attention blocks "
                    "(q_k_v_proj + g_proj, core, out_proj; random weights), B=1",
        "ms": ms, "kv_bytes": kv, "weight_bytes": weights, "gbs": gbs,
        "frac_hbm_peak": gbs / hbm_peak, "steps": steps,
        "graph_ms": graph_ms, "graph_gbs": (kv + weights) / graph_ms / 1e6,
        "projections": "library weight-streaming GEMV (M = 1; g_proj in the q_k_v_proj "
                       "pass), fp32 accumulation",
        "device_status": status,
    }


def time_other_configs(fga, dev, bf16_peak, hbm_peak):
    """The remaining workloads of the benchmark's configuration list, each
    timed on its own (CUDA events, inputs resident): the long 4B prefill
    (B=1, T=65536) as a full and as a sliding layer, and the batched 4B decode
    (B=64, per-sequence lengths 4096..131072) on a full layer and on
    512-slot rings.  Not part of the timed step."""
    import torch
    out = {}
    stream = torch.cuda.current_stream()

    def timed(fn, calls):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(calls):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / calls

    for key, c, calls in (("long_prefill_full", wl.PREFILL_FULL_4B_T65536, 3),
                          ("long_prefill_sliding", wl.PREFILL_SLIDING_4B_T65536, 10)):
        x = wl.make_prefill_inputs(c)
        q, g, p = (x[k].to(dev) for k in ("qkv", "gate", "pos"))
        o = torch.empty((c.B, c.T, c.H * 256), dtype=torch.bfloat16, device=dev)
        ws = fga.new_workspace(fga.spark_attn_prefill_workspace_size(c.B, c.T, c.H, c.Hkv,
                                                                     c.layer), dev)
        ms = timed(lambda: fga.spark_attn_prefill(q, g, p, c.layer, out=o, workspace=ws,
                                                  stream=stream), calls)
        flops = prefill_flops(c)
        out[key] = {"workload": f"{c.name}: B={c.B} T={c.T} H={c.H} Hkv={c.Hkv}", "ms": ms,
                    "tflops": flops / ms / 1e9, "frac_bf16_peak": flops / ms / 1e9 / bf16_peak,
                    "device_status": fga.spark_attn_read_status(ws)}
        del q, g, p, o, ws, x
        torch.cuda.empty_cache()
    for key, c in (("batched_decode_full", wl.DECODE_FULL_4B_B64),
                   ("batched_decode_sliding", wl.DECODE_SLIDING_4B_B64)):
        step = wl.make_decode_step_inputs(c)
        k = torch.empty((c.B, c.Hkv, c.cap, 256), dtype=torch.bfloat16, device=dev)
        v = torch.empty_like(k)
        gen = torch.Generator(dev).manual_seed(c.seed)
        k.normal_(generator=gen)
        v.normal_(generator=gen)
        q, g, p = (step[n].to(dev) for n in ("qkv", "gate", "pos"))
        o = torch.empty((c.B, c.H * 256), dtype=torch.bfloat16, device=dev)
        ws = fga.new_workspace(fga.spark_attn_decode_workspace_size(c.B, c.H, c.Hkv, c.cap,
                                                                    c.layer), dev)
        # ~30 us per ring call: 50 calls so that the events' own overhead is small
        calls = 10 if c.layer.kind == wl.FULL else 50
        ms = timed(lambda: fga.spark_attn_decode(q, g, p, k, v, c.layer, out=o, workspace=ws,
                                                 stream=stream), calls)
        # visible tokens per sequence, the new one included (as for the step's decode)
        lens = step["pos"].long() + 1
        visible = lens if c.layer.kind == wl.FULL else lens.clamp(max=c.layer.window)
        kv = int(visible.sum()) * KV_BYTES_PER_TOKEN
        gbs = kv / ms / 1e6
        out[key] = {"workload": f"{c.name}: B={c.B}, lengths {c.len_lo}..{c.len_hi}, "
                                f"cache slots {c.cap}", "ms": ms, "kv_bytes": kv, "kv_gbs": gbs,
                    "frac_hbm_peak": gbs / hbm_peak,
                    "device_status": fga.spark_attn_read_status(ws)}
        del k, v, q, g, p, o, ws
        torch.cuda.empty_cache()
    return out


# Per-launch DRAM traffic (read + write bytes) from ncu captures of the
# current kernels, scaled to one launch of the bench workload; None when the
# kernels changed since the counters were taken.
# prefill_attn_kernel: 391.4 MB read + 100.1 MB written, measured on this
# workload (the two-issuer kernel with the two-chunk epilogue).  decode_split_kernel: 536.9 MB read +
# 3.7 MB written in a 131,072-token capture (split K/V barriers), scaled x8 to
# the 1,048,576-token layer (the traffic grows with the cached tokens).
TRAFFIC: dict[str, float | None] = {
    "decode_split_kernel": 540.666112e6 * 8,
    "prefill_attn_kernel": 491.444224e6,
}


# ---------------------------------------------------------------- oracle arm

_ORACLE_INPUTS = {}


def _prefill_inputs(case):
    if case.name not in _ORACLE_INPUTS:
        x = wl.make_prefill_inputs(case)
        _ORACLE_INPUTS[case.name] = (x, wl.bf16_bits(x["qkv"]))
    return _ORACLE_INPUTS[case.name]


def _visible(t, case):
    """Visible keys of query rows at token indices t (mask definition)."""
    import numpy as np
    t = np.asarray(t, np.int64)
    if case.layer.kind == wl.FULL:
        return t + 1
    return np.minimum(t + 1, case.layer.window)


def oracle_prefill_rows(case, n_rows: int, seed: int = 0):
    """Times the fp64 oracle on n_rows random query rows (all heads) of a
    prefill workload, or on all of it when n_rows >= B*T.  Returns (seconds,
    algorithmic flops of those rows, fraction of the workload's flops,
    description, the rows (None: all), the oracle's output for them)."""
    import numpy as np
    import oracle
    x, bits = _prefill_inputs(case)
    total_rows = case.B * case.T
    L = case.layer
    if n_rows >= total_rows:
        rows = None
        vis = _visible(np.arange(case.T), case).sum() * case.B
        desc = f"the whole {case.name} workload ({total_rows} query rows)"
    else:
        rng = np.random.default_rng(seed)
        rows = np.sort(rng.integers(0, total_rows, n_rows)).astype(np.int64)
        vis = _visible(rows % case.T, case).sum()
        desc = f"{n_rows} random query rows (all {case.H} heads) of {case.name}"
    t0 = time.perf_counter()
    want = oracle.prefill(bits, x["gate"].numpy(), x["pos"].numpy(), L.kind, L.window, L.theta,
                          L.rot_dim, case.H, case.Hkv, rows=rows, gate_mode=L.gate_mode)
    dt = time.perf_counter() - t0
    flops = 4.0 * 256 * case.H * float(vis)
    return dt, flops, flops / prefill_flops(case), desc, rows, want


def prefill_parity(case, rows, want):
    """The library's output for the same workload against the oracle rows
    just timed: max-abs and rel-L2 over every element of those rows, beside
    the bar the tests hold it to (max-abs <= 2e-2, rel-L2 <= 1e-2 against
    fp64).  Only the CPU-baseline leg calls this."""
    import numpy as np
    import torch
    import full_gqa_attention_gb300 as fga
    x, _ = _prefill_inputs(case)
    dev = torch.device("cuda", torch.cuda.current_device())
    out = fga.spark_attn_prefill(x["qkv"].to(dev), x["gate"].to(dev), x["pos"].to(dev),
                                 case.layer)
    got = out.reshape(case.B * case.T, -1)
    if rows is not None:
        got = got[torch.as_tensor(rows, device=dev)]
    got = got.float().cpu().double().numpy()
    want = np.asarray(want, dtype=np.float64).reshape(got.shape)
    max_abs = float(np.abs(got - want).max())
    rel_l2 = float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-30))
    return {"rows": int(got.shape[0]), "max_abs": max_abs, "rel_l2": rel_l2,
            "bar": {"max_abs": 2e-2, "rel_l2": 1e-2},
            "ok": bool(max_abs <= 2e-2 and rel_l2 <= 1e-2)}


def oracle_prefill_sample(n_rows: int, seed: int = 0):
    """The oracle on n_rows random query rows of the benchmark's prefill."""
    dt, flops, _, desc, _, _ = oracle_prefill_rows(PREFILL, n_rows, seed)
    return dt, flops, desc


def _sized(run, target_s: float, n0: int, n_max: int):
    """Calls run(n) with n growing from n0 until one call takes >= target_s
    seconds or n reaches n_max; returns the last call's result (time first)."""
    n = n0
    while True:
        res = run(n)
        if res[0] >= target_s or n >= n_max:
            return res
        n = min(n_max, int(n * min(8.0, max(2.0, 1.5 * target_s / max(res[0], 1e-3)))))


def oracle_decode_time(case, positions, k_bits, v_bits, parity=None, step=None, k_dev=None,
                       v_dev=None):
    """Seconds the fp64 oracle takes for one decode step of the given
    sequences (qkv / gate from `step`, else the workload's seeded step
    inputs).  With a ParityTally, the library's decode of the same step on the
    same caches (device copies of k_bits / v_bits, or k_dev / v_dev as they
    are) is compared with the oracle's output."""
    import numpy as np
    import oracle
    if step is None:
        step = wl.make_decode_step_inputs(wl.scaled(case, B=len(positions)))
    L = case.layer
    pos = np.asarray(positions, np.int32)
    t0 = time.perf_counter()
    want, _, _ = oracle.decode(wl.bf16_bits(step["qkv"]), step["gate"].numpy(), pos, k_bits,
                               v_bits, L.kind, L.window, L.theta, L.rot_dim, case.H, case.Hkv,
                               gate_mode=L.gate_mode)
    dt = time.perf_counter() - t0
    if parity is not None:
        parity.add(decode_on_device(case, step, pos, k_bits, v_bits, k_dev, v_dev), want)
    return dt


class ParityTally:
    """max-abs and rel-L2 of the library's outputs against the oracle's, over
    every element compared (the tests' bar: max-abs <= 2e-2, rel-L2 <= 1e-2
    against fp64).  Only the CPU-baseline leg uses it."""

    def __init__(self):
        self.n, self.max_abs, self.err2, self.ref2 = 0, 0.0, 0.0, 0.0

    def add(self, got, want):
        import numpy as np
        got = np.asarray(got, np.float64).reshape(-1)
        want = np.asarray(want, np.float64).reshape(-1)
        d = got - want
        self.n += 1
        self.max_abs = max(self.max_abs, float(np.abs(d).max()))
        self.err2 += float(d @ d)
        self.ref2 += float(want @ want)

    def result(self, what):
        rel = (self.err2 / self.ref2) ** 0.5 if self.ref2 > 0 else 0.0
        return {what: self.n, "max_abs": self.max_abs, "rel_l2": rel,
                "bar": {"max_abs": 2e-2, "rel_l2": 1e-2},
                "ok": bool(self.max_abs <= 2e-2 and rel <= 1e-2)}


def decode_on_device(case, step, pos, k_bits, v_bits, k_dev=None, v_dev=None):
    """The library's decode of one step, on device copies of the given caches
    (or on device caches given as they are); returns the output as float64."""
    import numpy as np
    import torch
    import full_gqa_attention_gb300 as fga
    dev = torch.device("cuda", torch.cuda.current_device())
    if k_dev is None:
        k_dev = torch.from_numpy(np.ascontiguousarray(k_bits).view(np.int16)).view(
            torch.bfloat16).to(dev)
        v_dev = torch.from_numpy(np.ascontiguousarray(v_bits).view(np.int16)).view(
            torch.bfloat16).to(dev)
    out = fga.spark_attn_decode(step["qkv"].to(dev), step["gate"].to(dev),
                                torch.as_tensor(pos, dtype=torch.int32).to(dev), k_dev, v_dev,
                                case.layer)
    return out.float().cpu().double().numpy()


def _cpu_cache(B, Hkv, n, seed):
    """A seeded bf16 cache [B, Hkv, n, 256] on the host, as bit patterns."""
    import torch
    c = torch.empty((B, Hkv, n, 256), dtype=torch.bfloat16)
    g = torch.Generator().manual_seed(seed)
    for b in range(B):
        c[b].copy_(torch.randn((Hkv, n, 256), generator=g).to(torch.bfloat16))
    return wl.bf16_bits(c)


def oracle_decode_batched(case, n_seq: int, seed: int = 0):
    """The oracle on n_seq of the batched decode workload's sequences (all 64
    when n_seq >= B), each at its own length, caches seeded on the host.
    Returns (seconds, KV bytes read, fraction of the workload's KV bytes,
    description, parity of the library's decode of the same sequences)."""
    import numpy as np
    lengths = wl.make_decode_lengths(case).numpy().astype(np.int64)
    if n_seq >= case.B:
        seqs = np.arange(case.B)
    else:
        seqs = np.sort(np.random.default_rng(seed).choice(case.B, n_seq, replace=False))
    visible = lambda p: (p + 1) if case.layer.kind == wl.FULL else min(p + 1, case.layer.window)  # noqa: E731
    dt, kv = 0.0, 0
    tally = ParityTally()
    if case.layer.kind == wl.SLIDING:
        # rings: every sequence in one oracle call
        pos = lengths[seqs]
        k = _cpu_cache(len(seqs), case.Hkv, case.cap, seed + 1)
        v = _cpu_cache(len(seqs), case.Hkv, case.cap, seed + 2)
        dt = oracle_decode_time(case, pos, k, v, tally)
        kv = sum(visible(int(p)) for p in pos) * KV_BYTES_PER_TOKEN
    else:
        for i, b in enumerate(seqs):
            p = int(lengths[b])
            k = _cpu_cache(1, case.Hkv, p + 1, seed + 3 * i + 1)
            v = _cpu_cache(1, case.Hkv, p + 1, seed + 3 * i + 2)
            dt += oracle_decode_time(case, [p], k, v, tally)
            kv += visible(p) * KV_BYTES_PER_TOKEN
            del k, v
    total = sum(visible(int(p)) for p in lengths) * KV_BYTES_PER_TOKEN
    what = "all" if len(seqs) == case.B else f"{len(seqs)} seeded-random"
    return (dt, kv, kv / total, f"{what} of the {case.B} sequences of {case.name}",
            tally.result("calls"))


def oracle_decode_1m(dec):
    """The oracle on one full layer (1,048,575 cached tokens, the cache read
    back from the benchmark's own device copy) and one sliding layer of the
    1M-context decode step; the 36-layer step is extrapolated as 9 full + 27
    sliding layers.  Returns (step seconds extrapolated, KV bytes of the
    step, seconds measured, description, parity of the library's decode of
    those two layers against the oracle's)."""
    full = next((L for L in dec if L["layer"].kind == wl.FULL), None)
    slid = next((L for L in dec if L["layer"].kind == wl.SLIDING), None)
    n_full = sum(1 for L in dec if L["layer"].kind == wl.FULL)
    n_slid = len(dec) - n_full
    measured, t_full, t_slid = 0.0, 0.0, 0.0
    tally = ParityTally()
    for L, kind in ((full, "full"), (slid, "sliding")):
        if L is None:
            continue
        c = L["case"]
        p = int(L["host"]["pos"][0])
        n = min(p + 1, c.cap) if kind == "full" else c.cap
        k = wl.bf16_bits(L["k"][:, :, :n].cpu())
        v = wl.bf16_bits(L["v"][:, :, :n].cpu())
        # the layer's own step inputs; the library's decode of the same step runs
        # on the benchmark's own caches (each step rewrites slot p with the same
        # key and value)
        t = oracle_decode_time(c, [p], k, v, tally, step=L["host"], k_dev=L["k"], v_dev=L["v"])
        del k, v
        measured += t
        if kind == "full":
            t_full = t
        else:
            t_slid = t
    step_s = n_full * t_full + n_slid * t_slid
    kv, _ = decode_kv_bytes([L["layer"] for L in dec])
    return step_s, kv, measured, (f"one full layer (1,048,575 cached tokens) and one sliding "
                                  f"layer, extrapolated to the {n_full} + {n_slid} layers of "
                                  "the step"), tally.result("layers")


def cpu_threads() -> int:
    """Threads the OpenMP oracle runs with (its default: the usable cores)."""
    n = os.environ.get("OMP_NUM_THREADS")
    if n and n.isdigit():
        return int(n)
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(args, dec=None):
    """The fp64 oracle, as it stands, on host cores, beside every workload the
    line reports: bounded samples (~25 s of CPU in all), each extrapolated to
    its whole workload where it is a sample.  The headline entry is the
    benchmark's prefill; per_config holds one entry per workload."""
    cores = cpu_threads()
    per = {}

    def prefill_entry(case, target_s, n0):
        total_rows = case.B * case.T
        if target_s is None:
            dt, flops, frac, desc, rows, want = oracle_prefill_rows(case, total_rows)
        else:
            dt, flops, frac, desc, rows, want = _sized(lambda n: oracle_prefill_rows(case, n),
                                                       target_s, n0, total_rows)
        e = {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
             "sample": desc + f", {dt:.2f} s", "seconds": dt,
             "parity": prefill_parity(case, rows, want)}
        if frac < 1.0:
            e["workload_seconds_extrapolated"] = dt / frac
        return e

    per["small_prefill_1.7b_sliding_T1024"] = prefill_entry(wl.PREFILL_SLIDING_1P7B_T1024,
                                                            None, 0)
    per["prefill_4b_full_B2_T8192"] = prefill_entry(PREFILL, 5.0, 64)
    per["long_prefill_full_T65536"] = prefill_entry(wl.PREFILL_FULL_4B_T65536, 3.0, 16)
    per["long_prefill_sliding_T65536"] = prefill_entry(wl.PREFILL_SLIDING_4B_T65536, 3.0, 256)
    for key, case, n in (("batched_decode_full_B64", wl.DECODE_FULL_4B_B64, 8),
                         ("batched_decode_sliding_B64", wl.DECODE_SLIDING_4B_B64, 64)):
        dt, kv, frac, desc, par = oracle_decode_batched(case, n)
        e = {"value": kv / dt / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
             "sample": desc + f", {dt:.2f} s", "seconds": dt, "parity": par}
        if frac < 1.0:
            e["workload_seconds_extrapolated"] = dt / frac
        per[key] = e
    if dec:
        step_s, kv, measured, desc, par = oracle_decode_1m(dec)
        per["decode_step_1m_36_layers"] = {
            "value": kv / step_s / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": desc + f", {measured:.2f} s measured", "seconds": measured,
            "workload_seconds_extrapolated": step_s, "parity": par}
    head = per["prefill_4b_full_B2_T8192"]
    return {"value": head["value"], "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": head["sample"], "per_config": per}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    rows = 256
    dt, flops, desc = oracle_prefill_sample(rows, seed=1)
    # size the sample so the whole run stays within a few minutes
    per_row = dt / rows
    rows = max(8, min(4096, int(8.0 / max(per_row, 1e-6))))
    for _ in range(args.warmup):
        oracle_prefill_sample(max(8, rows // 8), seed=2)
    times, total_flops = [], 0.0
    for k in range(args.steps):
        dt, flops, desc = oracle_prefill_sample(rows, seed=10 + k)
        times.append(dt)
        total_flops += flops
    secs = sum(times)
    value = total_flops / secs / 1e12
    ms_per_step = 1000.0 * secs / args.steps
    return {
        "impl": "reference",
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded normal activations at the 4B model shapes)",
        "config": {"workload": "prefill 4B full_attention B=2 T=8192 H=16 Hkv=4 (oracle on a "
                               "sample of query rows per step)",
                   "parallelism": "host cores"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_threads(),
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


# ---------------------------------------------------------------- one workload alone

SINGLE = ("gemm_qkv", "gemm_out", "ring_decode_b64", "full_decode_b64", "small_prefill",
          "prefill_full_B2_T8192", "prefill_sliding_B2_T8192", "prefill_sliding_T65536",
          "layer_prefill_full", "layer_prefill_sliding")


def run_single(name: str, steps: int, warmup: int):
    """Runs one workload alone, warmup + steps calls on one stream, and returns a
    short JSON-able record with the mean time per timed call (CUDA events).  For
    profiler captures of one kernel (ncu -s <launches to skip> -c 1)."""
    import torch
    import full_gqa_attention_gb300 as fga
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    g = torch.Generator(dev).manual_seed(0)
    fn = None
    if name in ("gemm_qkv", "gemm_out"):
        M, N, K = (16384, 6144, 2560) if name == "gemm_qkv" else (16384, 2560, 4096)
        x = torch.randn((M, K), generator=g, device=dev).to(torch.bfloat16)
        w = (torch.randn((N, K), generator=g, device=dev) / K ** 0.5).to(torch.bfloat16)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        fn = lambda: fga.spark_attn_linear(x, w, y, device_status=st)  # noqa: E731
        work = {"flops": 2.0 * M * N * K}
    elif name in ("ring_decode_b64", "full_decode_b64"):
        c = wl.DECODE_SLIDING_4B_B64 if name == "ring_decode_b64" else wl.DECODE_FULL_4B_B64
        step = wl.make_decode_step_inputs(c)
        k = torch.empty((c.B, c.Hkv, c.cap, 256), dtype=torch.bfloat16, device=dev)
        v = torch.empty_like(k)
        k.normal_(generator=g)
        v.normal_(generator=g)
        q, gt, p = (step[n].to(dev) for n in ("qkv", "gate", "pos"))
        o = torch.empty((c.B, c.H * 256), dtype=torch.bfloat16, device=dev)
        ws = fga.new_workspace(fga.spark_attn_decode_workspace_size(c.B, c.H, c.Hkv, c.cap,
                                                                    c.layer), dev)
        fn = lambda: fga.spark_attn_decode(q, gt, p, k, v, c.layer, out=o, workspace=ws)  # noqa: E731
        lens = step["pos"].long() + 1
        vis = lens if c.layer.kind == wl.FULL else lens.clamp(max=c.layer.window)
        work = {"kv_bytes": int(vis.sum()) * KV_BYTES_PER_TOKEN}
    elif name in ("small_prefill", "prefill_full_B2_T8192", "prefill_sliding_B2_T8192",
                  "prefill_sliding_T65536"):
        c = {"small_prefill": wl.PREFILL_SLIDING_1P7B_T1024, "prefill_full_B2_T8192": PREFILL,
             "prefill_sliding_B2_T8192": PREFILL_SLIDING_B2_T8192,
             "prefill_sliding_T65536": wl.PREFILL_SLIDING_4B_T65536}[name]
        x = wl.make_prefill_inputs(c)
        q, gt, p = (x[n].to(dev) for n in ("qkv", "gate", "pos"))
        o = torch.empty((c.B, c.T, c.H * 256), dtype=torch.bfloat16, device=dev)
        ws = fga.new_workspace(fga.spark_attn_prefill_workspace_size(c.B, c.T, c.H, c.Hkv,
                                                                     c.layer), dev)
        fn = lambda: fga.spark_attn_prefill(q, gt, p, c.layer, out=o, workspace=ws)  # noqa: E731
        work = {"flops": prefill_flops(c)}
    elif name in ("layer_prefill_full", "layer_prefill_sliding"):
        c = PREFILL if name == "layer_prefill_full" else PREFILL_SLIDING_B2_T8192
        hidden, width = 2560, (c.H + 2 * c.Hkv) * 256
        x = torch.randn((c.B, c.T, hidden), generator=g, device=dev).to(torch.bfloat16)
        w_qkv = (torch.randn((width, hidden), generator=g, device=dev) / hidden ** 0.5).to(
            torch.bfloat16)
        w_g = (torch.randn((c.H, hidden), generator=g, device=dev) / hidden ** 0.5).to(
            torch.bfloat16)
        w_o = (torch.randn((hidden, c.H * 256), generator=g, device=dev) / 64.0).to(
            torch.bfloat16)
        pos = torch.arange(c.T, dtype=torch.int32, device=dev).repeat(c.B, 1)
        y = torch.empty((c.B, c.T, hidden), dtype=torch.bfloat16, device=dev)
        ws = fga.new_workspace(fga.spark_attn_layer_prefill_workspace_size(
            c.B, c.T, hidden, c.H, c.Hkv, c.layer), dev)
        fn = lambda: fga.spark_attn_layer_prefill(x, w_qkv, w_g, w_o, pos, c.layer, y=y,  # noqa: E731
                                                  workspace=ws)
        work = {"flops": 2.0 * c.B * c.T * hidden * (width + c.H + c.H * 256) + prefill_flops(c)}
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / max(steps, 1)
    rec = {"single": name, "steps": steps, "warmup": warmup, "ms_per_call": ms, **work}
    if "flops" in work:
        rec["tflops"] = work["flops"] / ms / 1e9
    if "kv_bytes" in work:
        rec["kv_gbs"] = work["kv_bytes"] / ms / 1e6
    return rec


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--only", choices=("all", "prefill", "decode"), default="all")
    ap.add_argument("--decode-layers", type=int, default=36)
    ap.add_argument("--decode-cache-tokens", type=int, default=None,
                    help="cached tokens of each full decode layer (default 1,048,575); "
                         "smaller values are for profiler captures")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-other-configs", action="store_true",
                    help="skip the extra lines for the long prefill and the batched decode")
    ap.add_argument("--single", choices=SINGLE, default=None,
                    help="time one workload alone (for profiler captures of one kernel)")
    ap.add_argument("--prefill-layer", choices=("full", "sliding"), default="full",
                    help="layer type of the prefill workload (sliding: for profiling; the "
                         "benchmark's workload is the full layer)")
    args = ap.parse_args(argv)
    if args.single:
        print(json.dumps(run_single(args.single, args.steps, args.warmup)), flush=True)
        return
    if args.warmup < 3 and args.impl == "ours":
        print("bench.py: warmup raised to 3", file=sys.stderr)
        args.warmup = 3
    if args.prefill_layer == "sliding":
        global PREFILL
        PREFILL = PREFILL_SLIDING_B2_T8192
    if args.decode_cache_tokens is not None:
        global DECODE_FULL
        n = args.decode_cache_tokens
        DECODE_FULL = wl.scaled(DECODE_FULL, cap=n + 1, len_lo=n, len_hi=n)
    rank, world, local = dist_setup()
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        line = run_ours(args, rank, world, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
