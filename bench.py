#!/usr/bin/env python3
"""Benchmark of the B300 selective scan (and the Mamba-2 SSD scan).

One step = one full selective-scan call (discretise, recurrence, readout,
skip, gate, final state) over the long-context workload: batch 1, d_inner
2048, d_state 16, L 262144, bf16 inputs, fp32 state, no z gate.  Inputs are
resident in HBM when the timed region starts; L2 is flushed (a 256 MB write)
before every timed step, outside the step's events.

Prints ONE JSON line (rank 0): channel-steps/s, the HBM roofline of the scan
kernel (with the MUFU exponential rate beside it, against the rate
ss_probe_ex2_rate measures in the same run), the end-to-end number through
the C ABI with host buffers, the fp64 oracle timed on the host cores, clocks
seen during the timed region, a full record (the same fields) for each of the
other benchmark workloads (the Mamba-130M and Mamba-2.8B layers and the
Mamba-2 SSD layer), and timing rows for the rest.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun every rank runs its own replica of the workload (weak
scaling); value = all ranks' channel-steps / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "selective-scan channel-steps/s (B·D·L/s) and achieved HBM GB/s vs B300 peak"
UNIT = "channel-steps/s"
HEADLINE = "long_context"
# the other benchmark workloads, each measured with the same fields as the headline
FULL_ROWS = ("mamba130m_layer", "mamba2p8b_layer", "mamba2_ssd")
L2_FLUSH_BYTES = 256 << 20
FALLBACK_HBM_GBS = 6400.0
FALLBACK_BF16_TFLOPS = 1800.0
# nominal B300 HBM3e bandwidth, for the fraction next to the measured one
NOMINAL_HBM_GBS = 7700.0
N_SM = 148
SM_MHZ_MAX = 2032.0

WORKLOAD_TEXT = {
    "long_context": "long-context scan, batch 1, d_inner 2048, d_state 16, L 262144, bf16 "
                    "inputs, fp32 state, no z gate, delta softplus with bias (dt log-uniform in "
                    "[1e-4, 1e-1]), final state returned",
    "mamba130m_layer": "Mamba-130M-shaped layer scan, batch 8, d_inner 1536, d_state 16, "
                       "L 2048, bf16 inputs, fp32 state, z gate on, delta softplus with bias, "
                       "final state returned",
    "mamba2p8b_layer": "Mamba-2.8B-shaped layer scan, batch 4, d_inner 5120, d_state 16, "
                       "L 8192, bf16 inputs, fp32 state, z gate on, delta softplus with bias, "
                       "final state returned",
    "mamba2_ssd": "Mamba-2 SSD chunked scan, batch 4, L 8192, 64 heads x headdim 64, d_state "
                  "128, ngroups 1, chunk 256, bf16 inputs, fp32 state, D skip, final state "
                  "returned",
    "tiny_f32": "tiny selective scan, batch 1, d_inner 64, d_state 16, L 256, fp32, z gate on",
}


def mufu_ops_per_channel_step(cfg):
    """MUFU operations the selective scan needs per channel-step, counted in
    ex2-equivalents: the N exponentials exp(delta A), softplus's exponential
    (its logarithm runs on the FMA pipe), and with a z gate the sigmoid's
    exponential and reciprocal (a reciprocal takes two ex2 slots)."""
    return cfg.d_state + (1 if cfg.softplus else 0) + (3 if cfg.gate else 0)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-rows", action="store_true", help="skip the secondary workload rows")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU baseline")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--probe-mufu", action="store_true",
                    help="print the measured ex2.approx rate (per SM per clock) and exit")
    ap.add_argument("--probe-scan-forms", action="store_true",
                    help="print the channel-steps/s of the sequential and the warp-shuffle "
                         "scan forms on synthetic tiles and exit")
    ap.add_argument("--profile", default=None, metavar="WORKLOAD",
                    help="run WORKLOAD's call warmup+steps times with no timing or output "
                         "(for ncu captures): a workload name, bwd_mamba130m_layer, "
                         "conv_mamba130m_layer, per_channel_bc_mamba130m_layer, "
                         "mamba130m_layer_N64, decode_mamba2_ssd, or WORKLOAD:L (a "
                         "benchmark workload with sequence length L)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# Algorithmic work per call.


def selective_bytes(cfg):
    es = 2 if cfg.dtype == "bf16" else 4
    steps = cfg.batch * cfg.d_inner * cfg.seqlen
    per_step = es * (3 + (1 if cfg.gate else 0))           # u, delta, (z) in; y out
    bc = 2 * cfg.batch * cfg.d_state * cfg.seqlen * es       # B and C, read once
    params = 4 * cfg.d_inner * (cfg.d_state + int(cfg.skip) + int(cfg.bias))  # A, D, delta_bias
    state = 4 * cfg.batch * cfg.d_inner * cfg.d_state if cfg.last_state else 0
    return steps * per_step + bc + params + state


def ssd_bytes(cfg):
    es = 2 if cfg.dtype == "bf16" else 4
    xy = 2 * cfg.batch * cfg.seqlen * cfg.nheads * cfg.headdim * es
    dt = cfg.batch * cfg.seqlen * cfg.nheads * es
    bc = 2 * cfg.batch * cfg.seqlen * cfg.ngroups * cfg.d_state * es
    state = 4 * cfg.batch * cfg.nheads * cfg.headdim * cfg.d_state if cfg.last_state else 0
    return xy + dt + bc + 4 * cfg.nheads * (1 + int(cfg.skip)) + state  # + A_head, D


def ssd_flops(cfg):
    """Dense-contraction flops of the chunked form (C B^T once per group)."""
    Q, nch = cfg.chunk, -(-cfg.seqlen // cfg.chunk)
    per_head_chunk = 2 * Q * Q * cfg.headdim + 4 * Q * cfg.headdim * cfg.d_state
    cb = 2 * Q * Q * cfg.d_state * cfg.ngroups
    return cfg.batch * nch * (cfg.nheads * per_head_chunk + cb)


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        return float(m["hbm_gbs"]), float(m["bf16_tflops"]), float(
            m.get("bf16_tflops_sustained", m["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1400.0, "fallback"


# The source files each measured kernel's device code is built from (the
# kernels take their own parameter structs, so the host-side declarations in
# internal.h do not enter).
KERNEL_SOURCES = {
    "scan_seq<bf16, 1 lane/channel>": ["selective_scan_seq.cu", "scan_common.cuh", "ptx.cuh"],
    "scan_seq<bf16, 2 lanes/channel>": ["selective_scan_seq.cu", "scan_common.cuh", "ptx.cuh"],
    "scan_seq<bf16, 4 lanes/channel>": ["selective_scan_seq.cu", "scan_common.cuh", "ptx.cuh"],
    "ssd_chunk_tc2": ["ssd_tc.cu", "tc.cuh", "ptx.cuh"],
    "scan_bwd_fast<bf16>": ["selective_scan_bwd.cu", "ptx.cuh"],
}


def _code_only(text):
    """C/C++ source without comments and blank lines: edits to comments do
    not change the kernel."""
    out, i, n = [], 0, len(text)
    while i < n:
        if text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        elif text[i] == '"':
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(text[i])
            i += 1
    lines = ("".join(out)).splitlines()
    return "\n".join(ln.rstrip() for ln in lines if ln.strip())


def source_hash(files=None):
    h = hashlib.sha256()
    d = os.path.join(ROOT, "selective_state_space_146_b300", "csrc")
    names = files or sorted(f for f in os.listdir(d) if f.endswith((".cu", ".cuh", ".h")))
    for f in names:
        with open(os.path.join(d, f), encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def measured_traffic(kernel_key):
    """DRAM bytes per launch from a committed ncu capture, if it was taken on
    the kernel's current sources (else None)."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)
        e = t[kernel_key]
        cur = source_hash(KERNEL_SOURCES.get(kernel_key))
        return e["bytes_per_launch"] if e.get("source_hash") == cur else None
    except Exception:
        return None


# ---------------------------------------------------------------------------
# Clock sampling during the timed region.


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.lines = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.gpu)], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=3)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            p = [x.strip() for x in ln.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                smax.append(float(p[2]))
                power.append(float(p[3]))
            except ValueError:
                continue
            for nm, v in zip(names, p[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------------------
# GPU timing.


def time_device(fn, flush, steps, warmup, torch, counter=None):
    """Per-step CUDA-event times (ms) of fn() on the current stream, with an
    L2 flush before every step outside the events.  With `counter`, also
    returns how many library kernels the timed steps launched."""
    st = torch.cuda.current_stream()
    for _ in range(warmup):
        flush.zero_()
        fn()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    n0 = counter() if counter else 0
    for a, b in evs:
        flush.zero_()
        a.record(st)
        fn()
        b.record(st)
    n1 = counter() if counter else 0
    torch.cuda.synchronize()
    times = [a.elapsed_time(b) for a, b in evs]
    return (times, n1 - n0) if counter else times


def run_selective_call(g, torch, abi, y, last):
    abi.selective_scan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"],
                           g["delta_bias"], softplus=True, y=y, last_state=last)


def _selective_device_inputs(cfg, dev, rank, inputs):
    host = inputs.workload_selective_inputs(cfg, seed=rank)
    g = {k: (None if v is None else v.to(dev)) for k, v in host.items()}
    return host, g


def measure_workload(name, args, dev, rank, torch, abi, inputs, dist_helpers, clocks=False):
    """One benchmark workload measured in full: device-resident timing of
    `args.steps` calls (L2 flushed before each), the library kernels they
    launched, the end-to-end time with host buffers, and (optionally) the SM
    clocks during the timed region."""
    cfg = inputs.WORKLOADS[name]
    ssd = name == "mamba2_ssd"
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    if ssd:
        host = inputs.workload_ssd_inputs(cfg, seed=rank)
        g = {k: (None if v is None else v.to(dev)) for k, v in host.items()}
        y = torch.empty_like(g["x"])
        last = torch.empty(cfg.batch, cfg.nheads, cfg.headdim, cfg.d_state, device=dev)

        def step():
            abi.ssd_chunk_scan_fwd(g["x"], g["dt"], g["A_head"], g["B"], g["C"], g["D"],
                                   chunk=cfg.chunk, y=y, last_state=last)
    else:
        host, g = _selective_device_inputs(cfg, dev, rank, inputs)
        y = torch.empty_like(g["u"])
        last = torch.empty(cfg.batch, cfg.d_inner, cfg.d_state, dtype=torch.float32, device=dev)

        def step():
            run_selective_call(g, torch, abi, y, last)

    dist_helpers.barrier(dev)
    torch.cuda.synchronize()
    if clocks:
        with ClockSampler(dev.index if dev.index is not None else 0) as clk:
            times, launches = time_device(step, flush, args.steps, args.warmup, torch,
                                          counter=abi.launch_count)
        clk_summary = clk.summary()
    else:
        times, launches = time_device(step, flush, args.steps, args.warmup, torch,
                                      counter=abi.launch_count)
        clk_summary = None
    torch.cuda.synchronize()
    dist_helpers.barrier(dev)
    ms = statistics.mean(times)
    ms_max = dist_helpers.max_over_ranks(ms, dev)

    # end to end: inputs in pinned host memory, copied in and the results
    # copied out inside every timed step
    pinned = {k: (None if v is None else v.pin_memory()) for k, v in host.items()}
    y_h = torch.empty(y.shape, dtype=y.dtype).pin_memory()
    last_h = torch.empty(last.shape, dtype=last.dtype).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in pinned.values() if v is not None)
    d2h = y_h.numel() * y_h.element_size() + last_h.numel() * last_h.element_size()
    if ssd:
        def e2e_step():
            # host buffers in, host buffers out: the library chunks the batch
            # rows (or a row's heads) and overlaps copies with the scan on two
            # streams
            abi.ssd_chunk_scan_fwd_host(pinned["x"], pinned["dt"], pinned["A_head"], pinned["B"],
                                        pinned["C"], pinned["D"], chunk=cfg.chunk, y=y_h,
                                        last_state=last_h)
        call = "ss_ssd_chunk_scan_fwd_host (pinned host tensors in and out)"
    else:
        def e2e_step():
            # host buffers in, host buffers out: the library chunks the rows and
            # overlaps copies with the scan on two streams
            abi.selective_scan_fwd_host(pinned["u"], pinned["delta"], pinned["A"], pinned["B"],
                                        pinned["C"], pinned["D"], pinned["z"],
                                        pinned["delta_bias"], softplus=True, y=y_h,
                                        last_state=last_h)
        call = "ss_selective_scan_fwd_host (pinned host tensors in and out)"
    e2e_times = time_device(e2e_step, flush, max(3, args.steps // 2), 2, torch)
    e2e_ms = dist_helpers.max_over_ranks(statistics.mean(e2e_times), dev)

    units = cfg.channel_steps
    total_units = dist_helpers.sum_over_ranks(units, dev)
    out = dict(cfg=cfg, host=host, ms=ms, ms_max=ms_max, times=times, launches=launches,
               clocks=clk_summary, e2e_ms=e2e_ms, h2d=h2d, d2h=d2h, units=units,
               total_units=total_units, e2e_call=call)
    del g, y, last, pinned, y_h, last_h
    torch.cuda.empty_cache()
    return out


def secondary_rows(dev, torch, abi, inputs, hbm_peak, tf_peak, mufu_peak):
    """Timing of the workloads outside the benchmark set (inputs drawn on the
    GPU with the same recipe; parity for these shapes is covered by tests/)."""
    rows = {}
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    for name in ("tiny_f32",):
        cfg = inputs.WORKLOADS[name]
        try:
            with inputs.on_device(dev):
                if name == "mamba2_ssd":
                    g = inputs.workload_ssd_inputs(cfg)
                else:
                    g = inputs.workload_selective_inputs(cfg)
            if name == "mamba2_ssd":
                yb = torch.empty_like(g["x"])
                ls = torch.empty(cfg.batch, cfg.nheads, cfg.headdim, cfg.d_state, device=dev)

                def fn():
                    abi.ssd_chunk_scan_fwd(g["x"], g["dt"], g["A_head"], g["B"], g["C"], g["D"],
                                           chunk=cfg.chunk, y=yb, last_state=ls)
                nbytes = ssd_bytes(cfg)
            else:
                yb = torch.empty_like(g["u"])
                ls = torch.empty(cfg.batch, cfg.d_inner, cfg.d_state, device=dev)

                def fn():
                    run_selective_call(g, torch, abi, yb, ls)
                nbytes = selective_bytes(cfg)
            times, nl = time_device(fn, flush, 5, 3, torch, counter=abi.launch_count)
            launches_per_call = nl / 5
            ms = statistics.mean(times)
            gbs = nbytes / (ms * 1e-3) / 1e9
            row = {"ms_per_call": round(ms, 4), "channel_steps_per_s": cfg.channel_steps / (ms * 1e-3),
                   "hbm_gbs": round(gbs, 1), "hbm_frac": round(gbs / hbm_peak, 4),
                   "launches_per_call": launches_per_call}
            if name == "mamba2_ssd":
                # executed MMA flops of the 128-step block form: C B^T once per
                # pair of heads of a group (once per head for odd heads per group)
                nblk = -(-cfg.seqlen // 128)
                P, N, Q = cfg.headdim, cfg.d_state, 128
                cb_share = 2 if (cfg.nheads // cfg.ngroups) % 2 == 0 else 1
                ex = cfg.batch * cfg.nheads * nblk * 2 * Q * (Q * N / cb_share + P * N + Q * P + N * P)
                tf = ex / (ms * 1e-3) / 1e12
                row["tensor_tflops_executed"] = round(tf, 1)
                row["tensor_tflops_algorithmic"] = round(ssd_flops(cfg) / (ms * 1e-3) / 1e12, 1)
                row["tensor_peak_tflops"] = tf_peak
                row["tensor_frac"] = round(tf / tf_peak, 4)
                row["traffic"] = measured_traffic("ssd_chunk_tc2")
            rows[name] = row
            del g, yb, ls
            torch.cuda.empty_cache()
        except Exception as e:  # a row failing must not hide the headline
            rows[name] = {"error": str(e)[:200]}
    try:
        cfg = inputs.WORKLOADS["mamba130m_layer"]
        with inputs.on_device(dev):
            g = inputs.workload_selective_inputs(cfg)
        gen = torch.Generator(device=dev).manual_seed(7)
        cw = torch.randn(cfg.d_inner, 4, generator=gen, device=dev) * 0.5
        cb = torch.randn(cfg.d_inner, generator=gen, device=dev) * 0.1
        yb = torch.empty_like(g["u"])
        ls = torch.empty(cfg.batch, cfg.d_inner, cfg.d_state, device=dev)

        def fn():
            abi.conv_selective_scan_fwd(g["u"], cw, cb, g["delta"], g["A"], g["B"], g["C"],
                                        g["D"], g["z"], g["delta_bias"], y=yb, last_state=ls)
        times, nl = time_device(fn, flush, 5, 3, torch, counter=abi.launch_count)
        ms = statistics.mean(times)
        nbytes = selective_bytes(cfg)  # x replaces u; the conv taps are negligible
        rows["conv_scan_mamba130m_layer"] = {
            "ms_per_call": round(ms, 4), "channel_steps_per_s": cfg.channel_steps / (ms * 1e-3),
            "hbm_gbs": round(nbytes / (ms * 1e-3) / 1e9, 1), "launches_per_call": nl / 5,
            "note": "causal conv1d (width 4) + SiLU fused in front of the scan"}
        del g, yb
    except Exception as e:
        rows["conv_scan_mamba130m_layer"] = {"error": str(e)[:200]}
    rows.update(length_sweep_rows(dev, torch, abi, inputs, hbm_peak, flush))
    rows.update(grouped_rows(dev, torch, abi, inputs, hbm_peak, flush))
    rows.update(odd_length_rows(dev, torch, abi, inputs, hbm_peak, flush))
    rows.update(wide_state_rows(dev, torch, abi, inputs, hbm_peak, flush, mufu_peak))
    rows.update(backward_rows(dev, torch, abi, inputs, hbm_peak, flush))
    rows.update(decode_rows(dev, torch, abi, inputs, hbm_peak))
    return rows


def length_sweep_rows(dev, torch, abi, inputs, hbm_peak, flush):
    """Scan-only length sweep (batch 1, d_inner 2048 = d_model 1024 x expand
    2, N 16, bf16, gate on): time per call should grow linearly in L."""
    out = {}
    for L in (1024, 2048, 4096, 8192, 16384):
        try:
            with inputs.on_device(dev):
                g = inputs.selective_inputs(1, 2048, 16, L, "bf16", seed=L)
            yb = torch.empty_like(g["u"])
            ls = torch.empty(1, 2048, 16, device=dev)

            def fn():
                run_selective_call(g, torch, abi, yb, ls)
            times, nl = time_device(fn, flush, 5, 3, torch, counter=abi.launch_count)
            ms = statistics.mean(times)
            out[str(L)] = {"ms_per_call": round(ms, 4),
                           "channel_steps_per_s": 2048 * L / (ms * 1e-3),
                           "launches_per_call": nl / 5}
            del g, yb, ls
        except Exception as ex:
            out[str(L)] = {"error": str(ex)[:200]}
    return {"length_sweep_d2048": {"by_L": out, "note": "batch 1, d_inner 2048, N 16, bf16; "
                                   "few channels, so the sequence is split into segments "
                                   "(summary pass + main pass)"}}


def odd_length_rows(dev, torch, abi, inputs, hbm_peak, flush):
    """The Mamba-130M layer one step short (8 x 1536 x 2047, bf16, gate on):
    rows of 4094 bytes, not a multiple of 16, so the call runs the TMA kernels
    on padded copies of its rows (the copies counted in the launches)."""
    import dataclasses
    base = inputs.WORKLOADS["mamba130m_layer"]
    cfg = dataclasses.replace(base, seqlen=base.seqlen - 1)
    name = "odd_length_mamba130m_layer"
    try:
        with inputs.on_device(dev):
            g = inputs.workload_selective_inputs(cfg)
        yb = torch.empty_like(g["u"])
        ls = torch.empty(cfg.batch, cfg.d_inner, cfg.d_state, device=dev)

        def fn():
            run_selective_call(g, torch, abi, yb, ls)
        times, nl = time_device(fn, flush, 5, 3, torch, counter=abi.launch_count)
        ms = statistics.mean(times)
        nbytes = selective_bytes(cfg)
        gbs = nbytes / (ms * 1e-3) / 1e9
        row = {"ms_per_call": round(ms, 4), "channel_steps_per_s": cfg.channel_steps / (ms * 1e-3),
               "hbm_gbs": round(gbs, 1), "hbm_frac": round(gbs / hbm_peak, 4),
               "launches_per_call": nl / 5, "seqlen": cfg.seqlen,
               "note": "algorithmic bytes of the scan only; the padded copies move about as "
                       "many again"}
        del g, yb, ls
        torch.cuda.empty_cache()
    except Exception as ex:
        row = {"error": str(ex)[:200]}
    return {name: row}


def wide_state_rows(dev, torch, abi, inputs, hbm_peak, flush, mufu_peak):
    """d_state 32, 64 and 128 at the Mamba-130M layer shape (bf16, gate on)."""
    rows = {}
    cfg = inputs.WORKLOADS["mamba130m_layer"]
    for N in (32, 64, 128):
        name = f"mamba130m_layer_N{N}"
        try:
            with inputs.on_device(dev):
                g = inputs.selective_inputs(cfg.batch, cfg.d_inner, N, cfg.seqlen, cfg.dtype)
            yb = torch.empty_like(g["u"])
            ls = torch.empty(cfg.batch, cfg.d_inner, N, device=dev)

            def fn():
                run_selective_call(g, torch, abi, yb, ls)
            times, nl = time_device(fn, flush, 3, 2, torch, counter=abi.launch_count)
            ms = statistics.mean(times)
            mufu = cfg.channel_steps * (N + 5) / (ms * 1e-3)
            rows[name] = {"ms_per_call": round(ms, 4),
                          "channel_steps_per_s": cfg.channel_steps / (ms * 1e-3),
                          "state_steps_per_s": cfg.channel_steps * N / (ms * 1e-3),
                          "mufu_frac": round(mufu / mufu_peak, 4) if mufu_peak else None,
                          "launches_per_call": nl / 3}
            del g, yb, ls
            torch.cuda.empty_cache()
        except Exception as ex:
            rows[name] = {"error": str(ex)[:200]}
    return rows


def grouped_rows(dev, torch, abi, inputs, hbm_peak, flush):
    """B, C per channel (G = d_inner) and per group of 64 channels at the
    Mamba-130M layer shape."""
    rows = {}
    cfg = inputs.WORKLOADS["mamba130m_layer"]
    for name, G in (("per_channel_bc_mamba130m_layer", cfg.d_inner),
                    ("groups24_bc_mamba130m_layer", cfg.d_inner // 64)):
        try:
            with inputs.on_device(dev):
                g = inputs.selective_inputs(cfg.batch, cfg.d_inner, cfg.d_state, cfg.seqlen,
                                            cfg.dtype, groups=G)
            yb = torch.empty_like(g["u"])
            ls = torch.empty(cfg.batch, cfg.d_inner, cfg.d_state, device=dev)

            def fn():
                run_selective_call(g, torch, abi, yb, ls)
            times, nl = time_device(fn, flush, 5, 3, torch, counter=abi.launch_count)
            ms = statistics.mean(times)
            e = 2
            nbytes = (cfg.channel_steps * 4 * e + cfg.batch * G * cfg.d_state * cfg.seqlen * 2 * e
                      + cfg.batch * cfg.d_inner * cfg.d_state * 4)
            gbs = nbytes / (ms * 1e-3) / 1e9
            rows[name] = {"ms_per_call": round(ms, 4),
                          "channel_steps_per_s": cfg.channel_steps / (ms * 1e-3),
                          "hbm_gbs": round(gbs, 1), "hbm_frac": round(gbs / hbm_peak, 4),
                          "launches_per_call": nl / 5, "algorithmic_bytes": nbytes,
                          "groups": G}
            del g, yb, ls
            torch.cuda.empty_cache()
        except Exception as ex:
            rows[name] = {"error": str(ex)[:200]}
    return rows


def backward_bytes(cfg):
    """Algorithmic bytes of one backward call: u, delta, z, dout read and du,
    ddelta, dz written once per channel-step; B, C read and dB, dC (f32)
    written once per (batch, state, step); A, D, bias and their gradients."""
    e = 2 if cfg.dtype == "bf16" else 4
    per_ch = (4 + 3) * e
    bnl = cfg.batch * cfg.d_state * cfg.seqlen
    return (cfg.channel_steps * per_ch + bnl * 2 * (e + 4)
            + cfg.d_inner * (cfg.d_state + 2) * 8)


def backward_rows(dev, torch, abi, inputs, hbm_peak, flush):
    """The selective scan's backward at the Mamba-130M layer shape."""
    rows = {}
    try:
        cfg = inputs.WORKLOADS["mamba130m_layer"]
        with inputs.on_device(dev):
            g = inputs.workload_selective_inputs(cfg)
            dout = inputs.grad_output((cfg.batch, cfg.d_inner, cfg.seqlen), cfg.dtype)

        def fn():
            abi.selective_scan_bwd(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"],
                                   g["delta_bias"], dout)
        times, nl = time_device(fn, flush, 5, 3, torch, counter=abi.launch_count)
        ms = statistics.mean(times)
        nbytes = backward_bytes(cfg)
        rows["bwd_mamba130m_layer"] = {
            "ms_per_call": round(ms, 4), "channel_steps_per_s": cfg.channel_steps / (ms * 1e-3),
            "hbm_gbs": round(nbytes / (ms * 1e-3) / 1e9, 1),
            "hbm_frac": round(nbytes / (ms * 1e-3) / 1e9 / hbm_peak, 4),
            "launches_per_call": nl / 5, "algorithmic_bytes": nbytes,
            "traffic": measured_traffic("scan_bwd_fast<bf16>"),
            "note": "all eight gradients, two launches (scan_bwd_fast + scan_bwd_finish); "
                    "stored states and partial sums in stream-ordered scratch"}
        del g, dout
        torch.cuda.empty_cache()
    except Exception as e:
        rows["bwd_mamba130m_layer"] = {"error": str(e)[:200]}
    try:
        # a training step's scan: forward then backward, plain and with the
        # forward's states kept for the backward
        cfg = inputs.WORKLOADS["mamba130m_layer"]
        with inputs.on_device(dev):
            g = inputs.workload_selective_inputs(cfg)
            dout = inputs.grad_output((cfg.batch, cfg.d_inner, cfg.seqlen), cfg.dtype)
        args = [g[k] for k in ("u", "delta", "A", "B", "C", "D", "z", "delta_bias")]
        yb = torch.empty_like(g["u"])
        ls = torch.empty(cfg.batch, cfg.d_inner, cfg.d_state, device=dev)
        ck = torch.empty(cfg.batch, cfg.d_inner, (cfg.seqlen + 7) // 8, 16, device=dev)

        def plain():
            abi.selective_scan_fwd(*args, y=yb, last_state=ls)
            abi.selective_scan_bwd(*args, dout)

        def kept():
            abi.selective_scan_fwd_ckpt(*args, y=yb, last_state=ls, ckpt=ck)
            abi.selective_scan_bwd_ckpt(*args, dout, ck)
        ms_plain = statistics.mean(time_device(plain, flush, 5, 3, torch))
        times, nl = time_device(kept, flush, 5, 3, torch, counter=abi.launch_count)
        ms = statistics.mean(times)
        rows["train_step_mamba130m_layer"] = {
            "ms_per_call": round(ms, 4), "channel_steps_per_s": cfg.channel_steps / (ms * 1e-3),
            "ms_plain_fwd_then_bwd": round(ms_plain, 4), "launches_per_call": nl / 5,
            "checkpoint_bytes": ck.numel() * 4,
            "note": "ss_selective_scan_fwd_ckpt then ss_selective_scan_bwd_ckpt (the backward "
                    "reads the forward's state every 8 steps); ms_plain_fwd_then_bwd is "
                    "ss_selective_scan_fwd then ss_selective_scan_bwd"}
        del g, dout, ck
        torch.cuda.empty_cache()
    except Exception as e:
        rows["train_step_mamba130m_layer"] = {"error": str(e)[:200]}
    return rows


def time_decode(step, steps, torch):
    """Microseconds per token, (eager, CUDA-graph replay).  Eager calls from
    Python are bound by the host-side marshalling; the graph holds `steps`
    launches captured on a side stream and shows the device time per step."""
    for _ in range(10):
        step()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record()
    for _ in range(steps):
        step()
    b.record()
    torch.cuda.synchronize()
    us_eager = a.elapsed_time(b) * 1e3 / steps
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # any one-time setup happens outside the capture
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=side):
            for _ in range(steps):
                step()
    torch.cuda.current_stream().wait_stream(side)
    graph.replay()
    torch.cuda.synchronize()
    reps = 5
    a.record()
    for _ in range(reps):
        graph.replay()
    b.record()
    torch.cuda.synchronize()
    return us_eager, a.elapsed_time(b) * 1e3 / (steps * reps)


def decode_row(us_eager, us, nbytes, hbm_peak):
    return {"us_per_token": round(us, 3), "us_per_token_eager": round(us_eager, 3),
            "state_bytes": nbytes, "hbm_gbs": round(nbytes / (us * 1e-6) / 1e9, 1),
            "hbm_frac": round(nbytes / (us * 1e-6) / 1e9 / hbm_peak, 4),
            "note": "one launch per token; us_per_token from a CUDA graph of 200 steps "
                    "(device time), us_per_token_eager from Python calls (host-bound)"}


def decode_rows(dev, torch, abi, inputs, hbm_peak):
    """One-token decode steps (the recurrent form): time per step and the
    state bytes read + written per step against HBM."""
    rows = {}
    steps = 200
    try:
        cfg = inputs.WORKLOADS["mamba130m_layer"]
        with inputs.on_device(dev):
            g = inputs.selective_inputs(cfg.batch, cfg.d_inner, cfg.d_state, 1, "bf16")
        state = torch.zeros(cfg.batch, cfg.d_inner, cfg.d_state, device=dev)
        u, dl, z = (g[k][..., 0].contiguous() for k in ("u", "delta", "z"))
        Bt, Ct = g["B"][..., 0].contiguous(), g["C"][..., 0].contiguous()
        y = torch.empty_like(u)

        def step():
            abi.selective_state_update(state, u, dl, g["A"], Bt, Ct, g["D"], z, g["delta_bias"],
                                       y=y)
        us_eager, us = time_decode(step, steps, torch)
        nbytes = 2 * state.numel() * 4
        rows["decode_step_mamba130m_layer"] = decode_row(us_eager, us, nbytes, hbm_peak)
    except Exception as e:
        rows["decode_step_mamba130m_layer"] = {"error": str(e)[:200]}
    try:
        cfg = inputs.WORKLOADS["mamba2_ssd"]
        with inputs.on_device(dev):
            g = inputs.ssd_inputs(cfg.batch, 1, cfg.nheads, cfg.headdim, cfg.d_state, cfg.ngroups)
        state = torch.zeros(cfg.batch, cfg.nheads, cfg.headdim, cfg.d_state, device=dev)
        x, dt = g["x"][:, 0].contiguous(), g["dt"][:, 0].contiguous()
        Bt, Ct = g["B"][:, 0].contiguous(), g["C"][:, 0].contiguous()
        y = torch.empty_like(x)

        def step2():
            abi.ssd_state_update(state, x, dt, g["A_head"], Bt, Ct, g["D"], y=y)
        us_eager, us = time_decode(step2, steps, torch)
        nbytes = 2 * state.numel() * 4
        rows["decode_step_mamba2_ssd"] = decode_row(us_eager, us, nbytes, hbm_peak)
    except Exception as e:
        rows["decode_step_mamba2_ssd"] = {"error": str(e)[:200]}
    return rows


# ---------------------------------------------------------------------------
# CPU oracle timing.


def oracle_throughput(host, cfg, seconds, oracle, threads=None):
    """Time the fp64 oracle on a bounded sample of the workload: whole
    channels (full length) in blocks, until `seconds` have passed."""
    import numpy as np
    nth = threads or oracle.max_threads()
    Dch = cfg.d_inner
    block = min(Dch, max(nth * 32, 64))
    f64 = {k: (None if v is None else v.double().numpy()) for k, v in host.items()}
    done, t_used, rounds = 0, 0.0, 0
    b = 0
    while t_used < seconds and rounds < 100000:
        d0 = (rounds * block) % Dch
        d1 = min(Dch, d0 + block)
        sub = dict(u=f64["u"][b:b + 1, d0:d1], delta=f64["delta"][b:b + 1, d0:d1],
                   z=None if f64["z"] is None else f64["z"][b:b + 1, d0:d1],
                   A=f64["A"][d0:d1], B=f64["B"][b:b + 1], C=f64["C"][b:b + 1],
                   D=None if f64["D"] is None else f64["D"][d0:d1],
                   delta_bias=None if f64["delta_bias"] is None else f64["delta_bias"][d0:d1])
        sub = {k: (None if v is None else np.ascontiguousarray(v)) for k, v in sub.items()}
        t0 = time.perf_counter()
        oracle.selective_scan(sub["u"], sub["delta"], sub["A"], sub["B"], sub["C"], sub["D"],
                              sub["z"], sub["delta_bias"], softplus=True, nthreads=nth)
        t_used += time.perf_counter() - t0
        done += (d1 - d0) * cfg.seqlen
        rounds += 1
        b = (b + 1) % cfg.batch
    return done / t_used, nth, done, t_used


def oracle_ssd_throughput(host, cfg, seconds, oracle, threads=None):
    """The SSD oracle on a bounded sample: whole heads (full length, all
    headdim channels) of one batch row at a time, until `seconds` have
    passed.  Channel-steps count H*P channels."""
    import numpy as np
    nth = threads or oracle.max_threads()
    H, G = cfg.nheads, cfg.ngroups
    block = min(H, max(nth, 1))
    f64 = {k: (None if v is None else v.double().numpy()) for k, v in host.items()}
    done, t_used, rounds, b = 0, 0.0, 0, 0
    while t_used < seconds and rounds < 100000:
        h0 = (rounds * block) % H
        h1 = min(H, h0 + block)
        g0, g1 = h0 // (H // G), (h1 - 1) // (H // G) + 1
        if g1 - g0 > 1:  # keep one group per block so the sub-call's head -> group map holds
            h1 = (g0 + 1) * (H // G)
            g1 = g0 + 1
        sub = dict(x=f64["x"][b:b + 1, :, h0:h1], dt=f64["dt"][b:b + 1, :, h0:h1],
                   A_head=f64["A_head"][h0:h1], B=f64["B"][b:b + 1, :, g0:g1],
                   C=f64["C"][b:b + 1, :, g0:g1],
                   D=None if f64["D"] is None else f64["D"][h0:h1])
        sub = {k: (None if v is None else np.ascontiguousarray(v)) for k, v in sub.items()}
        t0 = time.perf_counter()
        oracle.ssd(sub["x"], sub["dt"], sub["A_head"], sub["B"], sub["C"], sub["D"],
                   nthreads=nth)
        t_used += time.perf_counter() - t0
        done += (h1 - h0) * cfg.headdim * cfg.seqlen
        rounds += 1
        b = (b + 1) % cfg.batch
    return done / t_used, nth, done, t_used


def cpu_baseline(name, host, cfg, seconds, oracle):
    """The oracle as it stands, timed on the host cores on a bounded sample of
    the workload (whole channels or heads, full length)."""
    ssd = name == "mamba2_ssd"
    fn = oracle_ssd_throughput if ssd else oracle_throughput
    v, nth, done, used = fn(host, cfg, seconds, oracle)
    what = "whole heads (all headdim channels)" if ssd else "whole channels"
    return {"value": v, "unit": UNIT, "cores": nth, "kind": "oracle",
            "sample": f"{done} channel-steps ({what} of the workload, full length "
                      f"{cfg.seqlen}) in {used:.1f} s on {cpu_model()}"}


def cpu_model():
    try:
        for ln in open("/proc/cpuinfo"):
            if ln.startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


def config_dict(cfg):
    """The workload as the JSON line names it (the same in both arms)."""
    d = {"workload": f"{cfg.name}: {WORKLOAD_TEXT[cfg.name]}", "batch": cfg.batch}
    if cfg.name == "mamba2_ssd":
        d.update(seq_len=cfg.seqlen, nheads=cfg.nheads, headdim=cfg.headdim,
                 d_state=cfg.d_state, ngroups=cfg.ngroups, chunk=cfg.chunk)
    else:
        d.update(d_inner=cfg.d_inner, d_state=cfg.d_state, seq_len=cfg.seqlen,
                 z_gate=cfg.gate)
    d.update(io_dtype=cfg.dtype, state_dtype="f32", parallelism="replica per GPU",
             l2="flushed (256 MB write) before every timed step, outside the step's events")
    return d


# ---------------------------------------------------------------------------


def main_reference(args):
    from selective_state_space_146_b300 import dist as dh
    rank, _, world = dh.env_world()
    if rank != 0:
        return 0
    import oracle
    from selective_state_space_146_b300 import inputs
    cfg = inputs.WORKLOADS[HEADLINE]
    host = inputs.workload_selective_inputs(cfg)
    per_step = max(0.5, min(3.0, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_throughput(host, cfg, per_step, oracle)
    vals = []
    for _ in range(args.steps):
        v, nth, done, used = oracle_throughput(host, cfg, per_step, oracle)
        vals.append((v, done, used))
    value = sum(d for _, d, _ in vals) / sum(u for _, _, u in vals)
    ms = 1e3 * statistics.mean(u for _, _, u in vals)
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_dict(cfg), "impl": "reference",
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": nth, "kind": "oracle",
                             "sample": f"per step, whole channels of the workload (full length "
                                       f"{cfg.seqlen}) for ~{per_step:.1f} s on {cpu_model()}"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main_profile(args):
    """Run one workload's call `warmup + steps` times (inputs drawn on the GPU)."""
    import torch

    from selective_state_space_146_b300 import _abi as abi
    from selective_state_space_146_b300 import inputs
    dev = torch.device("cuda", 0)
    if args.profile == "bwd_mamba130m_layer":
        cfg = inputs.WORKLOADS["mamba130m_layer"]
        with inputs.on_device(dev):
            g = inputs.workload_selective_inputs(cfg)
            dout = inputs.grad_output((cfg.batch, cfg.d_inner, cfg.seqlen), cfg.dtype)
        for _ in range(args.warmup + args.steps):
            abi.selective_scan_bwd(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"],
                                   g["delta_bias"], dout)
        torch.cuda.synchronize()
        return 0 if abi.device_error() == 0 else 1
    layer = inputs.WORKLOADS["mamba130m_layer"]
    runs = args.warmup + args.steps
    if args.profile == "conv_mamba130m_layer":  # causal conv (width 4) + SiLU + scan
        with inputs.on_device(dev):
            g = inputs.workload_selective_inputs(layer)
        gen = torch.Generator(device=dev).manual_seed(7)
        cw = torch.randn(layer.d_inner, 4, generator=gen, device=dev) * 0.5
        cb = torch.randn(layer.d_inner, generator=gen, device=dev) * 0.1
        for _ in range(runs):
            abi.conv_selective_scan_fwd(g["u"], cw, cb, g["delta"], g["A"], g["B"], g["C"],
                                        g["D"], g["z"], g["delta_bias"], return_last_state=True)
        torch.cuda.synchronize()
        return 0 if abi.device_error() == 0 else 1
    if args.profile in ("per_channel_bc_mamba130m_layer", "mamba130m_layer_N64"):
        N = 64 if args.profile.endswith("N64") else layer.d_state
        G = layer.d_inner if args.profile.startswith("per_channel") else None
        with inputs.on_device(dev):
            g = inputs.selective_inputs(layer.batch, layer.d_inner, N, layer.seqlen, layer.dtype,
                                        groups=G)
        for _ in range(runs):
            abi.selective_scan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"],
                                   g["delta_bias"], return_last_state=True)
        torch.cuda.synchronize()
        return 0 if abi.device_error() == 0 else 1
    if args.profile == "decode_mamba2_ssd":  # one-token SSD state update, 4 x 64 heads x 64, N 128
        cfg = inputs.WORKLOADS["mamba2_ssd"]
        with inputs.on_device(dev):
            g = inputs.ssd_inputs(cfg.batch, 1, cfg.nheads, cfg.headdim, cfg.d_state, cfg.ngroups)
        state = torch.zeros(cfg.batch, cfg.nheads, cfg.headdim, cfg.d_state, device=dev)
        x, dt = g["x"][:, 0].contiguous(), g["dt"][:, 0].contiguous()
        Bt, Ct = g["B"][:, 0].contiguous(), g["C"][:, 0].contiguous()
        for _ in range(runs):
            abi.ssd_state_update(state, x, dt, g["A_head"], Bt, Ct, g["D"])
        torch.cuda.synchronize()
        return 0 if abi.device_error() == 0 else 1
    if ":" in args.profile:  # a benchmark workload with another sequence length
        import dataclasses
        name, _, length = args.profile.partition(":")
        cfg = dataclasses.replace(inputs.WORKLOADS[name], seqlen=int(length))
    else:
        cfg = inputs.WORKLOADS[args.profile]
    with inputs.on_device(dev):
        g = (inputs.workload_ssd_inputs(cfg) if cfg.name == "mamba2_ssd"
             else inputs.workload_selective_inputs(cfg))
    for _ in range(args.warmup + args.steps):
        if cfg.name == "mamba2_ssd":
            abi.ssd_chunk_scan_fwd(g["x"], g["dt"], g["A_head"], g["B"], g["C"], g["D"],
                                   chunk=cfg.chunk, return_last_state=True)
        else:
            abi.selective_scan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"],
                                   g["delta_bias"], return_last_state=True)
    torch.cuda.synchronize()
    return 0 if abi.device_error() == 0 else 1


def keep_pool_memory(dev_index, nbytes=1 << 30):
    """Let the device's default memory pool (the library's stream-ordered
    scratch) keep up to `nbytes` between calls instead of returning it at
    every synchronisation (the CUDA default threshold is 0).  Process-local;
    a caller that calls the library repeatedly would do the same."""
    try:
        from cuda.bindings import driver as drv
        from cuda.bindings import runtime as rt
        err, pool = rt.cudaDeviceGetDefaultMemPool(dev_index)
        if int(err) != 0:
            return False
        (err,) = rt.cudaMemPoolSetAttribute(
            pool, rt.cudaMemPoolAttr.cudaMemPoolAttrReleaseThreshold, drv.cuuint64_t(nbytes))
        return int(err) == 0
    except Exception:
        return False


def selective_kernel(cfg):
    """Name of the kernel the library runs for a d_state-16 workload in the
    TMA layout (the library's rule, with 3 x 148 resident CTA slots: two lanes
    per channel where its 64-channel tiles fill 60% of the slots, four lanes
    where its 32-channel tiles do, else the sequence is cut into segments and
    one lane per channel runs from 512 tiles of 64 steps, two from 32)."""
    ch, slots = cfg.batch * cfg.d_inner, 3 * N_SM
    tiles64 = -(-cfg.seqlen // 64)
    if (ch // 64) * 10 >= slots * 6:
        lanes = 2
    elif (ch // 32) * 10 >= slots * 6:
        lanes = 4
    else:
        lanes = 1 if tiles64 >= 512 and ch > 64 else 2 if tiles64 >= 32 and ch > 32 else 4
    return f"scan_seq<{cfg.dtype}, {lanes} lane{'s' if lanes > 1 else ''}/channel>"


def workload_record(name, m, pk, args, cpu=None):
    """The fields of one measured workload (the headline's layout)."""
    cfg, ms, ms_max = m["cfg"], m["ms"], m["ms_max"]
    sec = ms * 1e-3
    if name == "mamba2_ssd":
        nbytes, flops = ssd_bytes(cfg), ssd_flops(cfg)
        tf = flops / sec / 1e12
        gbs = nbytes / sec / 1e9
        roof = {"bound": "tensor", "achieved": round(tf, 1), "peak": pk["tf_burst"],
                "unit": "TFLOP/s", "frac": round(tf / pk["tf_burst"], 4),
                "traffic": measured_traffic("ssd_chunk_tc2"), "kernel": "ssd_chunk_tc2",
                "algorithmic_flops_per_launch": flops,
                "peak_source": f"{pk['src']} bf16_tflops (burst: the kernel is timed alone)",
                "frac_of_sustained": round(tf / pk["tf_sust"], 4),
                "hbm_achieved_gbs": round(gbs, 1), "hbm_frac": round(gbs / pk["hbm"], 4),
                "algorithmic_bytes_per_launch": nbytes}
    else:
        nbytes = selective_bytes(cfg)
        gbs = nbytes / sec / 1e9
        key = selective_kernel(cfg)
        roof = {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm"], "unit": "GB/s",
                "frac": round(gbs / pk["hbm"], 4), "traffic": measured_traffic(key),
                "kernel": key, "algorithmic_bytes_per_launch": nbytes,
                "peak_source": f"{pk['src']} hbm_gbs",
                "frac_of_nominal": round(gbs / NOMINAL_HBM_GBS, 4),
                "nominal_gbs": NOMINAL_HBM_GBS}
        if pk["mufu"]:
            ops = mufu_ops_per_channel_step(cfg)
            rate = cfg.channel_steps * ops / sec
            roof["mufu"] = {
                "achieved": round(rate / 1e9, 1), "peak": round(pk["mufu"] / 1e9, 1),
                "unit": "Gop/s (ex2-equivalents)", "frac": round(rate / pk["mufu"], 4),
                "ops_per_channel_step": ops,
                "peak_source": f"ss_probe_ex2_rate in this run: {pk['ex2_rate']:.2f} ex2 per SM "
                               f"per clock x {N_SM} SMs x {pk['sm_mhz']:.0f} MHz",
                "note": "the method's exponentials per channel-step; segment summaries "
                        "(long sequences over few channels) repeat them and are not counted"}
    return {
        "value": m["total_units"] / (ms_max * 1e-3), "unit": UNIT, "ms_per_step": ms_max,
        "steps": args.steps, "warmup": args.warmup, "dtype": cfg.dtype,
        "config": config_dict(cfg), "roofline": roof, "cpu_baseline": cpu,
        "e2e": {"value": m["total_units"] / (m["e2e_ms"] * 1e-3), "unit": UNIT,
                "h2d_bytes_per_step": m["h2d"], "d2h_bytes_per_step": m["d2h"],
                "ms_per_step": m["e2e_ms"], "call": m["e2e_call"]},
        "gpu_launches": m["launches"],
        "step_ms": {"median": statistics.median(m["times"]), "min": min(m["times"]),
                    "max": max(m["times"])},
    }


def main_ours(args):
    import torch
    import torch.distributed as tdist

    from selective_state_space_146_b300 import _abi as abi
    from selective_state_space_146_b300 import dist as dh
    from selective_state_space_146_b300 import inputs

    rank, local_rank, world = dh.env_world()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    if world > 1 and not tdist.is_initialized():
        tdist.init_process_group("nccl", device_id=dev)
    abi.load()
    pool_kept = keep_pool_memory(local_rank)
    hbm_peak, tf_peak, tf_sust, peak_src = peaks()
    try:
        ex2_rate = abi.probe_ex2_rate()
    except Exception:
        ex2_rate = None
    sm_mhz = SM_MHZ_MAX
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            sm_mhz = float(json.load(f).get("sm_max_mhz", SM_MHZ_MAX))
    except Exception:
        pass
    pk = {"hbm": hbm_peak, "tf_burst": tf_peak, "tf_sust": tf_sust, "src": peak_src,
          "ex2_rate": ex2_rate, "sm_mhz": sm_mhz,
          "mufu": ex2_rate * N_SM * sm_mhz * 1e6 if ex2_rate else None}
    if args.probe_scan_forms:
        if rank == 0:
            seq, shfl = abi.probe_scan_forms()
            print(json.dumps({"seq_channel_steps_per_s": seq, "shfl_channel_steps_per_s": shfl,
                              "seq_over_shfl": seq / shfl}))
        return 0
    if args.probe_mufu:
        if rank == 0:
            print(json.dumps({"ex2_per_sm_per_clock": ex2_rate, "sms": N_SM, "sm_mhz": sm_mhz,
                              "ex2_gop_s": pk["mufu"] / 1e9 if pk["mufu"] else None}))
        return 0

    h = measure_workload(HEADLINE, args, dev, rank, torch, abi, inputs, dh, clocks=True)
    import oracle
    cpu = None
    if rank == 0 and not args.no_cpu:
        cpu = cpu_baseline(HEADLINE, h["host"], h["cfg"], args.cpu_seconds, oracle)
    head = workload_record(HEADLINE, h, pk, args, cpu)
    del h["host"]

    rows = None
    if not args.no_rows:
        rows = {}
        for name in FULL_ROWS:
            try:
                m = measure_workload(name, args, dev, rank, torch, abi, inputs, dh)
                c = None
                if rank == 0 and not args.no_cpu:
                    c = cpu_baseline(name, m["host"], m["cfg"], max(2.0, args.cpu_seconds / 2),
                                     oracle)
                rows[name] = workload_record(name, m, pk, args, c)
                del m
            except Exception as e:  # a row failing must not hide the headline
                rows[name] = {"error": str(e)[:200]}
        if rank == 0:
            rows.update(secondary_rows(dev, torch, abi, inputs, hbm_peak, tf_sust, pk["mufu"]))
    if world > 1:
        dh.barrier(dev)
    if rank == 0:
        line = {
            "metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": head["dtype"], "data": "synthetic", "config": head["config"],
            "roofline": head["roofline"], "cpu_baseline": head["cpu_baseline"],
            "e2e": head["e2e"], "gpu_launches": head["gpu_launches"], "clocks": h["clocks"],
            "step_ms": head["step_ms"],
            "scratch_pool": "default pool keeps up to 1 GiB" if pool_kept
                            else "default pool at CUDA defaults",
            "rows": rows,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        tdist.destroy_process_group()
    return 0


if __name__ == "__main__":
    a = parse()
    if a.profile:
        sys.exit(main_profile(a))
    sys.exit(main_reference(a) if a.impl == "reference" else main_ours(a))
