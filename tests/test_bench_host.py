"""Host-side arithmetic of `bench.py` (CPU): the algorithmic bytes and flops
the roofline divides, the parsing of the clock samples, and the comment
stripping that decides whether a stored DRAM-traffic count still describes
the kernel's sources."""
import dataclasses

import pytest

import bench
from selective_state_space_146_b300 import inputs


def _nbytes(d):
    return sum(v.numel() * v.element_size() for v in d.values() if v is not None)


@pytest.mark.parametrize("flags", [dict(), dict(gate=False), dict(skip=False, bias=False),
                                   dict(last_state=False), dict(dtype="f32")])
def test_selective_bytes_equal_the_tensors_of_one_call(flags):
    """Every input read once, y written once, the f32 final state written
    once: the sizes of the tensors the generator makes for the same shape."""
    cfg = dataclasses.replace(inputs.WORKLOADS["mamba130m_layer"], batch=2, d_inner=24,
                              seqlen=40, **flags)
    inp = inputs.workload_selective_inputs(cfg)
    y = inp["u"].numel() * inp["u"].element_size()
    state = 4 * cfg.batch * cfg.d_inner * cfg.d_state if cfg.last_state else 0
    assert bench.selective_bytes(cfg) == _nbytes(inp) + y + state


def test_headline_bytes_and_channel_steps():
    """8 x 1536 x 2048 bf16 with z, D, delta_bias and the final state: 8 bytes
    per channel-step (u, delta, z in, y out) plus B, C, parameters and state,
    203.3 MB per call."""
    cfg = inputs.WORKLOADS["mamba130m_layer"]
    assert cfg.channel_steps == 25_165_824
    per_step = 8 * cfg.channel_steps
    bc = 2 * 8 * 16 * 2048 * 2
    params = 1536 * 18 * 4
    state = 8 * 1536 * 16 * 4
    assert bench.selective_bytes(cfg) == per_step + bc + params + state
    assert round(bench.selective_bytes(cfg) / 1e6, 1) == 203.3


@pytest.mark.parametrize("skip", [True, False])
def test_ssd_bytes_equal_the_tensors_of_one_call(skip):
    cfg = dataclasses.replace(inputs.WORKLOADS["mamba2_ssd"], batch=2, seqlen=48, nheads=4,
                              headdim=8, d_state=16, ngroups=2, chunk=16, skip=skip)
    inp = inputs.workload_ssd_inputs(cfg)
    y = inp["x"].numel() * inp["x"].element_size()
    state = 4 * cfg.batch * cfg.nheads * cfg.headdim * cfg.d_state
    assert bench.ssd_bytes(cfg) == _nbytes(inp) + y + state


def test_ssd_flops_are_the_four_contractions():
    """Per chunk of Q steps: C B^T (Q x Q, inner N) once per group; per head
    the diagonal block M X (Q x Q times Q x P), the chunk state (P x Q times
    Q x N) and the inter-chunk output (Q x N times N x P); 2 flops per
    multiply-add.  At batch 4, L 8192, 64 heads of 64, N 128, Q 256: 2.15 +
    68.7 + 34.4 + 34.4 = 139.6 GFLOP."""
    cfg = inputs.WORKLOADS["mamba2_ssd"]
    chunks = cfg.batch * (cfg.seqlen // cfg.chunk)
    Q, P, N, H, G = cfg.chunk, cfg.headdim, cfg.d_state, cfg.nheads, cfg.ngroups
    cb = chunks * G * 2 * Q * Q * N
    diag = chunks * H * 2 * Q * Q * P
    states = chunks * H * 2 * P * Q * N
    off = chunks * H * 2 * Q * N * P
    assert bench.ssd_flops(cfg) == cb + diag + states + off
    assert [round(v / 1e9, 2) for v in (cb, diag, states, off)] == [2.15, 68.72, 34.36, 34.36]
    # a ragged last chunk counts as a whole one (the kernel computes it so)
    short = dataclasses.replace(cfg, seqlen=cfg.seqlen - 1)
    assert bench.ssd_flops(short) == bench.ssd_flops(cfg)


def test_clock_summary_reads_samples_and_reasons():
    s = bench.ClockSampler(0)
    s.lines = [
        "0, 1965, 2032, 870.5, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2032, 910.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2032, 2032, 640.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbled line",
        "0, [N/A], 2032, 1.0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    out = s.summary()
    assert out["samples"] == 3
    assert out["sm_mhz"] == 1980 and out["sm_max_mhz"] == 2032
    assert out["reasons"] == ["sw_power_cap"]
    assert out["power_w_max"] == 910.0
    s.lines.append("0, 1500, 2032, 700, 0x40, Not Active, Active, Not Active, Not Active")
    assert s.summary()["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]


def test_clock_summary_without_samples():
    s = bench.ClockSampler(0)
    assert s.summary() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}


def test_code_only_ignores_comments_but_not_code():
    src = 'int a = 1; // one\n/* block\n comment */\nconst char* s = "// kept";\n\n  int b;  \n'
    base = bench._code_only(src)
    assert base == 'int a = 1;\nconst char* s = "// kept";\n  int b;'
    assert bench._code_only(src.replace("// one", "// changed comment")) == base
    assert bench._code_only(src.replace("/* block", "/* another")) == base
    assert bench._code_only(src.replace("int a = 1", "int a = 2")) != base
    assert bench._code_only('x = "a\\"//b";') == 'x = "a\\"//b";'


def test_stored_traffic_is_keyed_to_measured_kernels():
    """Each stored DRAM count names a kernel whose source files exist, and is
    reported only while its recorded hash matches those sources."""
    import json
    import os
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        stored = json.load(f)
    assert set(stored) <= set(bench.KERNEL_SOURCES)
    for key, e in stored.items():
        assert e["bytes_per_launch"] > 0 and len(e["source_hash"]) == 16
        assert e["sources"] == bench.KERNEL_SOURCES[key]
        assert e["bytes_per_launch"] == e["dram_bytes_read"] + e["dram_bytes_write"]
        want = e["bytes_per_launch"] if e["source_hash"] == bench.source_hash(
            bench.KERNEL_SOURCES[key]) else None
        assert bench.measured_traffic(key) == want
    assert bench.measured_traffic("no such kernel") is None
