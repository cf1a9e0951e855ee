"""The JSON line `bench.py` prints: every key a reader of the benchmark relies
on, with values of the right kind.  The CPU test runs the reference arm (the
fp64 oracle timed on the host) for one short step; the GPU test runs the
library's arm on the headline workload (long context) with the other
workloads and the CPU baseline left out."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _line(args, timeout):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, cwd=ROOT,
                         capture_output=True, text=True, timeout=timeout)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    return json.loads(lines[0])


def _common(d, steps, warmup):
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "e2e"):
        assert k in d, k
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["unit"] == "channel-steps/s" and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == steps and d["warmup"] == warmup
    assert d["scaling"] == "weak" and d["data"] == "synthetic"
    assert d["vs_baseline"] is None
    assert "workload" in d["config"]
    for k in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"):
        assert k in d["e2e"], k


def test_reference_arm_line():
    import bench
    from selective_state_space_146_b300 import inputs
    d = _line(["--impl", "reference", "--steps", "1", "--warmup", "1"], timeout=600)
    _common(d, 1, 1)
    # the same workload description as the library's arm prints
    assert d["config"] == json.loads(json.dumps(bench.config_dict(inputs.WORKLOADS[bench.HEADLINE])))
    assert d["impl"] == "reference" and d["dtype"] == "f64"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"]
    assert cb["value"] == d["value"]
    assert d["e2e"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


@pytest.mark.gpu
def test_library_arm_line(cuda_device):
    d = _line(["--steps", "3", "--warmup", "3", "--no-rows", "--no-cpu"], timeout=900)
    _common(d, 3, 3)
    assert "impl" not in d or d["impl"] != "reference"
    r = d["roofline"]
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in r, k
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and 0 < r["frac"] < 1.5
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3
    assert d["dtype"] == "bf16" and d["config"]["workload"].startswith("long_context")
    m = r["mufu"]  # the exponential rate against the probe measured in the same run
    assert 0 < m["frac"] < 1.5 and abs(m["frac"] - m["achieved"] / m["peak"]) < 1e-3
    assert d["e2e"]["h2d_bytes_per_step"] > 0 and d["e2e"]["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] > 0
    c = d["clocks"]
    for k in ("sm_mhz", "sm_max_mhz", "reasons"):
        assert k in c, k
    assert set(d["step_ms"]) >= {"median", "min", "max"}


def test_reference_arm_under_torchrun_prints_once():
    """Launched as the multi-GPU runs are (one process per rank), rank 0
    alone times the oracle and prints the line; the other rank exits 0."""
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "1"]
    out = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
