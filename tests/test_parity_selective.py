"""GPU parity of ss_selective_scan_fwd against the fp64 oracle.

Every call goes through the C ABI (libssscan.so) on cuda:0.  Small cases are
compared element by element over the whole output; the full-size workloads
(the same call the benchmark times) on sampled channels that the oracle
computes one by one.
"""
import numpy as np
import pytest
import torch

from selective_state_space_146_b300 import _abi, inputs
from tests.parity_util import (check_close, cuda_inputs, oracle_selective,
                               oracle_selective_channels, scan_switches, to_np)

pytestmark = pytest.mark.gpu


@pytest.fixture
def scan_path(request):
    val = getattr(request, "param", None)
    with _abi.debug_paths(**scan_switches(val)):
        yield val


# every selective-scan kernel for N = 16: the general one, scan_fast with each
# lane split, scan_seq with each launch shape (and forced time segments)
PATHS = [None, "general", "split1", "split2", "split4", "split8", "seq1", "seq2", "seq3", "seq4",
         "seq5", "seq6", "seq7", "seq1s5", "seq3s7", "seq7s5", "seq4s3"]


def _run(inp, dev, softplus=True, want_state=True):
    g = cuda_inputs(inp, dev)
    out = _abi.selective_scan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"],
                                  g["delta_bias"], softplus=softplus,
                                  return_last_state=want_state)
    torch.cuda.synchronize()
    assert _abi.device_error() == 0
    return out


@pytest.mark.parametrize("scan_path", PATHS, indirect=True)
def test_tiny_f32_workload(cuda_device, scan_path):
    cfg = inputs.WORKLOADS["tiny_f32"]
    inp = inputs.workload_selective_inputs(cfg)
    y, s = _run(inp, cuda_device)
    yo, so = oracle_selective(inp)
    check_close(to_np(y), yo, torch.float32, "y")
    check_close(to_np(s), so, torch.float32, "last_state")


CASES = [
    # Bsz, D, N, L, dtype, gate, skip, bias, softplus
    (2, 40, 16, 200, "bf16", True, True, True, True),     # ragged channel tile and t tail
    (2, 40, 16, 200, "f32", True, True, True, True),
    (1, 64, 16, 64, "bf16", False, False, False, False),  # everything optional off
    (3, 96, 16, 136, "f32", False, True, True, True),
    (1, 3, 16, 7, "f32", True, True, True, True),         # t rows not 16-byte multiples
    (1, 5, 16, 1, "bf16", True, True, True, True),        # L = 1
    (1, 8, 1, 33, "f32", True, True, True, True),         # N = 1
    (2, 4, 4, 64, "bf16", True, False, True, True),
    (1, 4, 64, 100, "f32", True, True, True, True),       # N = 64
    (1, 2, 256, 24, "f32", True, True, False, True),      # N = 256
    (1, 32, 16, 4096, "bf16", True, True, True, True),    # few channels: split into segments
    (1, 16, 16, 1000, "f32", True, True, True, True),     # segments with a ragged tail
    (1, 40, 16, 20000, "bf16", True, True, True, True),   # 39 segments, partial channel tile
    (1, 8, 16, 70000, "bf16", True, True, True, True),    # the 64-segment cap
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:5])))
@pytest.mark.parametrize("scan_path", PATHS, indirect=True)
def test_small_shapes(cuda_device, scan_path, case):
    Bsz, D, N, L, dt, gate, skip, bias, softplus = case
    inp = inputs.selective_inputs(Bsz, D, N, L, dt, gate=gate, skip=skip, bias=bias,
                                  seed=Bsz * 7 + D + L)
    if not bias and softplus is False:
        inp["delta"] = inp["delta"].abs()  # keep delta positive without softplus
    y, s = _run(inp, cuda_device, softplus=softplus)
    yo, so = oracle_selective(inp, softplus=softplus)
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    check_close(to_np(y), yo, tdt, "y")
    check_close(to_np(s), so, tdt if dt == "f32" else torch.bfloat16, "last_state")


def test_paths_agree_with_each_other(cuda_device):
    inp = inputs.selective_inputs(2, 48, 16, 520, "bf16", seed=3)
    outs = []
    for path in PATHS[1:]:
        with _abi.debug_paths(**scan_switches(path)):
            outs.append([to_np(t) for t in _run(inp, cuda_device)])
    for o in outs[1:]:
        check_close(o[0], outs[0][0], torch.bfloat16, "y fast vs general")
        check_close(o[1], outs[0][1], torch.bfloat16, "state fast vs general")


def test_strided_views(cuda_device):
    inp = inputs.selective_inputs(2, 24, 16, 256, "f32", seed=5)
    g = cuda_inputs(inp, cuda_device)
    # u read through a column slice of a wider buffer, B through a permuted copy
    wide = torch.zeros(2, 24, 512, device=cuda_device)
    wide[:, :, 128:384] = g["u"]
    u_view = wide[:, :, 128:384]
    Bt = g["B"].permute(0, 2, 1).contiguous().permute(0, 2, 1)  # stride in t = N
    y, s = _abi.selective_scan_fwd(u_view, g["delta"], g["A"], Bt, g["C"], g["D"], g["z"],
                                   g["delta_bias"], return_last_state=True)
    yo, so = oracle_selective(inp)
    check_close(to_np(y), yo, torch.float32, "y")
    check_close(to_np(s), so, torch.float32, "last_state")


def test_zero_length_gives_zero_state(cuda_device):
    inp = inputs.selective_inputs(2, 8, 16, 0, "bf16", seed=1)
    g = cuda_inputs(inp, cuda_device)
    last = torch.full((2, 8, 16), 7.0, device=cuda_device)
    _abi.selective_scan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"],
                            g["delta_bias"], last_state=last)
    torch.cuda.synchronize()
    assert bool((last == 0).all())


@pytest.mark.parametrize("name", ["mamba130m_layer", "mamba2p8b_layer", "long_context"])
def test_full_size_workloads_sampled(cuda_device, name, record_property):
    """The benchmark's call at full size (the library's own launch choice, as
    the benchmark times it); sampled channels against the oracle.  The
    relative L2 errors are recorded (junit properties) and printed."""
    cfg = inputs.WORKLOADS[name]
    inp = inputs.workload_selective_inputs(cfg)
    y, s = _run(inp, cuda_device)
    total = cfg.batch * cfg.d_inner
    chans = inputs.sample_units(total, 12 if cfg.seqlen > 100000 else 24, seed=1)
    yo, so = oracle_selective_channels(inp, chans)
    yg = to_np(y.reshape(total, cfg.seqlen)[torch.as_tensor(chans, device=y.device)])
    sg = to_np(s.reshape(total, cfg.d_state)[torch.as_tensor(chans, device=s.device)])
    ey = check_close(yg, yo, torch.bfloat16, f"{name} y (sampled channels)")
    es = check_close(sg, so, torch.bfloat16, f"{name} last_state (sampled channels)")
    record_property("rel_l2_y", float(ey))
    record_property("rel_l2_state", float(es))
    print(f"{name}: rel L2 y {ey:.3e}, last_state {es:.3e} (bar 3e-3)")
    assert bool(torch.isfinite(y).all())


@pytest.mark.parametrize("L", [1024, 4096, 16384])
def test_length_sweep_shapes_sampled(cuda_device, L):
    """The length-sweep shapes of the benchmark (batch 1, d_inner 2048, N 16,
    bf16): few channels, so the sequence is split into segments; sampled
    channels against the oracle."""
    inp = inputs.selective_inputs(1, 2048, 16, L, "bf16", seed=L)
    y, s = _run(inp, cuda_device)
    chans = inputs.sample_units(2048, 16, seed=L)
    yo, so = oracle_selective_channels(inp, chans)
    idx = torch.as_tensor(chans, device=y.device)
    check_close(to_np(y[0][idx]), yo, torch.bfloat16, f"L={L} y (sampled channels)")
    check_close(to_np(s[0][idx]), so, torch.bfloat16, f"L={L} last_state (sampled channels)")
