"""The selective scan with d_state 32, 64 and 128 (the wide-state kernel)
against the fp64 oracle, and sampled channels at the Mamba-130M layer shape."""
import numpy as np
import pytest
import torch

import oracle
from selective_state_space_146_b300 import _abi, inputs
from tests.parity_util import (check_close, cuda_inputs, oracle_selective_channels,
                               scan_switches, to_np)

pytestmark = pytest.mark.gpu


def _tdt(dt):
    return torch.float32 if dt == "f32" else torch.bfloat16


@pytest.fixture
def scan_path(request):
    val = getattr(request, "param", None)
    with _abi.debug_paths(**scan_switches(val)):
        yield val


CASES = [
    # Bsz, D, N, L, dtype, gate
    (2, 40, 32, 300, "bf16", True),
    (1, 64, 64, 256, "f32", True),
    (2, 20, 64, 100, "bf16", False),
    (1, 48, 128, 77, "f32", True),
    (2, 33, 128, 520, "bf16", True),
    (1, 3, 64, 1, "f32", True),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:5])))
@pytest.mark.parametrize("scan_path", [None, "general"], indirect=True)
def test_wide_state_matches_oracle(cuda_device, scan_path, case):
    Bsz, D, N, L, dt, gate = case
    inp = inputs.selective_inputs(Bsz, D, N, L, dt, gate=gate, seed=N + L)
    h0 = torch.randn(Bsz, D, N, generator=torch.Generator().manual_seed(L))
    g = cuda_inputs(inp, cuda_device)
    y, s = _abi.selective_scan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"],
                                   g["delta_bias"], return_last_state=True,
                                   initial_state=h0.to(cuda_device))
    torch.cuda.synchronize()
    assert _abi.device_error() == 0
    yo, so = oracle.selective_scan(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                                   inp["z"], inp["delta_bias"], h0=h0, nthreads=8)
    check_close(to_np(y), yo, _tdt(dt), "y")
    check_close(to_np(s), so, _tdt(dt), "last_state")


def test_wide_state_strided_activations(cuda_device):
    inp = inputs.selective_inputs(2, 24, 64, 150, "f32", seed=3)
    g = cuda_inputs(inp, cuda_device)
    tv = {k: g[k].transpose(1, 2).contiguous().transpose(1, 2) for k in ("u", "delta", "z")}
    y = _abi.selective_scan_fwd(tv["u"], tv["delta"], g["A"], g["B"], g["C"], g["D"], tv["z"],
                                g["delta_bias"])
    torch.cuda.synchronize()
    yo, _ = oracle.selective_scan(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                                  inp["z"], inp["delta_bias"], nthreads=8)
    check_close(to_np(y), yo, torch.float32, "y (strided views)")


@pytest.mark.parametrize("N", [64, 128])
def test_wide_state_layer_shape_sampled(cuda_device, N):
    """The benchmark's wide-state rows: 8 x 1536 x 2048 bf16 with d_state N."""
    inp = inputs.selective_inputs(8, 1536, N, 2048, "bf16", seed=N)
    g = cuda_inputs(inp, cuda_device)
    y, s = _abi.selective_scan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"],
                                   g["delta_bias"], return_last_state=True)
    torch.cuda.synchronize()
    total = 8 * 1536
    chans = inputs.sample_units(total, 12, seed=N)
    yo, so = oracle_selective_channels(inp, chans)
    idx = torch.as_tensor(chans, device=y.device)
    check_close(to_np(y.reshape(total, 2048)[idx]), yo, torch.bfloat16, "y (sampled channels)")
    check_close(to_np(s.reshape(total, N)[idx]), so, torch.bfloat16, "state (sampled channels)")
