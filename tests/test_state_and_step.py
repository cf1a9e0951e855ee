"""Initial states and the recurrent decode step, against the fp64 oracle (GPU).

The oracle already takes an initial state h0 (its split-invariance pin fixes
what continuing from a state means); the decode step is one iteration of the
oracle's time loop, so L steps in turn must reproduce the oracle's scan.
"""

import numpy as np
import pytest
import torch

import oracle
from selective_state_space_146_b300 import _abi, inputs
from tests.parity_util import SSD_SWITCHES, check_close, cuda_inputs, scan_switches, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture
def scan_path(request):
    val = getattr(request, "param", None)
    with _abi.debug_paths(**scan_switches(val)):
        yield val


def _tdt(dt):
    return torch.float32 if dt == "f32" else torch.bfloat16


def _h0(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g, dtype=torch.float32)


@pytest.mark.parametrize("case", [(2, 40, 16, 200, "bf16"), (1, 16, 16, 1000, "f32"),
                                  (1, 32, 16, 4096, "bf16"), (2, 6, 16, 33, "f32"),
                                  (1, 4, 64, 50, "f32")],
                         ids=lambda c: "x".join(map(str, c)))
@pytest.mark.parametrize("scan_path", [None, "general", "split1", "split4"], indirect=True)
def test_selective_scan_with_initial_state(cuda_device, scan_path, case):
    Bsz, D, N, L, dt = case
    inp = inputs.selective_inputs(Bsz, D, N, L, dt, seed=L + 3)
    h0 = _h0((Bsz, D, N), 11)
    g = cuda_inputs(inp, cuda_device)
    y, s = _abi.selective_scan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"],
                                   g["delta_bias"], return_last_state=True,
                                   initial_state=h0.to(cuda_device))
    torch.cuda.synchronize()
    yo, so = oracle.selective_scan(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                                   inp["z"], inp["delta_bias"], h0=h0, nthreads=8)
    check_close(to_np(y), yo, _tdt(dt), "y with initial state")
    check_close(to_np(s), so, _tdt(dt), "last_state with initial state")


def test_selective_scan_continues_across_calls(cuda_device):
    """[0, L1) then [L1, L) from the first call's final state == one call."""
    inp = inputs.selective_inputs(2, 48, 16, 1536, "bf16", seed=21)
    g = cuda_inputs(inp, cuda_device)
    y, s = _abi.selective_scan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"],
                                   g["delta_bias"], return_last_state=True)
    L1 = 1024

    def part(sl, h0=None):
        return _abi.selective_scan_fwd(g["u"][..., sl].contiguous(), g["delta"][..., sl].contiguous(),
                                       g["A"], g["B"][..., sl].contiguous(),
                                       g["C"][..., sl].contiguous(), g["D"],
                                       g["z"][..., sl].contiguous(), g["delta_bias"],
                                       return_last_state=True, initial_state=h0)

    y1, s1 = part(slice(0, L1))
    y2, s2 = part(slice(L1, None), s1)
    torch.cuda.synchronize()
    check_close(to_np(torch.cat([y1, y2], -1)), to_np(y), torch.bfloat16, "y split vs whole")
    check_close(to_np(s2), to_np(s), torch.bfloat16, "state split vs whole")


@pytest.mark.parametrize("case", [(2, 24, 16, 12, "f32"), (3, 40, 16, 10, "bf16"),
                                  (1, 8, 64, 6, "f32")], ids=lambda c: "x".join(map(str, c)))
def test_decode_steps_reproduce_the_scan(cuda_device, case):
    Bsz, D, N, L, dt = case
    inp = inputs.selective_inputs(Bsz, D, N, L, dt, seed=L * 7 + D)
    g = cuda_inputs(inp, cuda_device)
    h0 = _h0((Bsz, D, N), 5)
    state = h0.to(cuda_device).clone()
    ys = []
    for t in range(L):
        ys.append(_abi.selective_state_update(
            state, g["u"][..., t].contiguous(), g["delta"][..., t].contiguous(), g["A"],
            g["B"][..., t].contiguous(), g["C"][..., t].contiguous(), g["D"],
            g["z"][..., t].contiguous(), g["delta_bias"]))
    torch.cuda.synchronize()
    yo, so = oracle.selective_scan(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                                   inp["z"], inp["delta_bias"], h0=h0)
    check_close(to_np(torch.stack(ys, -1)), yo, _tdt(dt), "decode y")
    check_close(to_np(state), so, _tdt(dt), "decode state")


@pytest.mark.parametrize("case", [(1, 384, 4, 64, 128, 1, "bf16"), (2, 300, 4, 16, 32, 2, "f32"),
                                  (1, 1000, 8, 64, 128, 2, "bf16")],
                         ids=lambda c: "x".join(map(str, c)))
@pytest.mark.parametrize("ssd_path", [None, "general"])
def test_ssd_with_initial_state(cuda_device, case, ssd_path):
    with _abi.debug_paths(**SSD_SWITCHES[ssd_path]):
        _ssd_with_initial_state(cuda_device, case)


def _ssd_with_initial_state(cuda_device, case):
    Bsz, L, H, P, N, G, dt = case
    inp = inputs.ssd_inputs(Bsz, L, H, P, N, G, dt, seed=L + 1)
    h0 = _h0((Bsz, H, P, N), 13)
    g = cuda_inputs(inp, cuda_device)
    y, s = _abi.ssd_chunk_scan_fwd(g["x"], g["dt"], g["A_head"], g["B"], g["C"], g["D"],
                                   chunk=128, return_last_state=True,
                                   initial_state=h0.to(cuda_device))
    torch.cuda.synchronize()
    yo, so = oracle.ssd(inp["x"], inp["dt"], inp["A_head"], inp["B"], inp["C"], inp["D"], h0=h0,
                        nthreads=8)
    check_close(to_np(y), yo, _tdt(dt), "ssd y with initial state")
    check_close(to_np(s), so, _tdt(dt), "ssd state with initial state")


@pytest.mark.parametrize("case", [(2, 10, 4, 16, 32, 2, "f32"), (1, 8, 8, 64, 128, 1, "bf16")],
                         ids=lambda c: "x".join(map(str, c)))
def test_ssd_decode_steps_reproduce_the_scan(cuda_device, case):
    Bsz, L, H, P, N, G, dt = case
    inp = inputs.ssd_inputs(Bsz, L, H, P, N, G, dt, seed=L + H)
    g = cuda_inputs(inp, cuda_device)
    h0 = _h0((Bsz, H, P, N), 17)
    state = h0.to(cuda_device).clone()
    ys = []
    for t in range(L):
        ys.append(_abi.ssd_state_update(state, g["x"][:, t].contiguous(), g["dt"][:, t].contiguous(),
                                        g["A_head"], g["B"][:, t].contiguous(),
                                        g["C"][:, t].contiguous(), g["D"]))
    torch.cuda.synchronize()
    yo, so = oracle.ssd(inp["x"], inp["dt"], inp["A_head"], inp["B"], inp["C"], inp["D"], h0=h0)
    check_close(to_np(torch.stack(ys, 1)), yo, _tdt(dt), "ssd decode y")
    check_close(to_np(state), so, _tdt(dt), "ssd decode state")


@pytest.mark.parametrize("case", [(3, 3, 6, 5, 128, 3, "f32", False),
                                  (2, 2, 4, 7, 128, 2, "bf16", True),
                                  (1, 4, 3, 3, 128, 1, "bf16", False),
                                  (2, 3, 2, 64, 128, 2, "f32", True)],
                         ids=lambda c: "x".join(map(str, c[:7])) + ("-strided" if c[7] else ""))
def test_ssd_decode_n128_rows_cross_heads(cuda_device, case):
    """The N = 128 step takes several (b, h, p) rows per warp: head dims
    that are not a multiple of that count make one warp cross heads, groups
    and batch rows, and B, C with a state stride above one take the
    element-wise loads."""
    Bsz, L, H, P, N, G, dt, strided = case
    inp = inputs.ssd_inputs(Bsz, L, H, P, N, G, dt, seed=3 * L + P)
    g = cuda_inputs(inp, cuda_device)
    h0 = _h0((Bsz, H, P, N), 19)
    state = h0.to(cuda_device).clone()

    def bc(t):
        return t.transpose(-1, -2).contiguous().transpose(-1, -2) if strided else t.contiguous()
    ys = []
    for t in range(L):
        Bt, Ct = bc(g["B"][:, t]), bc(g["C"][:, t])
        assert (Bt.stride(-1) == 1) != strided
        ys.append(_abi.ssd_state_update(state, g["x"][:, t].contiguous(), g["dt"][:, t].contiguous(),
                                        g["A_head"], Bt, Ct, g["D"]))
    torch.cuda.synchronize()
    yo, so = oracle.ssd(inp["x"], inp["dt"], inp["A_head"], inp["B"], inp["C"], inp["D"], h0=h0)
    check_close(to_np(torch.stack(ys, 1)), yo, _tdt(dt), "ssd decode y")
    check_close(to_np(state), so, _tdt(dt), "ssd decode state")


def test_decode_steps_at_benchmark_shapes(cuda_device):
    """One decode step at the shapes the benchmark times: 8 x 1536 channels,
    N 16 (selective) and 4 x 64 heads x 64, N 128 (SSD), from a random state,
    against one step of the oracles."""
    Bsz, D, N = 8, 1536, 16
    inp = inputs.selective_inputs(Bsz, D, N, 1, "bf16", seed=8)
    h0 = _h0((Bsz, D, N), 9)
    state = h0.to(cuda_device).clone()
    g = cuda_inputs(inp, cuda_device)
    y = _abi.selective_state_update(state, g["u"][..., 0].contiguous(),
                                    g["delta"][..., 0].contiguous(), g["A"],
                                    g["B"][..., 0].contiguous(), g["C"][..., 0].contiguous(),
                                    g["D"], g["z"][..., 0].contiguous(), g["delta_bias"])
    torch.cuda.synchronize()
    yo, so = oracle.selective_scan(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                                   inp["z"], inp["delta_bias"], h0=h0, nthreads=8)
    check_close(to_np(y), yo[..., 0], torch.bfloat16, "selective decode y")
    check_close(to_np(state), so, torch.bfloat16, "selective decode state")

    Bsz, H, P, N = 4, 64, 64, 128
    inp = inputs.ssd_inputs(Bsz, 1, H, P, N, 1, "bf16", seed=10)
    h0 = _h0((Bsz, H, P, N), 11)
    state = h0.to(cuda_device).clone()
    g = cuda_inputs(inp, cuda_device)
    y = _abi.ssd_state_update(state, g["x"][:, 0].contiguous(), g["dt"][:, 0].contiguous(),
                              g["A_head"], g["B"][:, 0].contiguous(), g["C"][:, 0].contiguous(),
                              g["D"])
    torch.cuda.synchronize()
    yo, so = oracle.ssd(inp["x"], inp["dt"], inp["A_head"], inp["B"], inp["C"], inp["D"], h0=h0,
                        nthreads=8)
    check_close(to_np(y), yo[:, 0], torch.bfloat16, "ssd decode y")
    check_close(to_np(state), so, torch.bfloat16, "ssd decode state")
