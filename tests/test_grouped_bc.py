"""B and C per channel group (one per channel when G = D) on the GPU against
the fp64 oracle.

The oracle's grouped form is pinned by brute force (test_oracle_pins.py).
Cases reach the three kernels: groups of >= 64 channels run the shared-B, C
TMA kernel with a group coordinate, smaller groups the per-channel streaming
kernel, and odd layouts or N != 16 the general kernel.
"""
import numpy as np
import pytest
import torch

import oracle
from selective_state_space_146_b300 import _abi, inputs
from tests.parity_util import check_close, cuda_inputs, scan_switches, to_np

pytestmark = pytest.mark.gpu


def _tdt(dt):
    return torch.float32 if dt == "f32" else torch.bfloat16


@pytest.fixture
def scan_path(request):
    """None: the library's choice; "general": the any-stride kernel; "rows":
    per-channel B, C read row by row instead of through TMA tiles; "splitK" /
    "seqK": scan_fast or scan_seq forced (groups that fit their channel tiles)."""
    val = getattr(request, "param", None)
    sw = dict(grouped_path=0) if val == "rows" else scan_switches(val)
    with _abi.debug_paths(**sw):
        yield val


CASES = [
    # Bsz, D, G, N, L, dtype, gate/skip/bias
    (2, 128, 2, 16, 296, "bf16", True),    # groups of 64: TMA kernel with group rows
    (1, 192, 3, 16, 200, "f32", True),
    (1, 64, 64, 16, 500, "f32", True),     # one B, C per channel: streaming kernel
    (2, 48, 48, 16, 1000, "bf16", True),
    (2, 20, 20, 16, 136, "bf16", True),     # per channel, partial 8-channel tile
    (1, 24, 24, 16, 100, "f32", False),
    (2, 40, 8, 16, 72, "bf16", False),     # groups of 5 channels, no gate / skip / bias
    (2, 40, 20, 16, 200, "bf16", True),    # groups of 2 channels: TMA kernel, 4 group rows a tile
    (1, 36, 9, 16, 96, "f32", True),       # groups of 4, partial last tile
    (2, 96, 3, 16, 128, "bf16", True),     # groups of 32: shared-B, C kernel with group rows
    (2, 24, 4, 16, 77, "f32", True),       # odd length: general kernel
    (1, 16, 16, 8, 64, "f32", True),       # N = 8: general kernel
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:6])) +
                         ("" if c[6] else "-nogate"))
@pytest.mark.parametrize("scan_path", [None, "general", "rows", "seq3", "seq4"], indirect=True)
def test_grouped_bc_matches_oracle(cuda_device, scan_path, case):
    Bsz, D, G, N, L, dt, on = case
    inp = inputs.selective_inputs(Bsz, D, N, L, dt, gate=on, skip=on, bias=on, groups=G,
                                  seed=D + L)
    g = cuda_inputs(inp, cuda_device)
    y, s = _abi.selective_scan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"],
                                   g["delta_bias"], return_last_state=True)
    torch.cuda.synchronize()
    assert _abi.device_error() == 0
    yo, so = oracle.selective_scan(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                                   inp["z"], inp["delta_bias"], nthreads=8)
    check_close(to_np(y), yo, _tdt(dt), "y")
    check_close(to_np(s), so, _tdt(dt), "last_state")


@pytest.mark.parametrize("G", [1, 64])
def test_grouped_bc_with_initial_state(cuda_device, G):
    Bsz, D, N, L = 2, 64, 16, 256
    inp = inputs.selective_inputs(Bsz, D, N, L, "bf16", groups=G, seed=3)
    h0 = torch.randn(Bsz, D, N, generator=torch.Generator().manual_seed(4))
    g = cuda_inputs(inp, cuda_device)
    y, s = _abi.selective_scan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"],
                                   g["delta_bias"], return_last_state=True,
                                   initial_state=h0.to(cuda_device))
    torch.cuda.synchronize()
    yo, so = oracle.selective_scan(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                                   inp["z"], inp["delta_bias"], h0=h0, nthreads=8)
    check_close(to_np(y), yo, torch.bfloat16, "y")
    check_close(to_np(s), so, torch.bfloat16, "last_state")


def test_one_group_equals_shared(cuda_device):
    """(Bsz, 1, N, L) and (Bsz, N, L) describe the same scan: same bits."""
    inp = inputs.selective_inputs(2, 64, 16, 512, "bf16", seed=5)
    g = cuda_inputs(inp, cuda_device)
    y1 = _abi.selective_scan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"],
                                 g["delta_bias"])
    y2 = _abi.selective_scan_fwd(g["u"], g["delta"], g["A"], g["B"][:, None], g["C"][:, None],
                                 g["D"], g["z"], g["delta_bias"])
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)


def test_grouped_bc_rejects_bad_groups(cuda_device):
    inp = inputs.selective_inputs(1, 12, 16, 16, "f32", groups=5, seed=6)
    g = cuda_inputs(inp, cuda_device)
    with pytest.raises(_abi.SSError, match="SHAPE"):
        _abi.selective_scan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"],
                                g["delta_bias"])


@pytest.mark.parametrize("scan_path", [None, "rows"], indirect=True)
def test_per_channel_bc_layer_shape_sampled(cuda_device, scan_path):
    """One B, C per channel at the Mamba-130M layer's d_inner and length
    (batch 2; bf16): sampled channels against the oracle run channel by
    channel on its own B, C rows."""
    Bsz, D, N, L = 2, 1536, 16, 2048
    inp = inputs.selective_inputs(Bsz, D, N, L, "bf16", groups=D, seed=0)
    g = cuda_inputs(inp, cuda_device)
    y, s = _abi.selective_scan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"],
                                   g["delta_bias"], return_last_state=True)
    torch.cuda.synchronize()
    y, s = to_np(y), to_np(s)
    chans = inputs.sample_units(Bsz * D, 48, seed=1)
    for c in chans:
        b, d = divmod(int(c), D)
        yo, so = oracle.selective_scan(
            inp["u"][b:b + 1, d:d + 1], inp["delta"][b:b + 1, d:d + 1], inp["A"][d:d + 1],
            inp["B"][b:b + 1, d], inp["C"][b:b + 1, d], inp["D"][d:d + 1],
            inp["z"][b:b + 1, d:d + 1], inp["delta_bias"][d:d + 1])
        check_close(y[b, d], yo[0, 0], torch.bfloat16, f"y channel {c}")
        check_close(s[b, d], so[0, 0], torch.bfloat16, f"state channel {c}")


def test_groups_of_64_layer_shape_sampled(cuda_device):
    """B, C per group of 64 channels at the Mamba-130M layer shape (the
    benchmark's groups24 row, TMA kernel with group rows): sampled channels."""
    cfg = inputs.WORKLOADS["mamba130m_layer"]
    G = cfg.d_inner // 64
    inp = inputs.selective_inputs(cfg.batch, cfg.d_inner, cfg.d_state, cfg.seqlen, "bf16",
                                  groups=G, seed=2)
    g = cuda_inputs(inp, cuda_device)
    y, s = _abi.selective_scan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"],
                                   g["delta_bias"], return_last_state=True)
    torch.cuda.synchronize()
    y, s = to_np(y), to_np(s)
    for c in inputs.sample_units(cfg.batch * cfg.d_inner, 24, seed=4):
        b, d = divmod(int(c), cfg.d_inner)
        gi = d // 64
        yo, so = oracle.selective_scan(
            inp["u"][b:b + 1, d:d + 1], inp["delta"][b:b + 1, d:d + 1], inp["A"][d:d + 1],
            inp["B"][b:b + 1, gi], inp["C"][b:b + 1, gi], inp["D"][d:d + 1],
            inp["z"][b:b + 1, d:d + 1], inp["delta_bias"][d:d + 1])
        check_close(y[b, d], yo[0, 0], torch.bfloat16, f"y channel {c}")
        check_close(s[b, d], so[0, 0], torch.bfloat16, f"state channel {c}")
