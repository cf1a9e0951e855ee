"""The fused causal conv1d + SiLU + selective scan against the fp64 oracle
(GPU, C ABI).  The oracle composes its conv and scan functions."""

import numpy as np
import pytest
import torch

import oracle
from selective_state_space_146_b300 import _abi, inputs
from tests.parity_util import check_close, cuda_inputs, scan_switches, to_np

pytestmark = pytest.mark.gpu


def _conv_params(D, W, seed, bias=True):
    g = torch.Generator().manual_seed(seed)
    w = torch.randn(D, W, generator=g, dtype=torch.float32) * 0.5
    b = torch.randn(D, generator=g, dtype=torch.float32) * 0.1 if bias else None
    return w, b


CASES = [
    # Bsz, D, N, L, dtype, W, bias
    (2, 40, 16, 200, "bf16", 4, True),
    (2, 40, 16, 200, "f32", 4, True),
    (1, 32, 16, 4096, "bf16", 4, True),   # few channels: segments, halo across segment starts
    (1, 16, 16, 1000, "f32", 3, False),   # segments with a ragged tail
    (3, 64, 16, 136, "bf16", 2, True),
    (1, 5, 16, 7, "f32", 4, True),        # general kernel (t rows not 16-byte multiples)
    (1, 4, 64, 50, "f32", 1, True),       # N = 64: general kernel
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
@pytest.mark.parametrize("path", [None, "general", "split1", "split2", "split4", "seq1", "seq3",
                                  "seq4", "seq1s5", "seq3s3"])
def test_conv_scan_small(cuda_device, case, path):
    with _abi.debug_paths(**scan_switches(path)):
        _conv_scan_small(cuda_device, case)


def _conv_scan_small(cuda_device, case):
    Bsz, D, N, L, dt, W, bias = case
    inp = inputs.selective_inputs(Bsz, D, N, L, dt, seed=L + W)
    w, cb = _conv_params(D, W, L, bias)
    g = cuda_inputs(inp, cuda_device)
    y, s = _abi.conv_selective_scan_fwd(g["u"], w.to(cuda_device),
                                        None if cb is None else cb.to(cuda_device), g["delta"],
                                        g["A"], g["B"], g["C"], g["D"], g["z"], g["delta_bias"],
                                        return_last_state=True)
    torch.cuda.synchronize()
    assert _abi.device_error() == 0
    yo, so = oracle.conv_selective_scan(inp["u"], w, cb, inp["delta"], inp["A"], inp["B"],
                                        inp["C"], inp["D"], inp["z"], inp["delta_bias"], nthreads=8)
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    check_close(to_np(y), yo, tdt, "conv-scan y")
    check_close(to_np(s), so, tdt, "conv-scan last_state")


def test_conv_scan_full_size_sampled(cuda_device):
    """The Mamba-130M layer shape with the conv in front, sampled channels."""
    cfg = inputs.WORKLOADS["mamba130m_layer"]
    inp = inputs.workload_selective_inputs(cfg)
    w, cb = _conv_params(cfg.d_inner, 4, 7)
    g = cuda_inputs(inp, cuda_device)
    y, s = _abi.conv_selective_scan_fwd(g["u"], w.to(cuda_device), cb.to(cuda_device), g["delta"],
                                        g["A"], g["B"], g["C"], g["D"], g["z"], g["delta_bias"],
                                        return_last_state=True)
    torch.cuda.synchronize()
    total = cfg.batch * cfg.d_inner
    chans = inputs.sample_units(total, 16, seed=3)
    ys, ss = [], []
    for c in chans:
        b, d = divmod(int(c), cfg.d_inner)
        yo, so = oracle.conv_selective_scan(
            inp["u"][b:b + 1, d:d + 1], w[d:d + 1], cb[d:d + 1], inp["delta"][b:b + 1, d:d + 1],
            inp["A"][d:d + 1], inp["B"][b:b + 1], inp["C"][b:b + 1], inp["D"][d:d + 1],
            inp["z"][b:b + 1, d:d + 1], inp["delta_bias"][d:d + 1])
        ys.append(yo[0, 0])
        ss.append(so[0, 0])
    idx = torch.as_tensor(chans, device=y.device)
    check_close(to_np(y.reshape(total, -1)[idx]), np.stack(ys), torch.bfloat16, "conv-scan y")
    check_close(to_np(s.reshape(total, -1)[idx]), np.stack(ss), torch.bfloat16, "conv-scan state")


def test_conv_scan_layer_shape_sampled(cuda_device):
    """The fused call the benchmark times (8 x 1536 x 2048 bf16, width 4),
    sampled channels against the oracle run on those channels alone."""
    cfg = inputs.WORKLOADS["mamba130m_layer"]
    inp = inputs.workload_selective_inputs(cfg, seed=0)
    w, b = _conv_params(cfg.d_inner, 4, seed=7)
    g = {k: (None if v is None else v.to(cuda_device)) for k, v in inp.items()}
    y, s = _abi.conv_selective_scan_fwd(g["u"], w.to(cuda_device), b.to(cuda_device), g["delta"],
                                        g["A"], g["B"], g["C"], g["D"], g["z"], g["delta_bias"],
                                        return_last_state=True)
    torch.cuda.synchronize()
    chans = inputs.sample_units(cfg.batch * cfg.d_inner, 16, seed=5)
    ys, ss, yo, so = [], [], [], []
    for c in chans:
        bb, d = divmod(int(c), cfg.d_inner)
        y1, s1 = oracle.conv_selective_scan(
            inp["u"][bb:bb + 1, d:d + 1], w[d:d + 1], b[d:d + 1], inp["delta"][bb:bb + 1, d:d + 1],
            inp["A"][d:d + 1], inp["B"][bb:bb + 1], inp["C"][bb:bb + 1], inp["D"][d:d + 1],
            inp["z"][bb:bb + 1, d:d + 1], inp["delta_bias"][d:d + 1])
        yo.append(y1[0, 0]); so.append(s1[0, 0])
        ys.append(to_np(y[bb, d])); ss.append(to_np(s[bb, d]))
    check_close(np.stack(ys), np.stack(yo), torch.bfloat16, "conv y (sampled channels)")
    check_close(np.stack(ss), np.stack(so), torch.bfloat16, "conv state (sampled channels)")
