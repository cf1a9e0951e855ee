"""ss_selective_scan_fwd_host and ss_ssd_chunk_scan_fwd_host: host tensors
in, host tensors out, the batch cut into chunks that overlap on two streams
(rows, or blocks of one row's channels or heads when a row holds more than 32
MB).  Compared with the fp64 oracle on the same inputs (GPU)."""
import pytest
import torch

import oracle
from selective_state_space_146_b300 import _abi, inputs
from tests.parity_util import check_close, oracle_ssd_units, to_np

pytestmark = pytest.mark.gpu


def _tdt(dt):
    return torch.float32 if dt == "f32" else torch.bfloat16


def _pin(d):
    return {k: (None if v is None else v.pin_memory()) for k, v in d.items()}


# (odd lengths: each chunk goes to the device as it is and is scanned on padded copies)
@pytest.mark.parametrize("case", [(2, 64, 16, 512, "bf16", None), (5, 40, 16, 300, "f32", None),
                                  (3, 48, 16, 200, "bf16", 48), (4, 24, 8, 77, "f32", None),
                                  (1, 32, 16, 64, "bf16", None), (2, 64, 16, 511, "bf16", None),
                                  (3, 48, 16, 201, "bf16", 48), (2, 40, 16, 301, "f32", None)],
                         ids=lambda c: "x".join(map(str, c)))
def test_host_api_matches_oracle(cuda_device, case):
    Bsz, D, N, L, dt, G = case
    inp = inputs.selective_inputs(Bsz, D, N, L, dt, groups=G, seed=Bsz * 100 + L)
    h = _pin(inp)
    y, s = _abi.selective_scan_fwd_host(h["u"], h["delta"], h["A"], h["B"], h["C"], h["D"],
                                        h["z"], h["delta_bias"], return_last_state=True)
    torch.cuda.synchronize()
    assert y.device.type == "cpu" and s.device.type == "cpu"
    yo, so = oracle.selective_scan(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                                   inp["z"], inp["delta_bias"], nthreads=8)
    check_close(to_np(y), yo, _tdt(dt), "y")
    check_close(to_np(s), so, _tdt(dt), "last_state")


def test_host_api_pageable_memory_and_no_state(cuda_device):
    inp = inputs.selective_inputs(3, 32, 16, 128, "f32", seed=4)
    y = torch.empty(3, 32, 128)
    _abi.selective_scan_fwd_host(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                                 inp["z"], inp["delta_bias"], y=y)
    torch.cuda.synchronize()
    yo, _ = oracle.selective_scan(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                                  inp["z"], inp["delta_bias"])
    check_close(to_np(y), yo, torch.float32, "y (pageable host memory)")


def test_host_api_zero_length_writes_zero_state(cuda_device):
    inp = _pin(inputs.selective_inputs(2, 8, 16, 0, "f32", seed=1))
    last = torch.full((2, 8, 16), 3.0).pin_memory()
    _abi.selective_scan_fwd_host(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                                 inp["z"], inp["delta_bias"], y=torch.empty(2, 8, 0),
                                 last_state=last)
    torch.cuda.synchronize()
    assert bool((last == 0).all())


def test_host_api_layer_shape_sampled(cuda_device):
    """The end-to-end call of the benchmark (Mamba-130M layer, 8 x 1536 x 2048
    bf16): sampled channels against the oracle."""
    cfg = inputs.WORKLOADS["mamba130m_layer"]
    inp = inputs.workload_selective_inputs(cfg, seed=0)
    h = _pin(inp)
    y, s = _abi.selective_scan_fwd_host(h["u"], h["delta"], h["A"], h["B"], h["C"], h["D"],
                                        h["z"], h["delta_bias"], return_last_state=True)
    torch.cuda.synchronize()
    from tests.parity_util import oracle_selective_channels
    total = cfg.batch * cfg.d_inner
    chans = inputs.sample_units(total, 24, seed=3)
    yo, so = oracle_selective_channels(inp, chans)
    idx = torch.as_tensor(chans)
    check_close(to_np(y.reshape(total, cfg.seqlen)[idx]), yo, torch.bfloat16, "y (sampled)")
    check_close(to_np(s.reshape(total, cfg.d_state)[idx]), so, torch.bfloat16, "state (sampled)")


@pytest.mark.parametrize("case", [(1, 600, 16384, "bf16", None, True),
                                  (1, 512, 20000, "bf16", 4, True),
                                  (1, 96, 50000, "f32", None, False),
                                  (1, 600, 16383, "bf16", None, True)],
                         ids=lambda c: "x".join(map(str, c[:5])))
def test_host_api_channel_blocks(cuda_device, case):
    """Rows of more than 32 MB of inputs: the call cuts each row into blocks of
    channels (whole groups when B, C are grouped; a ragged last block), the
    row's B, C copied once per buffer set.  Sampled channels against the
    oracle."""
    from tests.parity_util import oracle_selective_channels
    Bsz, D, L, dt, G, gate = case
    inp = inputs.selective_inputs(Bsz, D, 16, L, dt, groups=G, gate=gate, seed=L)
    h = _pin(inp)
    y, s = _abi.selective_scan_fwd_host(h["u"], h["delta"], h["A"], h["B"], h["C"], h["D"],
                                        h["z"], h["delta_bias"], return_last_state=True)
    torch.cuda.synchronize()
    total = Bsz * D
    chans = inputs.sample_units(total, 10, seed=L)
    if G:
        sel = [int(c) for c in chans]
        ys, ss = [], []
        for c in sel:  # one channel with its group's B, C
            b, d = divmod(c, D)
            g = d // (D // G)
            sub = {"u": inp["u"][b:b + 1, d:d + 1], "delta": inp["delta"][b:b + 1, d:d + 1],
                   "z": None if inp["z"] is None else inp["z"][b:b + 1, d:d + 1],
                   "A": inp["A"][d:d + 1], "B": inp["B"][b:b + 1, g], "C": inp["C"][b:b + 1, g],
                   "D": inp["D"][d:d + 1], "delta_bias": inp["delta_bias"][d:d + 1]}
            yo1, so1 = oracle.selective_scan(sub["u"], sub["delta"], sub["A"], sub["B"], sub["C"],
                                             sub["D"], sub["z"], sub["delta_bias"])
            ys.append(yo1[0, 0])
            ss.append(so1[0, 0])
        import numpy as np
        yo, so = np.stack(ys), np.stack(ss)
    else:
        yo, so = oracle_selective_channels(inp, chans)
    idx = torch.as_tensor([int(c) for c in chans])
    check_close(to_np(y.reshape(total, L)[idx]), yo, _tdt(dt), "y (sampled)")
    check_close(to_np(s.reshape(total, 16)[idx]), so, _tdt(dt), "state (sampled)")


# ss_ssd_chunk_scan_fwd_host: (batch, L, heads, headdim, N, groups, dtype);
# the first three are small (whole batch rows per chunk), the others hold more
# than 32 MB of x per row, so a row is cut into blocks of heads: half of one
# group (G 1), whole groups (G 4), and an fp32 row on the CUDA-core kernel.
SSD_HOST_CASES = [
    (2, 256, 8, 64, 128, 1, "bf16"),
    (3, 130, 4, 16, 32, 2, "f32"),
    (1, 1, 2, 8, 16, 1, "f32"),
    (1, 8192, 64, 64, 128, 1, "bf16"),
    (2, 8192, 64, 64, 128, 4, "bf16"),
    (1, 4100, 32, 64, 16, 1, "f32"),
]


@pytest.mark.parametrize("case", SSD_HOST_CASES, ids=lambda c: "x".join(map(str, c)))
def test_ssd_host_api_matches_oracle(cuda_device, case):
    Bsz, L, H, P, N, G, dt = case
    inp = inputs.ssd_inputs(Bsz, L, H, P, N, G, dt, seed=L + H)
    h = _pin(inp)
    y, s = _abi.ssd_chunk_scan_fwd_host(h["x"], h["dt"], h["A_head"], h["B"], h["C"], h["D"],
                                        return_last_state=True)
    torch.cuda.synchronize()
    assert y.device.type == "cpu" and s.device.type == "cpu"
    assert _abi.device_error() == 0
    if Bsz * L * H <= 1 << 16:
        yo, so = oracle.ssd(inp["x"], inp["dt"], inp["A_head"], inp["B"], inp["C"], inp["D"],
                            nthreads=8)
        check_close(to_np(y), yo, _tdt(dt), "y")
        check_close(to_np(s), so, _tdt(dt), "last_state")
    else:
        # sampled heads, one from every head block and batch row at least
        units = sorted(set(int(u) for u in inputs.sample_units(Bsz * H, 6, seed=L)) | {0, H // 2, Bsz * H - 1})
        yo, so = oracle_ssd_units(inp, units)
        yg = torch.stack([y[u // H, :, u % H] for u in units])
        sg = torch.stack([s[u // H, u % H] for u in units])
        check_close(to_np(yg), yo, _tdt(dt), "y (sampled heads)")
        check_close(to_np(sg), so, _tdt(dt), "last_state (sampled heads)")
        # the device call on the same inputs gives the same bits
        dev = cuda_device
        yd, sd = _abi.ssd_chunk_scan_fwd(*[(None if inp[k] is None else inp[k].to(dev))
                                           for k in ("x", "dt", "A_head", "B", "C", "D")],
                                         return_last_state=True)
        torch.cuda.synchronize()
        if dt == "bf16":  # the tensor-core kernels: per head pair, whatever the blocking
            assert torch.equal(yd.cpu(), y) and torch.equal(sd.cpu(), s)


def test_ssd_host_api_rejects_strided(cuda_device):
    inp = inputs.ssd_inputs(1, 64, 4, 16, 16, 1, "f32", seed=3)
    x = inp["x"].transpose(1, 2).contiguous().transpose(1, 2)  # same shape, not contiguous
    with pytest.raises(_abi.SSError, match="UNSUPPORTED"):
        _abi.ssd_chunk_scan_fwd_host(x, inp["dt"], inp["A_head"], inp["B"], inp["C"], inp["D"])
