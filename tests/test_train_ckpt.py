"""Forward with checkpoints and the backward that reads them (GPU, C ABI).

ss_selective_scan_fwd_ckpt must give the oracle's y and final state (and the
plain forward's, up to rounding: the two calls run different kernels) and write
the state before every 8th step; those states are checked against the fp64
oracle's final state on the matching prefix of the sequence.
ss_selective_scan_bwd_ckpt, given them, must give the plain backward's
gradients (checked against the fp64 oracle's backward, and bit for bit against
the plain backward where the forward ran the sequence in one piece).
"""
import numpy as np
import pytest
import torch

import oracle
from selective_state_space_146_b300 import _abi, inputs
from tests.parity_util import check_close, cuda_inputs, to_np

pytestmark = pytest.mark.gpu

GRADS = ("du", "ddelta", "dz", "dA", "dB", "dC", "dD", "ddelta_bias")


def _tdt(dt):
    return torch.float32 if dt == "f32" else torch.bfloat16


def _args(g):
    return [g[k] for k in ("u", "delta", "A", "B", "C", "D", "z", "delta_bias")]


CASES = [
    # Bsz, D, L, dtype, gate, skip, bias
    (2, 40, 200, "bf16", True, True, True),    # partial channel tile, ragged tail
    (1, 64, 76, "f32", True, True, True),      # fp32: 4-step chunks, every other one kept
    (2, 32, 8, "bf16", False, False, False),   # one sub-chunk, optional inputs off
    (1, 48, 1000, "bf16", True, True, True),   # few channels: the forward splits in segments
    (2, 40, 203, "bf16", True, True, True),    # odd length: both calls on padded copies
    (1, 64, 77, "f32", True, False, True),     # fp32 rows of 308 bytes: padded copies
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:4])))
def test_forward_checkpoints(cuda_device, case):
    Bsz, D, L, dt, gate, skip, bias = case
    inp = inputs.selective_inputs(Bsz, D, 16, L, dt, gate=gate, skip=skip, bias=bias, seed=L + D)
    g = cuda_inputs(inp, cuda_device)
    y, last, ck = _abi.selective_scan_fwd_ckpt(*_args(g))
    y0, last0 = _abi.selective_scan_fwd(*_args(g), return_last_state=True)
    torch.cuda.synchronize()
    assert _abi.device_error() == 0
    yo, so = oracle.selective_scan(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"],
                                   inp["D"], inp["z"], inp["delta_bias"], nthreads=8)
    check_close(to_np(y), yo, _tdt(dt), "checkpointing forward y")
    check_close(to_np(last), so, _tdt(dt), "checkpointing forward last_state")
    check_close(to_np(y), to_np(y0), _tdt(dt), "checkpointing forward y vs plain forward")
    check_close(to_np(last), to_np(last0), _tdt(dt), "checkpointing forward state vs plain")
    assert ck.shape == (Bsz, D, (L + 7) // 8, 16)
    assert not ck[:, :, 0].any()  # the state before step 0
    for k in range(1, (L + 7) // 8):
        sub = {n: (None if v is None else (v[..., :8 * k] if v.dim() == 3 and v.shape[-1] == L
                                         else v)) for n, v in inp.items()}
        _, sk = oracle.selective_scan(sub["u"], sub["delta"], sub["A"], sub["B"], sub["C"],
                                      sub["D"], sub["z"], sub["delta_bias"], nthreads=8)
        check_close(to_np(ck[:, :, k]), sk, _tdt(dt), f"state before step {8 * k}")


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:4])))
def test_backward_from_checkpoints(cuda_device, case):
    Bsz, D, L, dt, gate, skip, bias = case
    inp = inputs.selective_inputs(Bsz, D, 16, L, dt, gate=gate, skip=skip, bias=bias, seed=L + D)
    dout = inputs.grad_output((Bsz, D, L), dt, seed=L + D)
    g = cuda_inputs(inp, cuda_device)
    _, _, ck = _abi.selective_scan_fwd_ckpt(*_args(g))
    out = _abi.selective_scan_bwd_ckpt(*_args(g), dout.to(cuda_device), ck)
    plain = _abi.selective_scan_bwd(*_args(g), dout.to(cuda_device))
    torch.cuda.synchronize()
    assert _abi.device_error() == 0
    ref = oracle.selective_scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"],
                                    inp["D"], inp["z"], inp["delta_bias"], dout)
    for k in GRADS:
        if ref[k] is None:
            assert out[k] is None, k
            continue
        check_close(to_np(out[k]), ref[k], _tdt(dt), f"{k} from checkpoints")
        check_close(to_np(out[k]), to_np(plain[k]), _tdt(dt), f"{k} against the plain backward")


def test_layer_shape_matches_plain_backward_bitwise(cuda_device):
    """At the Mamba-130M layer shape the forward runs each sequence in one
    piece, so its checkpoints are the plain backward's own states and every
    gradient comes out bit for bit the same."""
    cfg = inputs.WORKLOADS["mamba130m_layer"]
    with inputs.on_device(cuda_device):
        g = inputs.workload_selective_inputs(cfg, seed=3)
        dout = inputs.grad_output((cfg.batch, cfg.d_inner, cfg.seqlen), cfg.dtype, seed=3)
    _, _, ck = _abi.selective_scan_fwd_ckpt(*_args(g))
    out = _abi.selective_scan_bwd_ckpt(*_args(g), dout, ck)
    plain = _abi.selective_scan_bwd(*_args(g), dout)
    torch.cuda.synchronize()
    assert _abi.device_error() == 0
    for k in GRADS:
        assert torch.equal(out[k], plain[k]), k


def test_checkpoint_calls_reject_what_they_do_not_take(cuda_device):
    inp = inputs.selective_inputs(1, 32, 16, 64, "bf16", seed=1)
    g = cuda_inputs(inp, cuda_device)
    dout = torch.zeros(1, 32, 64, dtype=torch.bfloat16, device=cuda_device)
    with pytest.raises(_abi.SSError, match="SHAPE"):  # wrong number of checkpoints
        _abi.selective_scan_fwd_ckpt(*_args(g), ckpt=torch.empty(1, 32, 9, 16, device=cuda_device))
    with pytest.raises(_abi.SSError, match="INVALID_ARG"):  # the backward needs them
        _abi.selective_scan_bwd_ckpt(*_args(g), dout, None)
    grouped = cuda_inputs(inputs.selective_inputs(1, 32, 16, 64, "bf16", groups=2, seed=1),
                          cuda_device)
    with pytest.raises(_abi.SSError, match="UNSUPPORTED"):  # B, C per channel group
        _abi.selective_scan_fwd_ckpt(*_args(grouped))
    small = cuda_inputs(inputs.selective_inputs(1, 32, 8, 64, "bf16", seed=1), cuda_device)
    with pytest.raises(_abi.SSError, match="UNSUPPORTED"):  # N = 8
        _abi.selective_scan_fwd_ckpt(*_args(small))
    # a time stride other than 1 (rows whose pitch is not a multiple of 16 bytes
    # are accepted: they run on padded copies, in CASES above)
    tv = dict(g)
    for k in ("u", "delta", "z"):
        tv[k] = g[k].transpose(1, 2).contiguous().transpose(1, 2)
    with pytest.raises(_abi.SSError, match="UNSUPPORTED"):
        _abi.selective_scan_fwd_ckpt(*_args(tv))


def test_empty_sequence_writes_the_zero_state(cuda_device):
    """L = 0: no checkpoints, and the final state is the zero state, as from
    the plain forward."""
    inp = inputs.selective_inputs(2, 32, 16, 0, "bf16", seed=2)
    g = cuda_inputs(inp, cuda_device)
    last = torch.full((2, 32, 16), float("nan"), device=cuda_device)
    ck = torch.empty(2, 32, 0, 16, device=cuda_device)
    _abi.selective_scan_fwd_ckpt(*_args(g), last_state=last, ckpt=ck)
    torch.cuda.synchronize()
    assert not last.any() and not last.isnan().any()
