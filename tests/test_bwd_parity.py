"""Backward of the selective scan on the GPU against the fp64 oracle.

The oracle's backward is pinned independently (finite differences of the
oracle's forward and planted mistakes, in test_oracle_pins.py); here every
gradient the CUDA kernel writes is compared element by element with it, on
the same seeded inputs, at sizes that span several 32-step recompute chunks
with ragged tails, channel counts that leave a partial 16-channel block, and
at the full Mamba-130M layer shape.
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


def _run(inp, dout, softplus, device):
    g = cuda_inputs(inp, device)
    out = _abi.selective_scan_bwd(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"],
                                  g["delta_bias"], dout.to(device), softplus=softplus)
    torch.cuda.synchronize()
    assert _abi.device_error() == 0
    return out


def _compare(out, ref, dt, tag):
    for k in GRADS:
        if ref[k] is None:
            assert out[k] is None, k
            continue
        check_close(to_np(out[k]), ref[k], _tdt(dt), f"{tag} {k}")


@pytest.fixture
def bwd_path(request):
    """None: the library's choice (the TMA kernel where the layout allows);
    "general": the any-stride kernel."""
    val = getattr(request, "param", None)
    with _abi.debug_paths(**(dict(bwd_path=0) if val == "general" else {})):
        yield val


CASES = [
    # Bsz, D, N, L, dtype, gate, skip, bias, softplus
    (2, 24, 16, 100, "f32", True, True, True, True),
    (2, 70, 16, 200, "bf16", True, True, True, True),
    (1, 32, 16, 8, "f32", True, True, True, True),
    (1, 64, 16, 72, "bf16", False, True, True, True),
    (2, 40, 16, 136, "bf16", True, True, False, False),
    (1, 40, 16, 333, "bf16", True, True, True, True),
    (2, 7, 5, 65, "f32", False, False, False, False),
    (1, 17, 16, 32, "f32", True, False, True, True),
    (1, 3, 1, 1, "f32", True, True, True, True),
    (3, 33, 16, 1000, "bf16", True, True, True, True),
    (2, 16, 16, 4097, "f32", True, True, True, True),
    (1, 16, 12, 64, "bf16", False, True, False, True),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:5])) +
                         ("" if all(c[5:]) else "-" + "".join("gsbp"[i] for i in range(4)
                                                              if not c[5 + i])))
@pytest.mark.parametrize("bwd_path", [None, "general"], indirect=True)
def test_bwd_matches_oracle(cuda_device, bwd_path, case):
    Bsz, D, N, L, dt, gate, skip, bias, sp = case
    inp = inputs.selective_inputs(Bsz, D, N, L, dt, gate=gate, skip=skip, bias=bias,
                                  seed=L + D)
    if not sp:  # without softplus the step must already be positive
        inp["delta"] = inp["delta"].abs()
    dout = inputs.grad_output((Bsz, D, L), dt, seed=L + D)
    out = _run(inp, dout, sp, cuda_device)
    ref = oracle.selective_scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"],
                                    inp["D"], inp["z"], inp["delta_bias"], dout, softplus=sp)
    _compare(out, ref, dt, "x".join(map(str, case[:5])))


def test_bwd_noncontiguous_activations(cuda_device):
    """Activations and their gradients through views with a time stride."""
    Bsz, D, N, L = 2, 20, 16, 150
    inp = inputs.selective_inputs(Bsz, D, N, L, "f32", seed=5)
    dout = inputs.grad_output((Bsz, D, L), "f32", seed=5)
    g = cuda_inputs(inp, cuda_device)
    # (Bsz, L, D) storage seen as (Bsz, D, L)
    tv = {k: g[k].transpose(1, 2).contiguous().transpose(1, 2) for k in ("u", "delta", "z")}
    out = _abi.selective_scan_bwd(tv["u"], tv["delta"], g["A"], g["B"], g["C"], g["D"], tv["z"],
                                  g["delta_bias"],
                                  dout.to(cuda_device).transpose(1, 2).contiguous().transpose(1, 2))
    torch.cuda.synchronize()
    ref = oracle.selective_scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"],
                                    inp["D"], inp["z"], inp["delta_bias"], dout)
    _compare(out, ref, "f32", "transposed views")


def test_bwd_empty_inputs_zero_the_sums(cuda_device):
    for Bsz, D, L in ((2, 8, 0), (0, 8, 16)):
        inp = inputs.selective_inputs(Bsz, D, 16, L, "f32", seed=1)
        dout = inputs.grad_output((Bsz, D, L), "f32", seed=1)
        g = cuda_inputs(inp, cuda_device)
        out = _abi.selective_scan_bwd(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"],
                                      g["delta_bias"], dout.to(cuda_device))
        torch.cuda.synchronize()
        for k in ("dA", "dD", "ddelta_bias"):
            assert not out[k].any(), k
        assert out["du"].shape == (Bsz, D, L)


def test_bwd_rejects_wide_state(cuda_device):
    inp = inputs.selective_inputs(1, 4, 32, 16, "f32", seed=2)
    g = cuda_inputs(inp, cuda_device)
    dout = torch.zeros(1, 4, 16, device=cuda_device)
    with pytest.raises(_abi.SSError, match="UNSUPPORTED"):
        _abi.selective_scan_bwd(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"],
                                g["delta_bias"], dout)


def test_bwd_fast_path_is_deterministic(cuda_device, bwd_path):
    """The TMA kernel adds its partial sums in a fixed order: two calls give
    the same bits."""
    inp = inputs.selective_inputs(2, 96, 16, 512, "bf16", seed=9)
    dout = inputs.grad_output((2, 96, 512), "bf16", seed=9)
    a = _run(inp, dout, True, cuda_device)
    b = _run(inp, dout, True, cuda_device)
    for k in GRADS:
        assert torch.equal(a[k], b[k]), k


@pytest.mark.parametrize("bwd_path", [None, "general"], indirect=True)
def test_bwd_headline_layer_shape(cuda_device, bwd_path):
    """Every gradient at the Mamba-130M layer shape (8 x 1536 x 2048, N = 16,
    bf16) against the full oracle (single-threaded C, a few seconds)."""
    cfg = inputs.WORKLOADS["mamba130m_layer"]
    inp = inputs.workload_selective_inputs(cfg, seed=0)
    dout = inputs.grad_output((cfg.batch, cfg.d_inner, cfg.seqlen), cfg.dtype, seed=0)
    out = _run(inp, dout, True, cuda_device)
    ref = oracle.selective_scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"],
                                    inp["D"], inp["z"], inp["delta_bias"], dout)
    _compare(out, ref, cfg.dtype, "mamba130m_layer")
    # the fp32 sums at the full shape also hold elementwise to 1e-3 of their scale
    for k in ("dA", "dB", "dC", "dD", "ddelta_bias"):
        got, want = to_np(out[k]), ref[k]
        assert np.abs(got - want).max() <= 1e-3 * np.abs(want).max(), k
