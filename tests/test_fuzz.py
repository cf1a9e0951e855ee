"""Randomised parity: shapes, dtypes, optional inputs, strides and initial
states drawn by hypothesis (derandomised, so every run draws the same
examples), each compared with the fp64 oracle on the same seeded inputs.

Covers every compute entry point: the selective scan (shared and grouped
B, C, with and without an initial state; also with scan_seq forced to each
launch shape and to random segment counts), the fused conv + scan, the
backward, the SSD scan and both decode steps.  The sizes stay small so the
oracle answers in milliseconds; they still cross tile and chunk edges.
"""
import os

import numpy as np
import pytest
import torch
from hypothesis import HealthCheck, given, settings
from hypothesis import strategies as st

import oracle
from selective_state_space_146_b300 import _abi, inputs
from tests.parity_util import check_close, to_np

pytestmark = pytest.mark.gpu

# SS_FUZZ_EXAMPLES raises the number of drawn cases for a longer run (the
# default suite draws 30 per test, the same ones every run)
SETTINGS = settings(max_examples=int(os.environ.get("SS_FUZZ_EXAMPLES", "30")), deadline=None,
                    derandomize=True, database=None,
                    suppress_health_check=[HealthCheck.function_scoped_fixture])


def _tdt(dt):
    return torch.float32 if dt == "f32" else torch.bfloat16


def _to_dev(t, dev, layout):
    """Device copy of a (Bsz, D, L) activation in one of three layouts:
    contiguous, t-major storage seen as (Bsz, D, L), or a slice of a wider
    buffer (row stride larger than L)."""
    if t is None:
        return None
    t = t.to(dev)
    if layout == 1:
        return t.transpose(1, 2).contiguous().transpose(1, 2)
    if layout == 2:
        wide = torch.zeros(*t.shape[:-1], t.shape[-1] + 24, dtype=t.dtype, device=dev)
        wide[..., 8:8 + t.shape[-1]] = t
        return wide[..., 8:8 + t.shape[-1]]
    return t


def _dev(t, dev):
    return None if t is None else t.to(dev)


selective_case = st.fixed_dictionaries({
    "Bsz": st.integers(1, 3), "D": st.integers(1, 70), "N": st.sampled_from([1, 4, 8, 16, 16, 32]),
    "L": st.integers(1, 300), "dt": st.sampled_from(["f32", "bf16"]),
    "gate": st.booleans(), "skip": st.booleans(), "bias": st.booleans(), "sp": st.booleans(),
    "layout": st.sampled_from([0, 0, 1, 2]), "h0": st.booleans(),
    "groups": st.sampled_from([None, None, 1, "D", 2]), "seed": st.integers(0, 10_000),
})


@SETTINGS
@given(c=selective_case)
def test_fuzz_selective_scan(cuda_device, c):
    G = c["groups"]
    if G == "D":
        G = c["D"]
    if G == 2 and c["D"] % 2:
        G = 1
    inp = inputs.selective_inputs(c["Bsz"], c["D"], c["N"], c["L"], c["dt"], gate=c["gate"],
                                  skip=c["skip"], bias=c["bias"] and c["sp"], groups=G,
                                  seed=c["seed"])
    if not c["sp"]:
        inp["delta"] = inp["delta"].abs()  # without softplus the step must be positive
    h0 = (torch.randn(c["Bsz"], c["D"], c["N"], generator=torch.Generator().manual_seed(c["seed"]))
          if c["h0"] else None)
    dev = cuda_device
    y, s = _abi.selective_scan_fwd(
        _to_dev(inp["u"], dev, c["layout"]), _to_dev(inp["delta"], dev, c["layout"]),
        _dev(inp["A"], dev), _dev(inp["B"], dev), _dev(inp["C"], dev), _dev(inp["D"], dev),
        _to_dev(inp["z"], dev, c["layout"]), _dev(inp["delta_bias"], dev), softplus=c["sp"],
        return_last_state=True, initial_state=_dev(h0, dev))
    torch.cuda.synchronize()
    assert _abi.device_error() == 0
    yo, so = oracle.selective_scan(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                                   inp["z"], inp["delta_bias"], softplus=c["sp"], h0=h0, nthreads=8)
    check_close(to_np(y), yo, _tdt(c["dt"]), f"y {c}")
    check_close(to_np(s), so, _tdt(c["dt"]), f"state {c}")


@SETTINGS
@given(c=st.fixed_dictionaries({
    "Bsz": st.integers(1, 2), "D": st.integers(1, 300), "L": st.integers(1, 3000),
    "dt": st.sampled_from(["f32", "bf16"]), "gate": st.booleans(), "h0": st.booleans(),
    "shape": st.integers(1, 7), "segs": st.sampled_from([None, 1, 2, 3, 7, 40]),
    "groups": st.sampled_from([None, None, 2]), "seed": st.integers(0, 10_000)}))
def test_fuzz_scan_seq_shapes(cuda_device, c):
    """scan_seq forced to every launch shape and to random segment counts
    (summaries, the per-tile carry fold, ragged segments and channel tiles),
    with and without an initial state, against the oracle.  Calls the
    kernel does not take (rows not 16-byte multiples, groups not a multiple
    of the channel tile) run the library's other kernels."""
    G = c["groups"] if c["groups"] and c["D"] % 2 == 0 else None
    inp = inputs.selective_inputs(c["Bsz"], c["D"], 16, c["L"], c["dt"], gate=c["gate"],
                                  groups=G, seed=c["seed"])
    h0 = (torch.randn(c["Bsz"], c["D"], 16, generator=torch.Generator().manual_seed(c["seed"]))
          if c["h0"] else None)
    dev = cuda_device
    sw = dict(scan_path=2, scan_shape=c["shape"])
    if c["segs"]:
        sw["scan_segments"] = c["segs"]
    with _abi.debug_paths(**sw):
        y, s = _abi.selective_scan_fwd(*(_dev(inp[k], dev) for k in
                                         ("u", "delta", "A", "B", "C", "D", "z", "delta_bias")),
                                       return_last_state=True, initial_state=_dev(h0, dev))
        torch.cuda.synchronize()
    assert _abi.device_error() == 0
    yo, so = oracle.selective_scan(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                                   inp["z"], inp["delta_bias"], h0=h0, nthreads=8)
    check_close(to_np(y), yo, _tdt(c["dt"]), f"y {c}")
    check_close(to_np(s), so, _tdt(c["dt"]), f"state {c}")


@SETTINGS
@given(c=st.fixed_dictionaries({
    "Bsz": st.integers(1, 2), "D": st.integers(1, 48), "L": st.integers(1, 260),
    "W": st.integers(1, 4), "dt": st.sampled_from(["f32", "bf16"]), "cbias": st.booleans(),
    "seed": st.integers(0, 10_000)}))
def test_fuzz_conv_scan(cuda_device, c):
    inp = inputs.selective_inputs(c["Bsz"], c["D"], 16, c["L"], c["dt"], seed=c["seed"])
    g = torch.Generator().manual_seed(c["seed"] + 1)
    w = torch.randn(c["D"], c["W"], generator=g) * 0.5
    cb = torch.randn(c["D"], generator=g) * 0.1 if c["cbias"] else None
    dev = cuda_device
    y, s = _abi.conv_selective_scan_fwd(
        inp["u"].to(dev), w.to(dev), _dev(cb, dev), inp["delta"].to(dev), inp["A"].to(dev),
        inp["B"].to(dev), inp["C"].to(dev), inp["D"].to(dev), inp["z"].to(dev),
        inp["delta_bias"].to(dev), return_last_state=True)
    torch.cuda.synchronize()
    yo, so = oracle.conv_selective_scan(inp["u"], w, cb, inp["delta"], inp["A"], inp["B"],
                                        inp["C"], inp["D"], inp["z"], inp["delta_bias"],
                                        nthreads=8)
    check_close(to_np(y), yo, _tdt(c["dt"]), f"y {c}")
    check_close(to_np(s), so, _tdt(c["dt"]), f"state {c}")


@SETTINGS
@given(c=st.fixed_dictionaries({
    "Bsz": st.integers(1, 2), "D": st.integers(1, 70), "N": st.sampled_from([1, 5, 16, 16]),
    "L": st.integers(1, 300), "dt": st.sampled_from(["f32", "bf16"]), "gate": st.booleans(),
    "skip": st.booleans(), "bias": st.booleans(), "sp": st.booleans(),
    "seed": st.integers(0, 10_000)}))
def test_fuzz_backward(cuda_device, c):
    inp = inputs.selective_inputs(c["Bsz"], c["D"], c["N"], c["L"], c["dt"], gate=c["gate"],
                                  skip=c["skip"], bias=c["bias"] and c["sp"], seed=c["seed"])
    if not c["sp"]:
        inp["delta"] = inp["delta"].abs()
    dout = inputs.grad_output((c["Bsz"], c["D"], c["L"]), c["dt"], seed=c["seed"])
    dev = cuda_device
    out = _abi.selective_scan_bwd(*[_dev(inp[k], dev) for k in ("u", "delta", "A", "B", "C", "D",
                                                                "z", "delta_bias")],
                                  dout.to(dev), softplus=c["sp"])
    torch.cuda.synchronize()
    ref = oracle.selective_scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"],
                                    inp["D"], inp["z"], inp["delta_bias"], dout, softplus=c["sp"])
    for k, v in ref.items():
        if v is None:
            assert out[k] is None
        else:
            check_close(to_np(out[k]), v, _tdt(c["dt"]), f"{k} {c}")


@SETTINGS
@given(c=st.fixed_dictionaries({
    "Bsz": st.integers(1, 2), "L": st.integers(1, 400), "H": st.sampled_from([1, 2, 3, 4, 8]),
    "P": st.sampled_from([4, 16, 64]), "N": st.sampled_from([8, 32, 128]),
    "G": st.sampled_from([1, 2]), "dt": st.sampled_from(["f32", "bf16"]), "skip": st.booleans(),
    "h0": st.booleans(), "seed": st.integers(0, 10_000)}))
def test_fuzz_ssd(cuda_device, c):
    G = c["G"] if c["H"] % c["G"] == 0 else 1
    inp = inputs.ssd_inputs(c["Bsz"], c["L"], c["H"], c["P"], c["N"], G, c["dt"], skip=c["skip"],
                            seed=c["seed"])
    h0 = (torch.randn(c["Bsz"], c["H"], c["P"], c["N"],
                      generator=torch.Generator().manual_seed(c["seed"])) if c["h0"] else None)
    dev = cuda_device
    y, s = _abi.ssd_chunk_scan_fwd(*[_dev(inp[k], dev) for k in ("x", "dt", "A_head", "B", "C",
                                                                 "D")],
                                   chunk=128, return_last_state=True, initial_state=_dev(h0, dev))
    torch.cuda.synchronize()
    assert _abi.device_error() == 0
    yo, so = oracle.ssd(inp["x"], inp["dt"], inp["A_head"], inp["B"], inp["C"], inp["D"], h0=h0,
                        nthreads=8)
    check_close(to_np(y), yo, _tdt(c["dt"]), f"y {c}")
    check_close(to_np(s), so, _tdt(c["dt"]), f"state {c}")


@SETTINGS
@given(c=st.fixed_dictionaries({
    "Bsz": st.integers(1, 2), "L": st.integers(1, 1500), "H": st.sampled_from([1, 2, 3, 4, 6, 8, 16]),
    "G": st.sampled_from([1, 2, 4]), "skip": st.booleans(), "h0": st.booleans(),
    "late": st.booleans(), "seed": st.integers(0, 10_000)}))
def test_fuzz_ssd_tensor_core(cuda_device, c):
    """The tensor-core SSD kernels (bf16, headdim 64, d_state 128) with no
    fallback (a layout they do not take fails the test): random lengths over
    one to a dozen 128-step blocks with ragged tails, heads per group even
    (two-head kernel: the B buffers by block parity, M in TMEM) or odd
    (one-head kernel), initial state on or off, and the next block's
    cumulative sum forced late or left to timing; against the oracle."""
    H = c["H"]
    G = c["G"] if H % c["G"] == 0 else 1
    inp = inputs.ssd_inputs(c["Bsz"], c["L"], H, 64, 128, G, "bf16", skip=c["skip"], seed=c["seed"])
    h0 = (torch.randn(c["Bsz"], H, 64, 128, generator=torch.Generator().manual_seed(c["seed"]))
          if c["h0"] else None)
    dev = cuda_device
    # dt as a view into a buffer whose t-stride is a multiple of 8 (the
    # tensor map's rule for the tensor-core kernels)
    Hp = (H + 7) // 8 * 8
    dtb = torch.zeros(c["Bsz"], c["L"], Hp, dtype=inp["dt"].dtype, device=dev)
    dtb[:, :, :H] = inp["dt"].to(dev)
    sw = dict(ssd_path=1)
    if c["late"]:
        sw["ssd_late_cumsum"] = 1
    with _abi.debug_paths(**sw):
        y, s = _abi.ssd_chunk_scan_fwd(_dev(inp["x"], dev), dtb[:, :, :H],
                                       *[_dev(inp[k], dev) for k in ("A_head", "B", "C", "D")],
                                       chunk=256, return_last_state=True, initial_state=_dev(h0, dev))
        torch.cuda.synchronize()
    assert _abi.device_error() == 0
    yo, so = oracle.ssd(inp["x"], inp["dt"], inp["A_head"], inp["B"], inp["C"], inp["D"], h0=h0,
                        nthreads=8)
    check_close(to_np(y), yo, torch.bfloat16, f"y {c}")
    check_close(to_np(s), so, torch.bfloat16, f"state {c}")


@SETTINGS
@given(c=st.fixed_dictionaries({
    "Bsz": st.integers(1, 3), "D": st.integers(1, 40), "N": st.sampled_from([1, 16, 33]),
    "steps": st.integers(1, 6), "dt": st.sampled_from(["f32", "bf16"]), "gate": st.booleans(),
    "seed": st.integers(0, 10_000)}))
def test_fuzz_decode_steps(cuda_device, c):
    """Steps applied in turn reproduce the scan from the same initial state."""
    inp = inputs.selective_inputs(c["Bsz"], c["D"], c["N"], c["steps"], c["dt"], gate=c["gate"],
                                  seed=c["seed"])
    h0 = torch.randn(c["Bsz"], c["D"], c["N"], generator=torch.Generator().manual_seed(c["seed"]))
    dev = cuda_device
    state = h0.to(dev).clone()
    ys = []
    for t in range(c["steps"]):
        ys.append(_abi.selective_state_update(
            state, inp["u"][..., t].contiguous().to(dev), inp["delta"][..., t].contiguous().to(dev),
            inp["A"].to(dev), inp["B"][..., t].contiguous().to(dev),
            inp["C"][..., t].contiguous().to(dev), inp["D"].to(dev),
            None if inp["z"] is None else inp["z"][..., t].contiguous().to(dev),
            inp["delta_bias"].to(dev)))
    torch.cuda.synchronize()
    yo, so = oracle.selective_scan(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                                   inp["z"], inp["delta_bias"], h0=h0)
    check_close(to_np(torch.stack(ys, -1)), yo, _tdt(c["dt"]), f"y {c}")
    check_close(to_np(state), so, _tdt(c["dt"]), f"state {c}")


@SETTINGS
@given(c=st.fixed_dictionaries({
    "Bsz": st.integers(1, 2), "D": st.integers(1, 70), "L": st.integers(1, 260),
    "dt": st.sampled_from(["f32", "bf16"]), "gate": st.booleans(), "skip": st.booleans(),
    "bias": st.booleans(), "seed": st.integers(0, 10_000)}))
def test_fuzz_training_step_pair(cuda_device, c):
    """The forward that keeps the states and the backward that reads them:
    every gradient against the oracle, rows that are not 16-byte multiples
    included (those run on padded copies)."""
    inp = inputs.selective_inputs(c["Bsz"], c["D"], 16, c["L"], c["dt"], gate=c["gate"],
                                  skip=c["skip"], bias=c["bias"], seed=c["seed"])
    dout = inputs.grad_output((c["Bsz"], c["D"], c["L"]), c["dt"], seed=c["seed"])
    dev = cuda_device
    args = [_dev(inp[k], dev) for k in ("u", "delta", "A", "B", "C", "D", "z", "delta_bias")]
    y, _, ck = _abi.selective_scan_fwd_ckpt(*args)
    out = _abi.selective_scan_bwd_ckpt(*args, dout.to(dev), ck)
    torch.cuda.synchronize()
    assert _abi.device_error() == 0
    yo, _ = oracle.selective_scan(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                                  inp["z"], inp["delta_bias"], nthreads=8)
    check_close(to_np(y), yo, _tdt(c["dt"]), f"y {c}")
    ref = oracle.selective_scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"],
                                    inp["D"], inp["z"], inp["delta_bias"], dout)
    for k, v in ref.items():
        if v is None:
            assert out[k] is None
        else:
            check_close(to_np(out[k]), v, _tdt(c["dt"]), f"{k} {c}")
