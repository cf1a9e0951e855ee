"""Failure detection without a GPU fault (GPU).

* A kernel's bounded wait that runs out: ss_selftest_timeout waits on an
  mbarrier nothing arrives on, gives up after its limit and records the device
  error bit; the host reads SS_ERR_TIMEOUT, the word is cleared, and the next
  scan runs normally.
* Allocation failure injected on the host (ss_debug_set_path with
  SS_DEBUG_FAULT_ALLOC): calls that need stream-ordered scratch return
  SS_ERR_ALLOC without launching, calls that do not need it still run, and
  everything works again once the switch is off.
"""
import time

import pytest
import torch

import oracle
from selective_state_space_146_b300 import _abi, inputs
from tests.parity_util import check_close, cuda_inputs, to_np

pytestmark = pytest.mark.gpu

SS_ERR_ALLOC, SS_ERR_TIMEOUT = -6, -8


def _scan(g, **kw):
    return _abi.selective_scan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"],
                                   g["delta_bias"], **kw)


def test_bounded_wait_reports_timeout_and_context_survives(cuda_device):
    assert _abi.device_error() == 0
    t0 = time.perf_counter()
    _abi.selftest_timeout(limit_us=2000)
    assert _abi.device_error() == SS_ERR_TIMEOUT
    assert time.perf_counter() - t0 < 5.0
    assert _abi.device_error() == 0  # read and cleared
    inp = inputs.selective_inputs(1, 32, 16, 256, "f32", seed=3)
    g = cuda_inputs(inp, cuda_device)
    y = _scan(g)
    torch.cuda.synchronize()
    assert _abi.device_error() == 0
    yo, _ = oracle.selective_scan(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                                  inp["z"], inp["delta_bias"])
    check_close(to_np(y), yo, torch.float32, "y after the timeout self-test")


def test_selftest_rejects_bad_limits(cuda_device):
    for bad in (0, 100001):
        with pytest.raises(_abi.SSError, match="INVALID_ARG"):
            _abi.selftest_timeout(limit_us=bad)


def test_injected_allocation_failure(cuda_device):
    # few channels and a long sequence: the forward splits time into segments
    # and needs scratch for their summaries; the backward always needs scratch
    inp = inputs.selective_inputs(1, 32, 16, 8192, "bf16", seed=4)
    g = cuda_inputs(inp, cuda_device)
    dout = inputs.grad_output((1, 32, 8192), "bf16", seed=4).to(cuda_device)
    ref = _scan(g)
    torch.cuda.synchronize()
    n0 = _abi.launch_count()
    with _abi.debug_paths(fault_alloc=1):
        with pytest.raises(_abi.SSError, match="ALLOC"):
            _scan(g)
        with pytest.raises(_abi.SSError, match="ALLOC"):
            _abi.selective_scan_bwd(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"],
                                    g["delta_bias"], dout)
        pinned = {k: (None if v is None else v.pin_memory()) for k, v in inp.items()}
        with pytest.raises(_abi.SSError, match="ALLOC"):
            _abi.selective_scan_fwd_host(pinned["u"], pinned["delta"], pinned["A"], pinned["B"],
                                         pinned["C"], pinned["D"], pinned["z"],
                                         pinned["delta_bias"])
        assert _abi.launch_count() == n0  # nothing was launched
        # the fixed-scratch entry point allocates nothing and still runs
        y_fixed = torch.empty_like(g["u"])
        _abi.selective_scan_fwd_noalloc(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"],
                                        g["z"], g["delta_bias"], y=y_fixed)
        torch.cuda.synchronize()
    y = _scan(g)
    torch.cuda.synchronize()
    assert _abi.device_error() == 0
    assert torch.equal(y, ref)
    check_close(to_np(y_fixed), to_np(ref), torch.bfloat16, "fixed-scratch scan under the hook")
