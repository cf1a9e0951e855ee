"""The allocation-free entry point against the regular one (GPU, C ABI).

ss_selective_scan_fwd_noalloc serves callers that cannot allocate device
memory while a call runs (an arena or another runtime owns the allocator, a
loop must stay out of the CUDA allocator, or all free memory has been handed
to a pool).  It keeps its segment summaries in a fixed device array instead of
stream-ordered scratch.  Here it must give the same y and final state as
ss_selective_scan_fwd, on two calls in a row (the second call finds the first
call's data still in the shared array), both for a case that splits the
sequence into segments (so the fixed array is used) and for one that does not.

This file is collected last on purpose, and it also passes when run alone in a
fresh process (the first call on the device performs the array's set-up).
"""
import ctypes

import pytest
import torch

from selective_state_space_146_b300 import _abi, inputs
from tests.parity_util import check_close, cuda_inputs, to_np

pytestmark = pytest.mark.gpu


def _call(fn_name, g, y, last):
    lib = _abi.load()
    ts = [_abi.describe(t) for t in (g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"],
                                     g["delta_bias"])]
    ys, ls = _abi.describe(y), _abi.describe(last)
    refs = [None if t is None else ctypes.byref(t) for t in ts]
    rc = getattr(lib, fn_name)(*refs, 1, ctypes.byref(ys), ctypes.byref(ls),
                               torch.cuda.current_stream().cuda_stream)
    assert rc == 0, _abi.status_string(rc)


# (batch, d_inner, seqlen, dtype): the first three are split into segments
# (few channels, long sequence); in the third the fixed array holds fewer
# segments than the regular call uses (16 instead of 26); the last one is
# not split.
CASES = [(1, 64, 16384, "bf16"), (2, 24, 3000, "f32"), (1, 2048, 16384, "bf16"),
         (2, 256, 512, "bf16")]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_noalloc_matches_regular_entry_point(cuda_device, case):
    Bsz, D, L, dt = case
    inp = inputs.selective_inputs(Bsz, D, 16, L, dt, seed=L + D)
    g = cuda_inputs(inp, cuda_device)
    y_ref = torch.empty_like(g["u"])
    s_ref = torch.empty(Bsz, D, 16, device=cuda_device)
    _call("ss_selective_scan_fwd", g, y_ref, s_ref)
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    for _ in range(2):  # two calls in a row share the fixed array
        y = torch.full_like(g["u"], float("nan"))
        s = torch.full((Bsz, D, 16), float("nan"), device=cuda_device)
        _call("ss_selective_scan_fwd_noalloc", g, y, s)
        torch.cuda.synchronize()
        assert _abi.device_error() == 0
        check_close(to_np(y), to_np(y_ref), tdt, "y (no-alloc vs regular)")
        check_close(to_np(s), to_np(s_ref), tdt, "last_state (no-alloc vs regular)")
