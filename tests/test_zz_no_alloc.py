"""The allocation-free entry point against the regular one and the oracle (GPU, C ABI).

ss_selective_scan_fwd_noalloc serves callers that cannot allocate device
memory while a call runs (an arena or another runtime owns the allocator, a
loop must stay out of the CUDA allocator, or all free memory has been handed
to a pool).  It keeps its segment summaries in a fixed device array instead of
stream-ordered scratch.  Here it must give the same y and final state as
ss_selective_scan_fwd, on two calls in a row (the second call finds the first
call's data still in the shared array), and match the fp64 oracle on sampled
channels.  The cases cover a sequence split into segments (the fixed array
in use), one where the array holds fewer segments than the regular call uses,
one that is not split, B and C per channel group, and one with so many
channels that a single segment's summaries would not fit the array (the
segment count is capped to one, even when more are asked for).

This file is collected last on purpose, and it also passes when run alone in a
fresh process (the first call on the device performs the array's set-up).
"""
import ctypes

import pytest
import torch

import oracle
from selective_state_space_146_b300 import _abi, inputs
from tests.parity_util import check_close, cuda_inputs, oracle_selective_channels, to_np

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


# (batch, d_inner, seqlen, dtype, groups, forced segments)
CASES = [
    (1, 64, 16384, "bf16", None, None),    # split into segments: the fixed array in use
    (2, 24, 3000, "f32", None, None),
    (1, 2048, 16384, "bf16", None, None),  # the array holds fewer segments than the regular call
    (2, 256, 512, "bf16", None, None),     # not split
    (2, 128, 4096, "bf16", 2, None),       # B, C per group of 64 channels
    (2, 20480, 256, "bf16", None, 8),      # one segment's summaries exceed the array: capped to 1
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:4])) +
                         (f"-G{c[4]}" if c[4] else "") + (f"-s{c[5]}" if c[5] else ""))
def test_noalloc_matches_regular_entry_point_and_oracle(cuda_device, case):
    Bsz, D, L, dt, G, segs = case
    inp = inputs.selective_inputs(Bsz, D, 16, L, dt, groups=G, seed=L + D)
    g = cuda_inputs(inp, cuda_device)
    y_ref = torch.empty_like(g["u"])
    s_ref = torch.empty(Bsz, D, 16, device=cuda_device)
    _call("ss_selective_scan_fwd", g, y_ref, s_ref)
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    # the oracle on sampled channels (on all of them where B, C are grouped)
    if G:
        yo, so = oracle.selective_scan(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"],
                                       inp["D"], inp["z"], inp["delta_bias"], nthreads=8)
        chans = list(range(Bsz * D))
        yo, so = yo.reshape(Bsz * D, L), so.reshape(Bsz * D, 16)
    else:
        chans = inputs.sample_units(Bsz * D, 12, seed=L)
        yo, so = oracle_selective_channels(inp, chans)
    idx = torch.as_tensor(chans, device=cuda_device)
    with _abi.debug_paths(**({} if segs is None else dict(scan_segments=segs))):
        for _ in range(2):  # two calls in a row share the fixed array
            y = torch.full_like(g["u"], float("nan"))
            s = torch.full((Bsz, D, 16), float("nan"), device=cuda_device)
            _call("ss_selective_scan_fwd_noalloc", g, y, s)
            torch.cuda.synchronize()
            assert _abi.device_error() == 0
            check_close(to_np(y), to_np(y_ref), tdt, "y (no-alloc vs regular)")
            check_close(to_np(s), to_np(s_ref), tdt, "last_state (no-alloc vs regular)")
            check_close(to_np(y.reshape(Bsz * D, L)[idx]), yo, tdt, "y (no-alloc vs oracle)")
            check_close(to_np(s.reshape(Bsz * D, 16)[idx]), so, tdt,
                        "last_state (no-alloc vs oracle)")
