"""Sequence lengths whose rows are not a multiple of 16 bytes (odd lengths in
bf16, lengths not a multiple of 4 in fp32) cannot be mapped by the fast
kernels' tensor maps; the library runs them on padded copies of the inputs
(and copies y back).  These cases check that path against the fp64 oracle:
the layer and long-sequence shapes at full size on sampled channels, B, C per
group, wider states, the fused conv, strided batch rows and one channel per
row (GPU, C ABI).  The backward takes the same route: the odd-length layer
shape against the oracle's backward, and the padded route against the
any-stride backward kernel."""
import pytest
import torch

import oracle
from selective_state_space_146_b300 import _abi, inputs
from tests.parity_util import check_close, cuda_inputs, oracle_selective_channels, to_np

pytestmark = pytest.mark.gpu


def _tdt(dt):
    return torch.float32 if dt == "f32" else torch.bfloat16


def _run(g, **kw):
    out = _abi.selective_scan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"],
                                  g["delta_bias"], return_last_state=True, **kw)
    torch.cuda.synchronize()
    assert _abi.device_error() == 0
    return out


@pytest.mark.parametrize("case", [(8, 1536, 16, 2047, "bf16", True, None),
                                  (1, 2048, 16, 16383, "bf16", False, None),
                                  (2, 256, 16, 1001, "bf16", True, 4),
                                  (2, 96, 64, 777, "bf16", True, None),
                                  (3, 40, 16, 1203, "f32", True, None),
                                  (4, 1, 16, 515, "bf16", True, None)],
                         ids=lambda c: "x".join(map(str, c[:5])) + (f"-G{c[6]}" if c[6] else ""))
def test_odd_length_matches_oracle(cuda_device, case):
    Bsz, D, N, L, dt, gate, G = case
    inp = inputs.selective_inputs(Bsz, D, N, L, dt, gate=gate, groups=G, seed=L + D)
    g = cuda_inputs(inp, cuda_device)
    y, s = _run(g)
    if Bsz * D * L <= 1 << 20 or G:
        yo, so = oracle.selective_scan(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"],
                                       inp["D"], inp["z"], inp["delta_bias"], nthreads=8)
        check_close(to_np(y), yo, _tdt(dt), "y")
        check_close(to_np(s), so, _tdt(dt), "last_state")
    else:
        chans = inputs.sample_units(Bsz * D, 12, seed=L)
        yo, so = oracle_selective_channels(inp, chans)
        idx = torch.as_tensor(chans, device=y.device)
        check_close(to_np(y.reshape(Bsz * D, L)[idx]), yo, _tdt(dt), "y (sampled channels)")
        check_close(to_np(s.reshape(Bsz * D, N)[idx]), so, _tdt(dt), "last_state (sampled)")


def test_odd_length_strided_batch_rows(cuda_device):
    """Batch rows further apart than D rows (a slice of a larger tensor): one
    2-D copy per batch row in and out."""
    Bsz, D, N, L = 3, 64, 16, 999
    inp = inputs.selective_inputs(Bsz, D, N, L, "bf16", seed=7)
    dev = cuda_device
    g = cuda_inputs(inp, dev)
    big = {k: torch.zeros(Bsz, D + 5, L, dtype=v.dtype, device=dev)
           for k, v in g.items() if k in ("u", "delta", "z")}
    for k in big:
        big[k][:, :D] = g[k]
    yb = torch.full((Bsz, D + 5, L), 7.0, dtype=g["u"].dtype, device=dev)
    y, s = _abi.selective_scan_fwd(big["u"][:, :D], big["delta"][:, :D], g["A"], g["B"], g["C"],
                                   g["D"], big["z"][:, :D], g["delta_bias"], y=yb[:, :D],
                                   return_last_state=True)
    torch.cuda.synchronize()
    yo, so = oracle.selective_scan(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                                   inp["z"], inp["delta_bias"], nthreads=8)
    check_close(to_np(yb[:, :D]), yo, torch.bfloat16, "y")
    check_close(to_np(s), so, torch.bfloat16, "last_state")
    assert bool((yb[:, D:] == 7.0).all())  # rows outside the view untouched


def test_odd_length_conv(cuda_device):
    Bsz, D, N, L, W = 2, 64, 16, 1027, 4
    inp = inputs.selective_inputs(Bsz, D, N, L, "bf16", seed=11)
    gen = torch.Generator().manual_seed(3)
    cw = torch.randn(D, W, generator=gen) * 0.5
    cb = torch.randn(D, generator=gen) * 0.1
    g = cuda_inputs(inp, cuda_device)
    y, s = _abi.conv_selective_scan_fwd(g["u"], cw.to(cuda_device), cb.to(cuda_device), g["delta"],
                                        g["A"], g["B"], g["C"], g["D"], g["z"], g["delta_bias"],
                                        return_last_state=True)
    torch.cuda.synchronize()
    assert _abi.device_error() == 0
    u = oracle.causal_conv1d_silu(inp["u"], cw, cb)
    yo, so = oracle.selective_scan(u, inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                                   inp["z"], inp["delta_bias"], nthreads=8)
    check_close(to_np(y), yo, torch.bfloat16, "y")
    check_close(to_np(s), so, torch.bfloat16, "last_state")


def test_odd_length_general_switch_agrees(cuda_device):
    """The general kernel (forced) and the padded fast path give the same
    results to within the bf16 bar."""
    inp = inputs.selective_inputs(2, 128, 16, 777, "bf16", seed=5)
    g = cuda_inputs(inp, cuda_device)
    y1, s1 = _run(g)
    with _abi.debug_paths(scan_path=0):
        y0, s0 = _run(g)
    check_close(to_np(y1), to_np(y0), torch.bfloat16, "y")
    check_close(to_np(s1), to_np(s0), torch.bfloat16, "last_state")


BWD_GRADS = ("du", "ddelta", "dz", "dA", "dB", "dC", "dD", "ddelta_bias")


def _bwd(g, dout):
    out = _abi.selective_scan_bwd(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"],
                                  g["delta_bias"], dout)
    torch.cuda.synchronize()
    assert _abi.device_error() == 0
    return out


def test_odd_length_backward_layer_shape(cuda_device):
    """Every gradient at 8 x 1536 x 2047 (bf16, gate on) against the full
    oracle backward; the call launches the row copies, scan_bwd_fast and its
    finishing sums, not the any-stride kernel."""
    Bsz, D, L = 8, 1536, 2047
    inp = inputs.selective_inputs(Bsz, D, 16, L, "bf16", seed=L)
    dout = inputs.grad_output((Bsz, D, L), "bf16", seed=L)
    g = cuda_inputs(inp, cuda_device)
    n0 = _abi.launch_count()
    out = _bwd(g, dout.to(cuda_device))
    assert _abi.launch_count() - n0 == 4  # pack, scan_bwd_fast, scan_bwd_finish, unpack
    ref = oracle.selective_scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"],
                                    inp["D"], inp["z"], inp["delta_bias"], dout)
    for k in BWD_GRADS:
        check_close(to_np(out[k]), ref[k], torch.bfloat16, f"odd-length backward {k}")


@pytest.mark.parametrize("case", [(2, 70, 999, "bf16", True), (3, 24, 301, "f32", False),
                                  (1, 1, 515, "bf16", True)],
                         ids=lambda c: "x".join(map(str, c[:4])))
def test_odd_length_backward_matches_any_stride_kernel(cuda_device, case):
    Bsz, D, L, dt, gate = case
    inp = inputs.selective_inputs(Bsz, D, 16, L, dt, gate=gate, seed=L + D)
    dout = inputs.grad_output((Bsz, D, L), dt, seed=L + D)
    g = cuda_inputs(inp, cuda_device)
    fast = _bwd(g, dout.to(cuda_device))
    with _abi.debug_paths(bwd_path=0):
        gen = _bwd(g, dout.to(cuda_device))
    ref = oracle.selective_scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"],
                                    inp["D"], inp["z"], inp["delta_bias"], dout)
    for k in BWD_GRADS:
        if ref[k] is None:
            assert fast[k] is None and gen[k] is None, k
            continue
        check_close(to_np(fast[k]), ref[k], _tdt(dt), f"padded backward {k}")
        check_close(to_np(fast[k]), to_np(gen[k]), _tdt(dt), f"padded vs any-stride {k}")
