"""Shared helpers of the GPU parity tests: the tolerances and the comparison
against the fp64 oracle.

Tolerances (the stated bar for this scan): fp32 inputs -> max |err| <=
1e-4 * max |ref|; bf16 inputs -> relative L2 error <= 3e-3, against the
oracle run on the same bf16-rounded inputs (fp32 state and accumulation on
the GPU).  An output stored in bf16 carries its own rounding inside that
budget (about 1.7e-3 for normally distributed values); on an output of a few
elements rounding alone can cost more than 3e-3 (half a bf16 ulp is up to
2^-8 of the value), so there the bar is 1.5 times what rounding the oracle's
own values to bf16 costs (a value within a hair of a rounding midpoint may
round the other way), never less than 3e-3.
"""
import numpy as np
import torch

import oracle

TOL_F32_MAXABS = 1e-4
TOL_BF16_RELL2 = 3e-3


def to_np(t):
    return t.detach().float().cpu().double().numpy()


def check_close(got, want, dtype, what=""):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    scale = np.abs(want).max()
    if dtype == torch.float32:
        err = np.abs(got - want).max()
        assert err <= TOL_F32_MAXABS * max(scale, 1e-30), \
            f"{what}: max|err| {err:.3e} > 1e-4 * max|ref| ({scale:.3e})"
        return err / max(scale, 1e-30)
    num = np.linalg.norm((got - want).ravel())
    den = np.linalg.norm(want.ravel())
    rel = num / max(den, 1e-30)
    bar = TOL_BF16_RELL2
    if _bf16_valued(got):
        rounded = torch.from_numpy(want).to(torch.bfloat16).double().numpy()
        bar = max(bar, 1.5 * np.linalg.norm((rounded - want).ravel()) / max(den, 1e-30))
    assert rel <= bar, f"{what}: rel L2 {rel:.3e} > {bar:.3e}"
    return rel


def _bf16_valued(a):
    """Every value exactly a bf16 number (an output stored in bf16)."""
    bits = np.asarray(a, np.float32).view(np.uint32)
    return bool(np.all((bits & 0xFFFF) == 0))


def cuda_inputs(d, device):
    return {k: (None if v is None else v.to(device)) for k, v in d.items()}


def oracle_selective(inp, softplus=True, nthreads=8):
    return oracle.selective_scan(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                                 inp["z"], inp["delta_bias"], softplus=softplus, nthreads=nthreads)


def oracle_selective_channels(inp, chans, softplus=True, nthreads=8):
    """Oracle on a subset of (b, d) channels: each channel only needs its own
    row of u / delta / z, its row of A, D, bias and its batch row's B, C."""
    Dch = inp["u"].shape[1]
    ys, ss = [], []
    for c in chans:
        b, d = divmod(int(c), Dch)
        sub = {
            "u": inp["u"][b:b + 1, d:d + 1], "delta": inp["delta"][b:b + 1, d:d + 1],
            "z": None if inp["z"] is None else inp["z"][b:b + 1, d:d + 1],
            "A": inp["A"][d:d + 1], "B": inp["B"][b:b + 1], "C": inp["C"][b:b + 1],
            "D": None if inp["D"] is None else inp["D"][d:d + 1],
            "delta_bias": None if inp["delta_bias"] is None else inp["delta_bias"][d:d + 1],
        }
        y, s = oracle_selective(sub, softplus, nthreads=1)
        ys.append(y[0, 0])
        ss.append(s[0, 0])
    return np.stack(ys), np.stack(ss)


def oracle_ssd(inp, nthreads=8):
    return oracle.ssd(inp["x"], inp["dt"], inp["A_head"], inp["B"], inp["C"], inp["D"],
                      nthreads=nthreads)


def oracle_ssd_units(inp, units, nthreads=8):
    """Oracle on a subset of (b, h) units."""
    H = inp["x"].shape[2]
    G = inp["B"].shape[2]
    ys, ss = [], []
    for un in units:
        b, h = divmod(int(un), H)
        g = h // (H // G)
        y, s = oracle.ssd(inp["x"][b:b + 1, :, h:h + 1], inp["dt"][b:b + 1, :, h:h + 1],
                          inp["A_head"][h:h + 1], inp["B"][b:b + 1, :, g:g + 1],
                          inp["C"][b:b + 1, :, g:g + 1],
                          None if inp["D"] is None else inp["D"][h:h + 1], nthreads=1)
        ys.append(y[0, :, 0])
        ss.append(s[0, 0])
    return np.stack(ys), np.stack(ss)


def scan_switches(name):
    """Diagnostic switches (ss_debug_set_path) that force one selective-scan
    kernel: None (the library's choice), "general", "splitK" (scan_fast with K
    lanes per channel), "seqK" or "seqKsN" (scan_seq launch shape K, N time
    segments)."""
    if name is None:
        return {}
    if name == "general":
        return dict(scan_path=0)
    if name.startswith("split"):
        return dict(scan_path=1, scan_split=int(name[5:]))
    if name.startswith("seq"):
        shape, _, segs = name[3:].partition("s")
        sw = dict(scan_path=2, scan_shape=int(shape))
        if segs:
            sw["scan_segments"] = int(segs)
        return sw
    raise ValueError(name)


# SSD kernels: None (the library's choice), the CUDA-core kernel, the
# tensor-core kernels with no fallback, the one-head tensor-core kernel.
SSD_SWITCHES = {None: {}, "general": dict(ssd_path=0), "tc": dict(ssd_path=1),
                "tc1": dict(ssd_path=2)}
