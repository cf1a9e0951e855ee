"""fp64 CPU oracle for the selective scan and the Mamba-2 SSD scan.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The product
library never loads it and shares no code with it.

The arithmetic lives in ``oracle.c`` (plain C, double precision, one
sequential loop per independent unit).  This module only compiles it with
gcc, loads it with ctypes and converts numpy arrays to contiguous float64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def compile_source(src: str, out: str) -> str:
    """Compile a C source of the oracle's form into a shared library."""
    tmp = out + f".tmp{os.getpid()}"
    # -ffp-contract=off: no fused multiply-add, so every product and sum is
    # rounded exactly as written.
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", "-std=c99",
           src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, -O2, OpenMP over units)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        compile_source(_SRC, _LIB)
    return _LIB


def _bind(path):
    lib = ctypes.CDLL(path)
    i64, dp, ip = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
    lib.oracle_selective_scan.argtypes = [i64, i64, i64, i64] + [dp] * 8 + [ip, dp, dp, dp, ip]
    lib.oracle_selective_scan.restype = ip
    lib.oracle_selective_scan_grouped.argtypes = [i64] * 5 + [dp] * 8 + [ip, dp, dp, dp, ip]
    lib.oracle_selective_scan_grouped.restype = ip
    lib.oracle_ssd.argtypes = [i64] * 6 + [dp] * 6 + [dp, dp, dp, ip]
    lib.oracle_ssd.restype = ip
    lib.oracle_threads.restype = ip
    lib.oracle_causal_conv1d_silu.argtypes = [i64] * 4 + [dp] * 4 + [ip]
    lib.oracle_causal_conv1d_silu.restype = ip
    lib.oracle_selective_scan_bwd.argtypes = [i64] * 4 + [dp] * 8 + [ip] + [dp] * 9
    lib.oracle_selective_scan_bwd.restype = ip
    return lib


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = _bind(_LIB)
    return _lib


class _Bound:
    """The two oracle functions bound to one compiled library (used by the
    planted-mistake tests to run the pins against a mutated copy)."""

    def __init__(self, lib):
        self._lib = lib

    def selective_scan(self, *a, **k):
        return selective_scan(*a, _lib=self._lib, **k)

    def ssd(self, *a, **k):
        return ssd(*a, _lib=self._lib, **k)

    def causal_conv1d_silu(self, *a, **k):
        return causal_conv1d_silu(*a, _lib=self._lib, **k)

    def selective_scan_bwd(self, *a, **k):
        return selective_scan_bwd(*a, _lib=self._lib, **k)


def load_library(path: str) -> _Bound:
    return _Bound(_bind(path))


def max_threads() -> int:
    return int(_load().oracle_threads())


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor: exact upcast of bf16 / fp32 values
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def selective_scan(u, delta, A, B, C, D=None, z=None, delta_bias=None,
                   softplus=True, h0=None, nthreads=1, _lib=None):
    """Oracle of the selective scan.

    Shapes: u, delta, z (Bsz, Dch, L); A (Dch, N); B, C (Bsz, N, L), or
    (Bsz, G, N, L) with one B, C per group of Dch / G consecutive channels;
    D, delta_bias (Dch,); h0 (Bsz, Dch, N).  Returns (y, last_state), both
    float64 numpy arrays of shapes (Bsz, Dch, L) and (Bsz, Dch, N).
    """
    u, delta, A, B, C = (_f64(t) for t in (u, delta, A, B, C))
    D, z, delta_bias, h0 = (_f64(t) for t in (D, z, delta_bias, h0))
    Bsz, Dch, L = u.shape
    N = A.shape[1]
    grouped = B.ndim == 4
    G = B.shape[1] if grouped else 1
    assert delta.shape == u.shape and A.shape == (Dch, N)
    if grouped:
        assert B.shape == (Bsz, G, N, L) and C.shape == B.shape and Dch % G == 0
    else:
        assert B.shape == (Bsz, N, L) and C.shape == (Bsz, N, L)
    assert z is None or z.shape == u.shape
    assert D is None or D.shape == (Dch,)
    assert delta_bias is None or delta_bias.shape == (Dch,)
    assert h0 is None or h0.shape == (Bsz, Dch, N)
    y = np.empty((Bsz, Dch, L), np.float64)
    last = np.empty((Bsz, Dch, N), np.float64)
    lib = _lib or _load()
    if grouped:
        rc = lib.oracle_selective_scan_grouped(Bsz, Dch, G, N, L, _ptr(u), _ptr(delta), _ptr(A),
                                               _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                                               _ptr(delta_bias), int(bool(softplus)), _ptr(h0),
                                               _ptr(y), _ptr(last), int(nthreads))
    else:
        rc = lib.oracle_selective_scan(Bsz, Dch, N, L, _ptr(u), _ptr(delta), _ptr(A), _ptr(B),
                                       _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias),
                                       int(bool(softplus)), _ptr(h0), _ptr(y), _ptr(last),
                                       int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_selective_scan rejected its arguments (rc={rc})")
    return y, last


def ssd(x, dt, A_head, B, C, D=None, h0=None, nthreads=1, _lib=None):
    """Oracle of the Mamba-2 SSD scan (recurrent form).

    Shapes: x (Bsz, L, H, P); dt (Bsz, L, H); A_head (H,); B, C (Bsz, L, G, N);
    D (H,); h0 (Bsz, H, P, N).  Returns (y, last_state) as float64 arrays of
    shapes (Bsz, L, H, P) and (Bsz, H, P, N).
    """
    x, dt, A_head, B, C = (_f64(t) for t in (x, dt, A_head, B, C))
    D, h0 = _f64(D), _f64(h0)
    Bsz, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    assert dt.shape == (Bsz, L, H) and A_head.shape == (H,)
    assert B.shape == (Bsz, L, G, N) and C.shape == B.shape and H % G == 0
    assert D is None or D.shape == (H,)
    assert h0 is None or h0.shape == (Bsz, H, P, N)
    y = np.empty((Bsz, L, H, P), np.float64)
    last = np.empty((Bsz, H, P, N), np.float64)
    rc = (_lib or _load()).oracle_ssd(Bsz, L, H, P, G, N, _ptr(x), _ptr(dt), _ptr(A_head), _ptr(B),
                            _ptr(C), _ptr(D), _ptr(h0), _ptr(y), _ptr(last), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_ssd rejected its arguments (rc={rc})")
    return y, last


def causal_conv1d_silu(x, w, bias=None, nthreads=1, _lib=None):
    """Oracle of the causal depthwise conv1d + SiLU.  x (Bsz, D, L); w (D, W);
    bias (D,).  Returns u (Bsz, D, L) float64."""
    x, w, bias = _f64(x), _f64(w), _f64(bias)
    Bsz, D, L = x.shape
    W = w.shape[1]
    assert w.shape == (D, W) and (bias is None or bias.shape == (D,))
    u = np.empty_like(x)
    rc = (_lib or _load()).oracle_causal_conv1d_silu(Bsz, D, L, W, _ptr(x), _ptr(w), _ptr(bias),
                                                     _ptr(u), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_causal_conv1d_silu rejected its arguments (rc={rc})")
    return u


def conv_selective_scan(x, conv_w, conv_bias, delta, A, B, C, D=None, z=None, delta_bias=None,
                        softplus=True, h0=None, nthreads=1):
    """The conv branch feeding the scan: u = silu(causal_conv1d(x)), then the
    selective scan of u (the two oracle functions composed)."""
    u = causal_conv1d_silu(x, conv_w, conv_bias, nthreads=nthreads)
    return selective_scan(u, delta, A, B, C, D, z, delta_bias, softplus=softplus, h0=h0,
                          nthreads=nthreads)


def selective_scan_bwd(u, delta, A, B, C, D, z, delta_bias, dout, softplus=True, _lib=None):
    """Oracle of the selective scan's backward pass.  Returns a dict of float64
    arrays: du, ddelta, dz (like u), dA (like A), dB, dC (like B), dD,
    ddelta_bias (like D); entries for absent optional inputs are None."""
    u, delta, A, B, C, dout = (_f64(t) for t in (u, delta, A, B, C, dout))
    D, z, delta_bias = _f64(D), _f64(z), _f64(delta_bias)
    Bsz, Dch, L = u.shape
    N = A.shape[1]
    out = {"du": np.empty_like(u), "ddelta": np.empty_like(u), "dA": np.empty_like(A),
           "dB": np.empty_like(B), "dC": np.empty_like(C),
           "dD": None if D is None else np.empty_like(D),
           "dz": None if z is None else np.empty_like(z),
           "ddelta_bias": None if delta_bias is None else np.empty_like(delta_bias)}
    rc = (_lib or _load()).oracle_selective_scan_bwd(
        Bsz, Dch, N, L, _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
        _ptr(delta_bias), int(bool(softplus)), _ptr(dout), _ptr(out["du"]), _ptr(out["ddelta"]),
        _ptr(out["dA"]), _ptr(out["dB"]), _ptr(out["dC"]), _ptr(out["dD"]), _ptr(out["dz"]),
        _ptr(out["ddelta_bias"]))
    if rc != 0:
        raise ValueError(f"oracle_selective_scan_bwd failed (rc={rc})")
    return out
