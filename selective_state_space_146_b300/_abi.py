"""ctypes binding of libssscan.so (include/ssscan.h).

Argument marshalling only: torch tensors are described as ss_tensor
(pointer, dtype, shape, strides) and passed with the current CUDA stream.
Every step of the scan runs in the library's CUDA kernels; there is no other
implementation behind these functions.  If the library is missing the first
call raises.
"""
from __future__ import annotations

import contextlib
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libssscan.so")

SS_F32, SS_BF16 = 0, 1
STATUS = {0: "SS_OK", -1: "SS_ERR_INVALID_ARG", -2: "SS_ERR_SHAPE", -3: "SS_ERR_DTYPE",
          -4: "SS_ERR_ALIGNMENT", -5: "SS_ERR_UNSUPPORTED", -6: "SS_ERR_ALLOC",
          -7: "SS_ERR_LAUNCH", -8: "SS_ERR_TIMEOUT", -9: "SS_ERR_CUDA"}
EXPORTS = ("ss_selective_scan_fwd", "ss_selective_scan_fwd_noalloc", "ss_ssd_chunk_scan_fwd",
           "ss_selective_scan_fwd_init", "ss_ssd_chunk_scan_fwd_init", "ss_selective_state_update",
           "ss_conv_selective_scan_fwd", "ss_selective_scan_bwd", "ss_selective_scan_fwd_host",
           "ss_ssd_state_update", "ss_status_string", "ss_get_device_error", "ss_launch_count",
           "ss_version", "ss_selftest_timeout", "ss_selective_scan_fwd_ckpt",
           "ss_selective_scan_bwd_ckpt", "ss_debug_set_path", "ss_probe_ex2_rate",
           "ss_probe_scan_forms", "ss_ssd_chunk_scan_fwd_host")
# Diagnostic switches of ss_debug_set_path (include/ssscan.h, SS_DEBUG_*).
DEBUG = dict(scan_path=0, scan_split=1, scan_shape=2, scan_segments=3, ssd_path=4, bwd_path=5,
             grouped_path=6, fault_alloc=7, scan_seg_tiles=8, ssd_late_cumsum=9)


class SSTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4), ("stride", ctypes.c_int64 * 4)]


class SSError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)} ({status_string(status)})")


_lib = None


def load(path: str | None = None):
    """Load the library (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libssscan.so not built at {p}; run "
                           "`python -m selective_state_space_146_b300.csrc.build`")
    lib = ctypes.CDLL(p)
    T = ctypes.POINTER(SSTensor)
    vp, i = ctypes.c_void_p, ctypes.c_int
    lib.ss_selective_scan_fwd.argtypes = [T, T, T, T, T, T, T, T, i, T, T, vp]
    lib.ss_selective_scan_fwd.restype = i
    lib.ss_selective_scan_fwd_noalloc.argtypes = [T, T, T, T, T, T, T, T, i, T, T, vp]
    lib.ss_selective_scan_fwd_noalloc.restype = i
    lib.ss_ssd_chunk_scan_fwd.argtypes = [T, T, T, T, T, T, i, T, T, vp]
    lib.ss_ssd_chunk_scan_fwd.restype = i
    lib.ss_ssd_chunk_scan_fwd_host.argtypes = [T, T, T, T, T, T, i, T, T, vp]
    lib.ss_ssd_chunk_scan_fwd_host.restype = i
    lib.ss_selective_scan_fwd_init.argtypes = [T, T, T, T, T, T, T, T, i, T, T, T, vp]
    lib.ss_selective_scan_fwd_init.restype = i
    lib.ss_ssd_chunk_scan_fwd_init.argtypes = [T, T, T, T, T, T, i, T, T, T, vp]
    lib.ss_ssd_chunk_scan_fwd_init.restype = i
    lib.ss_selective_state_update.argtypes = [T, T, T, T, T, T, T, T, T, i, T, vp]
    lib.ss_selective_state_update.restype = i
    lib.ss_conv_selective_scan_fwd.argtypes = [T, T, T, T, T, T, T, T, T, T, i, T, T, vp]
    lib.ss_conv_selective_scan_fwd.restype = i
    lib.ss_selective_scan_fwd_host.argtypes = [T, T, T, T, T, T, T, T, i, T, T, vp]
    lib.ss_selective_scan_fwd_host.restype = i
    lib.ss_selective_scan_bwd.argtypes = [T, T, T, T, T, T, T, T, i, T, T, T, T, T, T, T, T, T,
                                          vp]
    lib.ss_selective_scan_bwd.restype = i
    lib.ss_selective_scan_fwd_ckpt.argtypes = [T, T, T, T, T, T, T, T, i, T, T, T, vp]
    lib.ss_selective_scan_fwd_ckpt.restype = i
    lib.ss_selective_scan_bwd_ckpt.argtypes = [T, T, T, T, T, T, T, T, i, T, T, T, T, T, T, T, T,
                                               T, T, vp]
    lib.ss_selective_scan_bwd_ckpt.restype = i
    lib.ss_ssd_state_update.argtypes = [T, T, T, T, T, T, T, T, vp]
    lib.ss_ssd_state_update.restype = i
    lib.ss_status_string.argtypes = [i]
    lib.ss_status_string.restype = ctypes.c_char_p
    lib.ss_get_device_error.argtypes = [vp]
    lib.ss_get_device_error.restype = i
    lib.ss_selftest_timeout.argtypes = [ctypes.c_uint, vp]
    lib.ss_selftest_timeout.restype = i
    lib.ss_launch_count.argtypes = []
    lib.ss_launch_count.restype = ctypes.c_uint64
    lib.ss_version.restype = i
    lib.ss_debug_set_path.argtypes = [i, i]
    lib.ss_debug_set_path.restype = i
    lib.ss_probe_ex2_rate.argtypes = [ctypes.POINTER(ctypes.c_double), vp]
    lib.ss_probe_ex2_rate.restype = i
    lib.ss_probe_scan_forms.argtypes = [ctypes.POINTER(ctypes.c_double),
                                        ctypes.POINTER(ctypes.c_double), vp]
    lib.ss_probe_scan_forms.restype = i
    if path is None:
        _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().ss_status_string(int(status)).decode()


_DT = {torch.float32: SS_F32, torch.bfloat16: SS_BF16}


def describe(t: torch.Tensor | None):
    """ss_tensor for a torch tensor (None -> NULL)."""
    if t is None:
        return None
    s = SSTensor()
    s.data = t.data_ptr() if t.numel() > 0 else 0
    s.dtype = _DT.get(t.dtype, 99)
    s.ndim = t.dim()
    for k in range(t.dim()):
        s.shape[k] = t.shape[k]
        s.stride[k] = t.stride(k)
    return s


def _ref(s):
    return None if s is None else ctypes.byref(s)


def _stream_ptr(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def selective_scan_fwd(u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True,
                       y=None, last_state=None, return_last_state=False, initial_state=None,
                       stream=None):
    """Selective scan forward (ss_selective_scan_fwd; ss_selective_scan_fwd_init
    when an initial state is given).

    u, delta, z: (batch, d_inner, L); A: (d_inner, N) f32; B, C: (batch, N, L);
    D, delta_bias: (d_inner,) f32; initial_state (batch, d_inner, N) f32.
    Returns y (same dtype as u), or (y, last_state) with last_state
    (batch, d_inner, N) f32.
    """
    if y is None:
        y = torch.empty_like(u, memory_format=torch.contiguous_format)
    if last_state is None and return_last_state:
        last_state = torch.empty(u.shape[0], u.shape[1], A.shape[1], dtype=torch.float32,
                                 device=u.device)
    ts = [describe(t) for t in (u, delta, A, B, C, D, z, delta_bias)]
    ys, ls = describe(y), describe(last_state)
    if initial_state is None:
        rc = load().ss_selective_scan_fwd(*[_ref(t) for t in ts], int(bool(softplus)), _ref(ys),
                                          _ref(ls), _stream_ptr(stream))
        what = "ss_selective_scan_fwd"
    else:
        rc = load().ss_selective_scan_fwd_init(*[_ref(t) for t in ts], int(bool(softplus)),
                                               _ref(describe(initial_state)), _ref(ys), _ref(ls),
                                               _stream_ptr(stream))
        what = "ss_selective_scan_fwd_init"
    if rc != 0:
        raise SSError(rc, what)
    return (y, last_state) if (return_last_state or last_state is not None) else y


def selective_scan_fwd_host(u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True,
                            y=None, last_state=None, return_last_state=False, stream=None):
    """ss_selective_scan_fwd_host: the selective scan with every tensor in
    host memory (contiguous CPU tensors, pinned for asynchronous copies).
    The results are valid once `stream` (default: the current CUDA stream) has
    completed."""
    if y is None:
        y = torch.empty(u.shape, dtype=u.dtype, pin_memory=True)
    if last_state is None and return_last_state:
        last_state = torch.empty(u.shape[0], u.shape[1], A.shape[1], dtype=torch.float32,
                                 pin_memory=True)
    ts = [describe(t) for t in (u, delta, A, B, C, D, z, delta_bias)]
    rc = load().ss_selective_scan_fwd_host(*[_ref(t) for t in ts], int(bool(softplus)),
                                           _ref(describe(y)), _ref(describe(last_state)),
                                           _stream_ptr(stream))
    if rc != 0:
        raise SSError(rc, "ss_selective_scan_fwd_host")
    return (y, last_state) if (return_last_state or last_state is not None) else y


def ssd_chunk_scan_fwd_host(x, dt, A_head, B, C, D=None, chunk=256, y=None, last_state=None,
                            return_last_state=False, stream=None):
    """ss_ssd_chunk_scan_fwd_host: the SSD scan with every tensor in host
    memory (contiguous CPU tensors, pinned for asynchronous copies).  The
    results are valid once `stream` (default: the current CUDA stream) has
    completed."""
    if y is None:
        y = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
    if last_state is None and return_last_state:
        last_state = torch.empty(x.shape[0], x.shape[2], x.shape[3], B.shape[3],
                                 dtype=torch.float32, pin_memory=True)
    ts = [describe(t) for t in (x, dt, A_head, B, C, D)]
    rc = load().ss_ssd_chunk_scan_fwd_host(*[_ref(t) for t in ts], int(chunk), _ref(describe(y)),
                                           _ref(describe(last_state)), _stream_ptr(stream))
    if rc != 0:
        raise SSError(rc, "ss_ssd_chunk_scan_fwd_host")
    return (y, last_state) if (return_last_state or last_state is not None) else y


def selective_scan_fwd_noalloc(u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True,
                               y=None, last_state=None, stream=None):
    """ss_selective_scan_fwd_noalloc: the selective scan for callers that
    cannot allocate device memory during a call.  The library allocates
    nothing; the caller passes every input and output, here y and (optionally)
    last_state already allocated.  See include/ssscan.h for the fixed 4 MiB
    scratch array it uses and for the rule that overlapping calls race."""
    if y is None:
        raise ValueError("selective_scan_fwd_noalloc needs a caller-allocated y")
    ts = [describe(t) for t in (u, delta, A, B, C, D, z, delta_bias)]
    ys, ls = describe(y), describe(last_state)
    rc = load().ss_selective_scan_fwd_noalloc(*[_ref(t) for t in ts], int(bool(softplus)),
                                              _ref(ys), _ref(ls), _stream_ptr(stream))
    if rc != 0:
        raise SSError(rc, "ss_selective_scan_fwd_noalloc")
    return (y, last_state) if last_state is not None else y


def ssd_chunk_scan_fwd(x, dt, A_head, B, C, D=None, chunk=256, y=None, last_state=None,
                       return_last_state=False, initial_state=None, stream=None):
    """Mamba-2 SSD chunked scan forward (ss_ssd_chunk_scan_fwd; the _init
    variant when an initial state is given).

    x: (batch, L, H, P); dt: (batch, L, H) positive; A_head, D: (H,) f32;
    B, C: (batch, L, G, N); initial_state (batch, H, P, N) f32.  Returns y, or
    (y, last_state (batch, H, P, N) f32).
    """
    if y is None:
        y = torch.empty_like(x, memory_format=torch.contiguous_format)
    if last_state is None and return_last_state:
        last_state = torch.empty(x.shape[0], x.shape[2], x.shape[3], B.shape[3],
                                 dtype=torch.float32, device=x.device)
    ts = [describe(t) for t in (x, dt, A_head, B, C, D)]
    ys, ls = describe(y), describe(last_state)
    if initial_state is None:
        rc = load().ss_ssd_chunk_scan_fwd(*[_ref(t) for t in ts], int(chunk), _ref(ys), _ref(ls),
                                          _stream_ptr(stream))
    else:
        rc = load().ss_ssd_chunk_scan_fwd_init(*[_ref(t) for t in ts], int(chunk),
                                               _ref(describe(initial_state)), _ref(ys), _ref(ls),
                                               _stream_ptr(stream))
    if rc != 0:
        raise SSError(rc, "ss_ssd_chunk_scan_fwd")
    return (y, last_state) if (return_last_state or last_state is not None) else y


def conv_selective_scan_fwd(x, conv_weight, conv_bias, delta, A, B, C, D=None, z=None,
                            delta_bias=None, softplus=True, y=None, last_state=None,
                            return_last_state=False, stream=None):
    """Fused causal conv1d + SiLU + selective scan (ss_conv_selective_scan_fwd).
    x: (batch, d_inner, L); conv_weight: (d_inner, W <= 4) f32; conv_bias (d_inner,)."""
    if y is None:
        y = torch.empty_like(x, memory_format=torch.contiguous_format)
    if last_state is None and return_last_state:
        last_state = torch.empty(x.shape[0], x.shape[1], A.shape[1], dtype=torch.float32,
                                 device=x.device)
    ts = [describe(t) for t in (x, conv_weight, conv_bias, delta, A, B, C, D, z, delta_bias)]
    rc = load().ss_conv_selective_scan_fwd(*[_ref(t) for t in ts], int(bool(softplus)),
                                           _ref(describe(y)), _ref(describe(last_state)),
                                           _stream_ptr(stream))
    if rc != 0:
        raise SSError(rc, "ss_conv_selective_scan_fwd")
    return (y, last_state) if (return_last_state or last_state is not None) else y


def selective_scan_bwd(u, delta, A, B, C, D, z, delta_bias, dout, softplus=True, stream=None):
    """Gradients of the selective scan (ss_selective_scan_bwd) for the
    incoming gradient dout of y.  Returns a dict with du, ddelta, dz (dtype of
    u), dA, dB, dC, dD, ddelta_bias (f32); the optional ones are None when the
    matching input is None."""
    f32 = dict(dtype=torch.float32, device=u.device)
    Bsz, Dch, L = u.shape
    N = A.shape[1]
    g = dict(du=torch.empty_like(u, memory_format=torch.contiguous_format),
             ddelta=torch.empty_like(u, memory_format=torch.contiguous_format),
             dz=None if z is None else torch.empty_like(u, memory_format=torch.contiguous_format),
             dA=torch.empty(Dch, N, **f32), dB=torch.empty(Bsz, N, L, **f32),
             dC=torch.empty(Bsz, N, L, **f32),
             dD=None if D is None else torch.empty(Dch, **f32),
             ddelta_bias=None if delta_bias is None else torch.empty(Dch, **f32))
    ins = [describe(t) for t in (u, delta, A, B, C, D, z, delta_bias)]
    outs = [describe(g[k]) for k in ("du", "ddelta", "dA", "dB", "dC", "dD", "dz", "ddelta_bias")]
    rc = load().ss_selective_scan_bwd(*[_ref(t) for t in ins], int(bool(softplus)),
                                      _ref(describe(dout)), *[_ref(t) for t in outs],
                                      _stream_ptr(stream))
    if rc != 0:
        raise SSError(rc, "ss_selective_scan_bwd")
    return g


def selective_scan_fwd_ckpt(u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True,
                            y=None, last_state=None, ckpt=None, stream=None):
    """Forward of a training step (ss_selective_scan_fwd_ckpt): y, the final
    state and the state every 8 steps for selective_scan_bwd_ckpt.  Returns
    (y, last_state, ckpt) with ckpt (batch, d_inner, ceil(L / 8), 16) f32."""
    Bsz, Dch, L = u.shape
    if y is None:
        y = torch.empty_like(u, memory_format=torch.contiguous_format)
    if last_state is None:
        last_state = torch.empty(Bsz, Dch, A.shape[1], dtype=torch.float32, device=u.device)
    if ckpt is None:
        ckpt = torch.empty(Bsz, Dch, (L + 7) // 8, 16, dtype=torch.float32, device=u.device)
    ts = [describe(t) for t in (u, delta, A, B, C, D, z, delta_bias)]
    rc = load().ss_selective_scan_fwd_ckpt(*[_ref(t) for t in ts], int(bool(softplus)),
                                           _ref(describe(y)), _ref(describe(last_state)),
                                           _ref(describe(ckpt)), _stream_ptr(stream))
    if rc != 0:
        raise SSError(rc, "ss_selective_scan_fwd_ckpt")
    return y, last_state, ckpt


def selective_scan_bwd_ckpt(u, delta, A, B, C, D, z, delta_bias, dout, ckpt, softplus=True,
                            stream=None):
    """Backward of a training step (ss_selective_scan_bwd_ckpt) from the
    forward's checkpoints; returns the same dict as selective_scan_bwd."""
    f32 = dict(dtype=torch.float32, device=u.device)
    Bsz, Dch, L = u.shape
    N = A.shape[1]
    g = dict(du=torch.empty_like(u, memory_format=torch.contiguous_format),
             ddelta=torch.empty_like(u, memory_format=torch.contiguous_format),
             dz=None if z is None else torch.empty_like(u, memory_format=torch.contiguous_format),
             dA=torch.empty(Dch, N, **f32), dB=torch.empty(Bsz, N, L, **f32),
             dC=torch.empty(Bsz, N, L, **f32),
             dD=None if D is None else torch.empty(Dch, **f32),
             ddelta_bias=None if delta_bias is None else torch.empty(Dch, **f32))
    ins = [describe(t) for t in (u, delta, A, B, C, D, z, delta_bias)]
    outs = [describe(g[k]) for k in ("du", "ddelta", "dA", "dB", "dC", "dD", "dz", "ddelta_bias")]
    rc = load().ss_selective_scan_bwd_ckpt(*[_ref(t) for t in ins], int(bool(softplus)),
                                           _ref(describe(dout)), _ref(describe(ckpt)),
                                           *[_ref(t) for t in outs], _stream_ptr(stream))
    if rc != 0:
        raise SSError(rc, "ss_selective_scan_bwd_ckpt")
    return g


def selective_state_update(state, u, delta, A, B, C, D=None, z=None, delta_bias=None,
                           softplus=True, y=None, stream=None):
    """One decode step (ss_selective_state_update); state (batch, d_inner, N)
    f32 is updated in place.  u, delta, z: (batch, d_inner); B, C: (batch, N)."""
    if y is None:
        y = torch.empty_like(u, memory_format=torch.contiguous_format)
    ts = [describe(t) for t in (u, delta, A, B, C, D, z, delta_bias)]
    rc = load().ss_selective_state_update(_ref(describe(state)), *[_ref(t) for t in ts],
                                          int(bool(softplus)), _ref(describe(y)),
                                          _stream_ptr(stream))
    if rc != 0:
        raise SSError(rc, "ss_selective_state_update")
    return y


def ssd_state_update(state, x, dt, A_head, B, C, D=None, y=None, stream=None):
    """One Mamba-2 decode step (ss_ssd_state_update); state (batch, H, P, N) f32
    is updated in place.  x: (batch, H, P); dt: (batch, H); B, C: (batch, G, N)."""
    if y is None:
        y = torch.empty_like(x, memory_format=torch.contiguous_format)
    ts = [describe(t) for t in (x, dt, A_head, B, C, D)]
    rc = load().ss_ssd_state_update(_ref(describe(state)), *[_ref(t) for t in ts],
                                    _ref(describe(y)), _stream_ptr(stream))
    if rc != 0:
        raise SSError(rc, "ss_ssd_state_update")
    return y


def device_error(stream=None) -> int:
    return int(load().ss_get_device_error(_stream_ptr(stream)))


def selftest_timeout(limit_us=2000, stream=None) -> None:
    """ss_selftest_timeout: a kernel whose bounded wait runs out; afterwards
    device_error() returns the SS_ERR_TIMEOUT code."""
    rc = load().ss_selftest_timeout(int(limit_us), _stream_ptr(stream))
    if rc != 0:
        raise SSError(rc, "ss_selftest_timeout")


def launch_count() -> int:
    return int(load().ss_launch_count())


def set_debug_path(name: str, value: int | None) -> None:
    """ss_debug_set_path: force one kernel choice (value None or -1 restores
    the library's own choice).  Names are the keys of DEBUG."""
    rc = load().ss_debug_set_path(DEBUG[name], -1 if value is None else int(value))
    if rc != 0:
        raise SSError(rc, "ss_debug_set_path")


@contextlib.contextmanager
def debug_paths(**switches):
    """Set diagnostic switches for the duration of a with-block, e.g.
    ``with debug_paths(scan_path=1, scan_split=4): ...``; every switch given
    is restored to the library's own choice afterwards."""
    for k, v in switches.items():
        set_debug_path(k, v)
    try:
        yield
    finally:
        for k in switches:
            set_debug_path(k, None)


def probe_ex2_rate(stream=None) -> float:
    """ss_probe_ex2_rate: measured ex2.approx.f32 operations per SM per clock."""
    v = ctypes.c_double(0.0)
    rc = load().ss_probe_ex2_rate(ctypes.byref(v), _stream_ptr(stream))
    if rc != 0:
        raise SSError(rc, "ss_probe_ex2_rate")
    return float(v.value)


def probe_scan_forms(stream=None) -> tuple[float, float]:
    """ss_probe_scan_forms: channel-steps per second of the sequential and the
    warp-shuffle (associative) scan forms on synthetic tiles."""
    a, b = ctypes.c_double(0.0), ctypes.c_double(0.0)
    rc = load().ss_probe_scan_forms(ctypes.byref(a), ctypes.byref(b), _stream_ptr(stream))
    if rc != 0:
        raise SSError(rc, "ss_probe_scan_forms")
    return float(a.value), float(b.value)
