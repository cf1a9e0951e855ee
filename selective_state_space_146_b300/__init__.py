"""B300-native Mamba selective scan and Mamba-2 SSD scan.

The compute lives in ``libssscan.so`` (hand-written sm_103a CUDA behind the C
ABI declared in ``include/ssscan.h``); this package only binds it, and every
call raises ``SSError`` with the library's status if the call is refused.
Tensors are torch tensors on the GPU unless a call says otherwise; layouts:

* selective scan: u, delta, z, y (batch, d_inner, L); A (d_inner, N) f32;
  B, C (batch, N, L), or (batch, G, N, L) with one B, C per group of
  d_inner / G channels; D, delta_bias (d_inner,) f32; states (batch,
  d_inner, N) f32.
* SSD: x, y (batch, L, heads, headdim); dt (batch, L, heads), positive;
  A_head, D (heads,) f32; B, C (batch, L, groups, N); states (batch, heads,
  headdim, N) f32.

Calls:

* ``selective_scan_fwd`` -- y (and the final state), optionally from an
  initial state; ``selective_scan_fwd_noalloc`` -- the same without any
  device allocation during the call; ``selective_scan_fwd_host`` -- pinned
  host tensors in and out, copies overlapped with the scan.
* ``conv_selective_scan_fwd`` -- causal depthwise conv (width <= 4) and SiLU
  fused in front of the scan.
* ``selective_scan_bwd`` -- all eight gradients for an incoming dy;
  ``selective_scan_fwd_ckpt`` / ``selective_scan_bwd_ckpt`` -- a training
  step's pair, the forward keeping the state every 8 steps for the backward.
* ``ssd_chunk_scan_fwd`` -- the Mamba-2 SSD scan in chunked form;
  ``ssd_chunk_scan_fwd_host`` -- the same with pinned host tensors in and out.
* ``selective_state_update`` / ``ssd_state_update`` -- one decoding step,
  the state updated in place.
* ``device_error`` -- the device error word (a bounded wait that ran out);
  ``launch_count`` -- kernels launched so far; ``status_string``.
"""
from ._abi import (SSError, conv_selective_scan_fwd, device_error,  # noqa: F401
                   launch_count, selective_scan_bwd, selective_scan_bwd_ckpt,
                   selective_scan_fwd, selective_scan_fwd_ckpt, selective_scan_fwd_host,
                   selective_scan_fwd_noalloc, selective_state_update, ssd_chunk_scan_fwd,
                   ssd_chunk_scan_fwd_host, ssd_state_update, status_string)

__all__ = ["selective_scan_fwd", "selective_scan_fwd_host", "conv_selective_scan_fwd", "selective_scan_fwd_noalloc",
           "ssd_chunk_scan_fwd", "ssd_chunk_scan_fwd_host", "selective_scan_bwd", "selective_scan_fwd_ckpt",
           "selective_scan_bwd_ckpt",
           "selective_state_update", "ssd_state_update", "SSError", "device_error",
           "launch_count", "status_string"]
