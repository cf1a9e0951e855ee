"""B300-native Mamba selective scan and Mamba-2 SSD scan.

The compute lives in ``libssscan.so`` (hand-written sm_103a CUDA behind the C
ABI declared in ``include/ssscan.h``); this package only binds it.

    from selective_state_space_146_b300 import selective_scan_fwd, ssd_chunk_scan_fwd
"""
from ._abi import (SSError, conv_selective_scan_fwd, device_error,  # noqa: F401
                   launch_count, selective_scan_bwd, selective_scan_bwd_ckpt,
                   selective_scan_fwd, selective_scan_fwd_ckpt, selective_scan_fwd_host,
                   selective_scan_fwd_noalloc, selective_state_update, ssd_chunk_scan_fwd,
                   ssd_state_update, status_string)

__all__ = ["selective_scan_fwd", "selective_scan_fwd_host", "conv_selective_scan_fwd", "selective_scan_fwd_noalloc",
           "ssd_chunk_scan_fwd", "selective_scan_bwd", "selective_scan_fwd_ckpt",
           "selective_scan_bwd_ckpt",
           "selective_state_update", "ssd_state_update", "SSError", "device_error",
           "launch_count", "status_string"]
