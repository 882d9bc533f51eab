"""B300-native selective-scan (Mamba) and SSD (Mamba-2) forward passes.

The compute lives in libssmscan.so (CUDA for sm_103a, C ABI in include/ssmscan.h); this
package holds its build script, a ctypes binding and the seeded input generators.
"""
from .binding import (SSMError, ScanCall, causal_conv1d_fwd, check_status, load_library, new_workspace,
                      ssd_chunk_scan_fwd, ssm_scan_fwd, ssm_scan_fwd_host)

__all__ = ["SSMError", "ScanCall", "load_library", "ssm_scan_fwd", "ssd_chunk_scan_fwd", "ssm_scan_fwd_host",
           "causal_conv1d_fwd", "check_status", "new_workspace"]
