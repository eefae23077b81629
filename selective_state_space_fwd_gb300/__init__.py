"""selective_state_space_fwd_gb300 -- the fused selective-scan forward on GB300.

The compute lives in ``libssmscan.so`` (C ABI, include/ssmscan.h, hand-written
sm_103a kernels under csrc/).  This package is its Python binding plus the
seeded synthetic workloads used by the benchmark and tests.
"""
from ._binding import (Kernel, SsmError, Status, check_device_errors, chunk_count,
                       decode_step, declared_functions,
                       host_workspace_bytes, kernel_name, load, plan, scan_bwd, scan_fwd, scan_fwd_host,
                       scan_fwd_host_static, scan_fwd_split, selftest_wait_timeout, split_plan,
                       ssd_fwd, static_capacity,
                       status_string, version)
from .autograd import selective_scan

__all__ = ["Kernel", "SsmError", "Status", "check_device_errors", "chunk_count", "decode_step",
           "declared_functions",
           "host_workspace_bytes", "kernel_name", "load", "plan", "scan_bwd", "scan_fwd",
           "scan_fwd_host", "scan_fwd_host_static", "scan_fwd_split", "selftest_wait_timeout",
           "selective_scan", "split_plan", "ssd_fwd",
           "static_capacity",
           "status_string", "version"]
