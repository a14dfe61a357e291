"""Chunkwise-parallel causal linear attention for GB300 (sm_103a).

The computation runs in the CUDA library built from ``csrc/`` (C ABI in
``include/la_gb300.h``); this package is its Python binding (``api``), the
build step (``build``) and the seeded synthetic workloads (``workloads``).
"""
from .api import (LAError, la_chunk_fwd, la_chunk_fwd_kernel_count, la_chunk_fwd_workspace_bytes,
                  la_decode_step,
                  la_device_status, la_get_feature_map, la_last_error, la_selftest_wait_timeout,
                  la_set_feature_map)

__all__ = ["LAError", "la_chunk_fwd", "la_chunk_fwd_kernel_count", "la_chunk_fwd_workspace_bytes", "la_decode_step",
           "la_device_status", "la_get_feature_map", "la_last_error", "la_selftest_wait_timeout",
           "la_set_feature_map"]
