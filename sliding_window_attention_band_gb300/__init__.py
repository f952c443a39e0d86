"""Sliding-window (banded, "diagonal") attention for one NVIDIA GB300 (sm_103a).

The compute runs in hand-written CUDA kernels behind a C ABI (include/swab.h,
built into ``_lib/libswab.so`` by ``build.build()``); this package is the thin
ctypes binding over it plus the seeded input generators.  Nothing here
computes attention on the host.
"""
from ._binding import (API_FUNCTIONS, Desc, SwabError, add_bias_transpose,  # noqa: F401
                       band_attention,
                       band_attention_bwd, band_attention_bwd_noalloc,
                       band_attention_bwd_workspace, band_attention_dropout_mask_bytes, band_pv,
                       band_pv_bwd_t, band_qk, band_qk_bwd_t, band_softmax, band_softmax_bwd,
                       band_softmax_dropout,
                       device_status, global_attention, global_attention_bwd,
                       global_attention_workspace, library_path, load, selftest_wait_timeout,
                       bounds_checked, bounds_report, selftest_bounds,
                       status_string, version)
from .inputs import WORKLOADS, Workload, seeded_qkvo, workload_inputs  # noqa: F401

__all__ = ["Desc", "SwabError", "add_bias_transpose", "band_qk", "band_softmax",
           "band_softmax_dropout", "band_pv", "band_qk_bwd_t", "global_attention",
           "global_attention_bwd", "global_attention_workspace",
           "band_pv_bwd_t", "band_softmax_bwd", "band_attention", "band_attention_bwd",
           "band_attention_bwd_noalloc",
           "band_attention_bwd_workspace", "band_attention_dropout_mask_bytes", "device_status", "selftest_wait_timeout", "bounds_checked", "bounds_report",
           "selftest_bounds", "load",
           "library_path", "version", "status_string", "WORKLOADS", "Workload",
           "seeded_qkvo", "workload_inputs"]
