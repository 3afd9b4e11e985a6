"""GB300 (sm_103a) Gated Delta Network chunked-prefill forward and its backward.

The compute lives in libgdn.so (C ABI in include/gdn.h); this package is its
thin Python binding plus the seeded input generators.
"""
from .api import (Plan, describe_device_status, gdn_bwd_workspace_bytes, gdn_chunk_bwd, gdn_chunk_fwd, gdn_debug_stall_ns, gdn_chunk_fwd_static, gdn_cp_head_modes, gdn_cp_plan, gdn_decode_step,
                  gdn_get_device_status, gdn_get_static_device_status, gdn_set_trace_events, gdn_trace_last)

__all__ = ["Plan", "describe_device_status", "gdn_bwd_workspace_bytes", "gdn_chunk_bwd", "gdn_chunk_fwd", "gdn_debug_stall_ns", "gdn_chunk_fwd_static", "gdn_cp_head_modes", "gdn_cp_plan", "gdn_decode_step",
           "gdn_get_device_status", "gdn_get_static_device_status", "gdn_set_trace_events", "gdn_trace_last"]
