"""ctypes view of libgdn.so, the C ABI declared in include/gdn.h.

Loading fails loudly when the library has not been built: there is no other
implementation behind these names.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgdn.so")

GDN_OK = 0
GDN_ERR_INVALID_ARG = 1
GDN_ERR_UNSUPPORTED = 2
GDN_ERR_MISALIGNED = 3
GDN_ERR_CUDA = 4
GDN_ERR_DEVICE_TIMEOUT = 5
GDN_ERR_WORKSPACE = 6
GDN_ERR_DEVICE_CHECK = 7

GDN_BF16 = 0
GDN_F32 = 1
GDN_TOL_FIXED = 0
GDN_TOL_NOISE = 1

GDN_CP_OFF = 0
GDN_CP_EXACT = 1
GDN_CP_WARMUP = 2
GDN_CP_AUTO = 3

EXPORTED = ["gdn_cp_plan", "gdn_chunk_fwd", "gdn_status_string", "gdn_last_cuda_error",
            "gdn_get_device_status", "gdn_cp_head_modes", "gdn_set_trace_events", "gdn_trace_last", "gdn_chunk_fwd_static",
            "gdn_get_static_device_status", "gdn_decode_step", "gdn_debug_stall_ns", "gdn_bwd_workspace_bytes",
            "gdn_chunk_bwd", "gdn_chunk_fwd_train"]


class gdn_dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("h_qk", ctypes.c_int), ("h_v", ctypes.c_int),
                ("d_k", ctypes.c_int), ("d_v", ctypes.c_int), ("n_seqs", ctypes.c_int),
                ("scale", ctypes.c_float), ("dtype", ctypes.c_int)]


class gdn_cp_opts(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int), ("lambda_", ctypes.c_float), ("warmup_chunks", ctypes.c_int),
                ("warmup_tol", ctypes.c_float), ("sm_count", ctypes.c_int), ("tol_rule", ctypes.c_int)]


class gdn_cp_plan_t(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int), ("n_seqs", ctypes.c_int), ("T_total", ctypes.c_int),
                ("h_v", ctypes.c_int), ("h_qk", ctypes.c_int), ("dtype", ctypes.c_int),
                ("lambda_q8", ctypes.c_int), ("warmup_chunks", ctypes.c_int),
                ("warmup_tol", ctypes.c_float), ("sm_count", ctypes.c_int), ("tol_rule", ctypes.c_int),
                ("n_seg_total", ctypes.c_int), ("max_seg_chunks", ctypes.c_int),
                ("max_chunks", ctypes.c_int), ("workspace_bytes", ctypes.c_size_t),
                ("off_head", ctypes.c_size_t), ("off_seg_bound", ctypes.c_size_t),
                ("off_R", ctypes.c_size_t), ("off_Sloc", ctypes.c_size_t), ("off_Sstart", ctypes.c_size_t),
                ("n_chunks_total", ctypes.c_int), ("off_chunk_map", ctypes.c_size_t),
                ("off_wy", ctypes.c_size_t)]


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH):
    """Load libgdn.so (built in-tree by gated_deltanet_linear_fwd_gb300.build)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"libgdn.so not found at {path}: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` (nvcc, sm_103a)")
        lib = ctypes.CDLL(path)
        vp, i32p, fp = ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_float)
        lib.gdn_cp_plan.argtypes = [ctypes.POINTER(gdn_dims), i32p, ctypes.POINTER(gdn_cp_opts),
                                    ctypes.POINTER(gdn_cp_plan_t)]
        lib.gdn_cp_plan.restype = ctypes.c_int
        lib.gdn_chunk_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.POINTER(gdn_dims),
                                      ctypes.POINTER(gdn_cp_plan_t), vp, ctypes.c_size_t, vp]
        lib.gdn_chunk_fwd.restype = ctypes.c_int
        lib.gdn_status_string.argtypes = [ctypes.c_int]
        lib.gdn_status_string.restype = ctypes.c_char_p
        lib.gdn_last_cuda_error.argtypes = []
        lib.gdn_last_cuda_error.restype = ctypes.c_int
        lib.gdn_get_device_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]
        lib.gdn_get_device_status.restype = ctypes.c_int
        lib.gdn_cp_head_modes.argtypes = [vp, ctypes.POINTER(gdn_cp_plan_t), i32p, fp, vp]
        lib.gdn_cp_head_modes.restype = ctypes.c_int
        lib.gdn_chunk_fwd_static.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.POINTER(gdn_dims),
                                             ctypes.POINTER(gdn_cp_plan_t), vp]
        lib.gdn_chunk_fwd_static.restype = ctypes.c_int
        lib.gdn_get_static_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]
        lib.gdn_get_static_device_status.restype = ctypes.c_int
        lib.gdn_decode_step.argtypes = [vp, vp, vp, vp, vp, vp, vp, ctypes.POINTER(gdn_dims), vp]
        lib.gdn_decode_step.restype = ctypes.c_int
        lib.gdn_set_trace_events.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_int]
        lib.gdn_set_trace_events.restype = ctypes.c_int
        lib.gdn_trace_last.argtypes = [ctypes.POINTER(ctypes.c_char_p), ctypes.c_int]
        lib.gdn_trace_last.restype = ctypes.c_int
        lib.gdn_bwd_workspace_bytes.argtypes = [ctypes.POINTER(gdn_cp_plan_t), ctypes.POINTER(ctypes.c_size_t)]
        lib.gdn_bwd_workspace_bytes.restype = ctypes.c_int
        lib.gdn_chunk_bwd.argtypes = [vp] * 15 + [ctypes.POINTER(gdn_dims), ctypes.POINTER(gdn_cp_plan_t), vp,
                                                  ctypes.c_size_t, ctypes.c_int, vp]
        lib.gdn_chunk_fwd_train.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.POINTER(gdn_dims),
                                            ctypes.POINTER(gdn_cp_plan_t), vp, ctypes.c_size_t, vp]
        lib.gdn_chunk_fwd_train.restype = ctypes.c_int
        lib.gdn_chunk_bwd.restype = ctypes.c_int
        lib.gdn_debug_stall_ns.argtypes = [ctypes.c_uint32]
        lib.gdn_debug_stall_ns.restype = ctypes.c_int
        _lib = lib
        return lib


class GDNError(RuntimeError):
    def __init__(self, status: int, where: str):
        lib = load()
        msg = lib.gdn_status_string(status).decode()
        if status == GDN_ERR_CUDA:
            msg += f" (cuda error {lib.gdn_last_cuda_error()})"
        super().__init__(f"{where}: {msg}")
        self.status = status


def check(status: int, where: str):
    if status != GDN_OK:
        raise GDNError(status, where)
