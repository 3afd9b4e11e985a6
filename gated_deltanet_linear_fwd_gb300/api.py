"""Python binding of the C ABI (include/gdn.h): argument marshalling only.

Every step of the forward runs in libgdn.so's CUDA kernels; PyTorch only
provides device memory and the stream.  The names mirror the C entry points.
"""
from __future__ import annotations

import ctypes
import dataclasses
from typing import Optional, Sequence

import torch

from . import _lib as L

_MODES = {"off": L.GDN_CP_OFF, "exact": L.GDN_CP_EXACT, "warmup": L.GDN_CP_WARMUP, "auto": L.GDN_CP_AUTO}
_DT = {torch.bfloat16: L.GDN_BF16, torch.float32: L.GDN_F32}
_TOL_RULES = {"fixed": L.GDN_TOL_FIXED, "noise": L.GDN_TOL_NOISE}


@dataclasses.dataclass
class Plan:
    """A filled gdn_cp_plan_t together with the dims it was made for."""
    raw: L.gdn_cp_plan_t
    dims: L.gdn_dims
    cu_seqlens_host: Optional[list]

    @property
    def mode(self) -> str:
        return {v: k for k, v in _MODES.items()}[self.raw.mode]

    @property
    def workspace_bytes(self) -> int:
        return int(self.raw.workspace_bytes)

    @property
    def n_seg_total(self) -> int:
        return int(self.raw.n_seg_total)


def _cu_list(cu_seqlens) -> Optional[list]:
    if cu_seqlens is None:
        return None
    if isinstance(cu_seqlens, torch.Tensor):
        return [int(x) for x in cu_seqlens.tolist()]
    return [int(x) for x in cu_seqlens]


def gdn_cp_plan(*, T: int, h_qk: int, h_v: int, B: int = 1, cu_seqlens=None,
                dtype: torch.dtype = torch.bfloat16, mode: str = "auto", lambda_: float = 0.0,
                warmup_chunks: int = 8, warmup_tol: float = 1e-4, sm_count: int = 0,
                scale: float = 0.0, d_k: int = 128, d_v: int = 128, tol_rule: str = "noise") -> Plan:
    """Host-only planning (gdn_cp_plan).  T = tokens per row (varlen: total).
    tol_rule: "noise" (a warmup's tolerance is at least the exact path's noise
    floor at the segment start) or "fixed" (warmup_tol alone)."""
    cu = _cu_list(cu_seqlens)
    n_seqs = B if cu is None else len(cu) - 1
    dims = L.gdn_dims(B, T, h_qk, h_v, d_k, d_v, n_seqs, scale, _DT.get(dtype, -1))
    opts = L.gdn_cp_opts(_MODES[mode], lambda_, warmup_chunks, warmup_tol, sm_count, _TOL_RULES[tol_rule])
    raw = L.gdn_cp_plan_t()
    cu_arr = None if cu is None else (ctypes.c_int32 * len(cu))(*cu)
    L.check(L.load().gdn_cp_plan(ctypes.byref(dims), cu_arr, ctypes.byref(opts), ctypes.byref(raw)),
            "gdn_cp_plan")
    return Plan(raw, dims, cu)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def gdn_chunk_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor, beta: torch.Tensor,
                  initial_state: Optional[torch.Tensor] = None, cu_seqlens: Optional[torch.Tensor] = None,
                  *, plan: Optional[Plan] = None, out: Optional[torch.Tensor] = None,
                  final_state: Optional[torch.Tensor] = None, output_final_state: bool = True,
                  workspace: Optional[torch.Tensor] = None, stream=None, scale: float = 0.0,
                  mode: str = "auto", lambda_: float = 0.0, warmup_chunks: int = 8,
                  warmup_tol: float = 1e-4, tol_rule: str = "noise", for_backward: bool = False):
    """The chunked-prefill forward (gdn_chunk_fwd).

    q,k [B,T,h_qk,128] or [T,h_qk,128]; v [.., h_v, 128]; g,beta [.., h_v] fp32;
    initial_state [N,h_v,128,128] fp32 or None; cu_seqlens int32 [N+1] on the
    device (varlen, B = 1) or None.  Returns (o, final_state or None).
    for_backward: gdn_chunk_fwd_train -- the workspace (of gdn_bwd_workspace_bytes)
    keeps what gdn_chunk_bwd(..., reuse_forward=True) needs with the same plan.
    """
    batched = q.dim() == 4
    B = q.shape[0] if batched else 1
    T = q.shape[-3]
    h_qk, h_v = q.shape[-2], v.shape[-2]
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if g.dtype != torch.float32 or beta.dtype != torch.float32:
        raise ValueError("g and beta must be float32")
    if plan is None:
        plan = gdn_cp_plan(T=T, h_qk=h_qk, h_v=h_v, B=B, cu_seqlens=cu_seqlens, dtype=q.dtype, mode=mode,
                           lambda_=lambda_, warmup_chunks=warmup_chunks, warmup_tol=warmup_tol, scale=scale,
                           tol_rule=tol_rule)
    dims = L.gdn_dims(B, T, h_qk, h_v, q.shape[-1], v.shape[-1], plan.raw.n_seqs, scale, _DT.get(q.dtype, -1))
    if out is None:
        out = torch.empty_like(v)
    if final_state is None and output_final_state:
        final_state = torch.empty(plan.raw.n_seqs, h_v, 128, 128, dtype=torch.float32, device=q.device)
    if workspace is None:
        n_ws = gdn_bwd_workspace_bytes(plan) if for_backward else plan.workspace_bytes
        workspace = torch.empty(max(n_ws, 256), dtype=torch.uint8, device=q.device)
    if initial_state is not None and (initial_state.dtype != torch.float32 or not initial_state.is_contiguous()):
        raise ValueError("initial_state must be contiguous float32")
    fn = L.load().gdn_chunk_fwd_train if for_backward else L.load().gdn_chunk_fwd
    st = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(initial_state), _ptr(cu_seqlens), _ptr(out),
            _ptr(final_state), ctypes.byref(dims), ctypes.byref(plan.raw), _ptr(workspace), workspace.numel(),
            _stream_handle(stream))
    L.check(st, "gdn_chunk_fwd_train" if for_backward else "gdn_chunk_fwd")
    return out, final_state


def gdn_bwd_workspace_bytes(plan: Plan) -> int:
    """Device workspace bytes gdn_chunk_bwd needs for `plan` (gdn_bwd_workspace_bytes)."""
    n = ctypes.c_size_t(0)
    L.check(L.load().gdn_bwd_workspace_bytes(ctypes.byref(plan.raw), ctypes.byref(n)), "gdn_bwd_workspace_bytes")
    return int(n.value)


def gdn_chunk_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor, beta: torch.Tensor,
                  d_out: torch.Tensor, initial_state: Optional[torch.Tensor] = None,
                  d_final_state: Optional[torch.Tensor] = None, cu_seqlens: Optional[torch.Tensor] = None,
                  *, plan: Optional[Plan] = None, grads=None, workspace: Optional[torch.Tensor] = None,
                  stream=None, scale: float = 0.0, mode: str = "auto", lambda_: float = 0.0,
                  want_initial_state_grad: bool = True, reuse_forward: bool = False):
    """Gradients of sum(o * d_out) + sum(final_state * d_final_state) (gdn_chunk_bwd).

    Inputs as gdn_chunk_fwd (bf16 q/k/v); d_out like v (bf16); d_final_state
    [N, h_v, 128, 128] fp32 or None.  grads: optional preallocated
    (dq, dk, dv, dg, dbeta, dh0).  Returns (dq, dk, dv, dg, dbeta, dh0 or None).
    reuse_forward: `workspace` and `plan` are those of a gdn_chunk_fwd(...,
    for_backward=True) on the same inputs; the forward is not recomputed.
    """
    batched = q.dim() == 4
    B = q.shape[0] if batched else 1
    T = q.shape[-3]
    h_qk, h_v = q.shape[-2], v.shape[-2]
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("d_out", d_out)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if q.dtype != torch.bfloat16 or d_out.dtype != torch.bfloat16:
        raise ValueError("the backward takes bf16 q/k/v and d_out")
    if reuse_forward and (workspace is None or plan is None):
        raise ValueError("reuse_forward needs the plan and workspace of the gdn_chunk_fwd(for_backward=True) call")
    if g.dtype != torch.float32 or beta.dtype != torch.float32:
        raise ValueError("g and beta must be float32")
    for name, t in (("initial_state", initial_state), ("d_final_state", d_final_state)):
        if t is not None and (t.dtype != torch.float32 or not t.is_contiguous()):
            raise ValueError(f"{name} must be contiguous float32")
    if plan is None:
        plan = gdn_cp_plan(T=T, h_qk=h_qk, h_v=h_v, B=B, cu_seqlens=cu_seqlens, dtype=q.dtype, mode=mode,
                           lambda_=lambda_, scale=scale)
    dims = L.gdn_dims(B, T, h_qk, h_v, q.shape[-1], v.shape[-1], plan.raw.n_seqs, scale, _DT.get(q.dtype, -1))
    if grads is None:
        dh0 = (torch.empty(plan.raw.n_seqs, h_v, 128, 128, dtype=torch.float32, device=q.device)
               if want_initial_state_grad else None)
        grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), torch.empty_like(g),
                 torch.empty_like(beta), dh0)
    dq, dk, dv, dg, dbeta, dh0 = grads
    if workspace is None:
        workspace = torch.empty(max(gdn_bwd_workspace_bytes(plan), 256), dtype=torch.uint8, device=q.device)
    st = L.load().gdn_chunk_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(initial_state),
                                _ptr(cu_seqlens), _ptr(d_out), _ptr(d_final_state), _ptr(dq), _ptr(dk), _ptr(dv),
                                _ptr(dg), _ptr(dbeta), _ptr(dh0), ctypes.byref(dims), ctypes.byref(plan.raw),
                                _ptr(workspace), workspace.numel(), int(bool(reuse_forward)),
                                _stream_handle(stream))
    L.check(st, "gdn_chunk_bwd")
    return dq, dk, dv, dg, dbeta, dh0


def gdn_decode_step(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor, beta: torch.Tensor,
                    state: torch.Tensor, *, out: Optional[torch.Tensor] = None, scale: float = 0.0, stream=None):
    """One new token per sequence (gdn_decode_step): q,k [B,h_qk,128], v [B,h_v,128]
    (bf16 or fp32), g,beta [B,h_v] fp32, state [B,h_v,128,128] fp32 (H = S^T,
    updated in place).  Returns o [B,h_v,128]."""
    B, h_qk, h_v = q.shape[0], q.shape[1], v.shape[1]
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("state", state)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if g.dtype != torch.float32 or beta.dtype != torch.float32 or state.dtype != torch.float32:
        raise ValueError("g, beta and state must be float32")
    if out is None:
        out = torch.empty_like(v)
    dims = L.gdn_dims(B, 1, h_qk, h_v, q.shape[-1], v.shape[-1], B, scale, _DT.get(q.dtype, -1))
    st = L.load().gdn_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state), _ptr(out),
                                  ctypes.byref(dims), _stream_handle(stream))
    L.check(st, "gdn_decode_step")
    return out


def gdn_get_device_status(workspace: torch.Tensor, stream=None):
    """(code, detail) of the status word of the last call on this workspace (synchronises)."""
    code, detail = ctypes.c_int(), ctypes.c_int()
    L.check(L.load().gdn_get_device_status(_ptr(workspace), _stream_handle(stream), ctypes.byref(code),
                                           ctypes.byref(detail)), "gdn_get_device_status")
    return code.value, detail.value


_DETAILS = {1: "a bulk copy's wait", 2: "an MMA's wait", 3: "the chunk index or segments disagree with the plan",
            4: "segments combined out of order", 5: "a value outside the fp16 range of the MMA operands",
            6: "the test hook's stall"}


def describe_device_status(code: int, detail: int) -> str:
    """Text for a (code, detail) pair read from the status word: code is a
    gdn_status (0, 5 timeout or 7 check); detail says which check or wait
    tripped (100 + b: a bounded wait on mbarrier b of the kernel)."""
    if code == L.GDN_OK:
        return "ok"
    what = {L.GDN_ERR_DEVICE_TIMEOUT: "timeout", L.GDN_ERR_DEVICE_CHECK: "check failed"}.get(code, f"code {code}")
    if detail >= 100:
        where = f"the bounded wait on barrier {detail - 100}"
    else:
        where = _DETAILS.get(detail, f"detail {detail}")
    return f"{what}: {where}"


def gdn_debug_stall_ns(ns: int) -> None:
    """Test hook (gdn_debug_stall_ns): while ns > 0 every later forward's
    chunk-local kernel waits ns nanoseconds on a barrier nothing arrives on,
    so the call takes its timeout path; 0 turns it off."""
    L.check(L.load().gdn_debug_stall_ns(int(ns)), "gdn_debug_stall_ns")


def gdn_get_static_device_status(stream=None):
    """(code, detail) of the status word of the last gdn_chunk_fwd_static call
    on the current device (synchronises)."""
    code, detail = ctypes.c_int(), ctypes.c_int()
    L.check(L.load().gdn_get_static_device_status(_stream_handle(stream), ctypes.byref(code), ctypes.byref(detail)),
            "gdn_get_static_device_status")
    return code.value, detail.value


def gdn_cp_head_modes(workspace: torch.Tensor, plan: Plan, stream=None):
    """Per (sequence, head): the mode taken (1 exact, 2 warmup, 0 off) and log warmup bound."""
    n = plan.raw.n_seqs * plan.raw.h_v
    modes = (ctypes.c_int32 * n)()
    bounds = (ctypes.c_float * n)()
    L.check(L.load().gdn_cp_head_modes(_ptr(workspace), ctypes.byref(plan.raw), modes, bounds,
                                       _stream_handle(stream)), "gdn_cp_head_modes")
    shape = (plan.raw.n_seqs, plan.raw.h_v)
    return (torch.tensor(list(modes), dtype=torch.int32).reshape(shape),
            torch.tensor(list(bounds), dtype=torch.float32).reshape(shape))


def gdn_set_trace_events(events) -> None:
    """Register torch.cuda.Event objects (enable_timing=True, recorded once so
    they exist) for per-kernel timing of this thread's next gdn_chunk_fwd
    calls; [] turns it off."""
    n = len(events)
    arr = (ctypes.c_void_p * max(n, 1))(*[ctypes.c_void_p(e.cuda_event) for e in events])
    L.check(L.load().gdn_set_trace_events(arr if n else None, n), "gdn_set_trace_events")


def gdn_trace_last() -> list:
    """Names of the kernels the last gdn_chunk_fwd on this thread launched."""
    names = (ctypes.c_char_p * 16)()
    n = L.load().gdn_trace_last(names, 16)
    return [names[i].decode() for i in range(n)]


def gdn_chunk_fwd_static(q, k, v, g, beta, initial_state=None, cu_seqlens=None, *, plan: Plan, out, final_state=None,
                         stream=None):
    """gdn_chunk_fwd_static: the forward with the library's built-in 8 MiB
    device workspace, for callers that cannot allocate device memory.  The
    caller passes every input and output (nothing is allocated here)."""
    dims = L.gdn_dims(q.shape[0] if q.dim() == 4 else 1, q.shape[-3], q.shape[-2], v.shape[-2], q.shape[-1],
                      v.shape[-1], plan.raw.n_seqs, 0.0, _DT.get(q.dtype, -1))
    st = L.load().gdn_chunk_fwd_static(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(initial_state),
                                       _ptr(cu_seqlens), _ptr(out), _ptr(final_state), ctypes.byref(dims),
                                       ctypes.byref(plan.raw), _stream_handle(stream))
    L.check(st, "gdn_chunk_fwd_static")
    return out, final_state
