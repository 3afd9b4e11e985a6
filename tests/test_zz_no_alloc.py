"""The forward without a caller workspace (gdn_chunk_fwd_static).

Some callers cannot allocate device memory: a runtime that owns all of it
(an inference server's arena, a plugin interface that passes only inputs and
outputs) or code that must not allocate once it is running.  For them the
library has an entry point that uses its own fixed 8 MiB device array as the
workspace.  These tests call it through the C ABI and check it against
gdn_chunk_fwd, which takes a caller workspace: both run the same
deterministic kernels on the same inputs, so o and the final state must be
bitwise equal.  The array keeps the previous call's contents, so the calls
come in a row with a larger plan first (stale data left behind in the array
would show).  They also check that a plan needing more than the array is
refused, and that the kernels' status word of these calls can be read.
The file name makes pytest collect it last.
"""
from __future__ import annotations

import ctypes
import dataclasses

import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU, skipped there
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from gated_deltanet_linear_fwd_gb300 import _lib as L  # noqa: E402
from gated_deltanet_linear_fwd_gb300 import (gdn_chunk_fwd, gdn_chunk_fwd_static, gdn_cp_plan,  # noqa: E402
                                             gdn_get_static_device_status)
from gated_deltanet_linear_fwd_gb300.inputs import make_inputs, workload  # noqa: E402

DEV = "cuda:0"
STATIC_BYTES = 8 << 20


def _static_call(d, plan, out, hT):
    """gdn_chunk_fwd_static through the C ABI with caller-allocated outputs."""
    dims = L.gdn_dims(1, d.T, d.h_qk, d.h_v, 128, 128, plan.raw.n_seqs, 0.0, L.GDN_BF16)
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    return L.load().gdn_chunk_fwd_static(p(d.q), p(d.k), p(d.v), p(d.g), p(d.beta), p(d.h0), p(d.cu_seqlens),
                                         p(out), p(hT), ctypes.byref(dims), ctypes.byref(plan.raw),
                                         ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _nan_outputs(w, d):
    return (torch.full_like(d.v, float("nan")),
            torch.full((w.n_seqs, w.h_v, 128, 128), float("nan"), device=DEV))


CASES = [  # the largest in-limit plan first, then smaller ones with other shapes and modes
    ("big", lambda: make_inputs(cu_seqlens=[0, 1500, 2600], h_qk=2, h_v=4, seed=21, with_h0=True), "off", 0.0),
    ("exact", lambda: make_inputs(700, h_qk=2, h_v=4, seed=22, with_h0=True), "exact", 0.5),
    ("tiny", lambda: workload("tiny_T512_h2x4"), "auto", 0.0),
    ("ragged", lambda: make_inputs(cu_seqlens=[0, 1, 65, 200, 200, 391, 1000], h_qk=2, h_v=6, seed=7,
                                   with_h0=True), "off", 0.0),
]


def test_static_workspace_matches_caller_workspace_in_a_row():
    sizes = []
    for i, (tag, make, mode, lam) in enumerate(CASES):
        w = make()
        d = w.to(DEV)
        plan = gdn_cp_plan(T=w.T, h_qk=w.h_qk, h_v=w.h_v, cu_seqlens=w.cu_seqlens, mode=mode, lambda_=lam)
        assert plan.workspace_bytes <= STATIC_BYTES, tag
        sizes.append(plan.workspace_bytes)
        o_ref, h_ref = gdn_chunk_fwd(d.q, d.k, d.v, d.g, d.beta, d.h0, d.cu_seqlens, plan=plan)
        out, hT = _nan_outputs(w, d)
        if i == 1:  # one case through the Python wrapper of the same entry point
            gdn_chunk_fwd_static(d.q, d.k, d.v, d.g, d.beta, d.h0, d.cu_seqlens, plan=plan, out=out,
                                 final_state=hT)
        else:
            assert _static_call(d, plan, out, hT) == L.GDN_OK, tag
        assert gdn_get_static_device_status() == (0, 0), tag
        assert torch.equal(out, o_ref), tag
        assert torch.equal(hT, h_ref), tag
    assert sizes[0] > max(sizes[1:])  # the first plan really did leave more behind in the array


def test_static_workspace_reports_device_checks():
    """The kernels' own checks reach the caller: values past the fp16 operand
    range report status 7 (detail 5) through gdn_get_static_device_status,
    and the next ordinary call reads clean."""
    w = make_inputs(700, h_qk=2, h_v=4, seed=3)
    bad = dataclasses.replace(w, v=(w.v.float() * 1e6).to(torch.bfloat16))
    for inputs, expect in ((bad, (7, 5)), (w, (0, 0))):
        d = inputs.to(DEV)
        plan = gdn_cp_plan(T=w.T, h_qk=w.h_qk, h_v=w.h_v, mode="exact", lambda_=0.5)
        out, hT = _nan_outputs(w, d)
        assert _static_call(d, plan, out, hT) == L.GDN_OK
        assert gdn_get_static_device_status() == expect


def test_static_workspace_refuses_plans_above_its_size():
    w = make_inputs(32768, h_qk=2, h_v=8, seed=1)
    plan = gdn_cp_plan(T=w.T, h_qk=w.h_qk, h_v=w.h_v, mode="exact")
    assert plan.workspace_bytes > STATIC_BYTES
    d = w.to(DEV)
    out = torch.empty_like(d.v)
    assert _static_call(d, plan, out, None) == L.GDN_ERR_WORKSPACE
