"""The forward without a caller workspace (gdn_chunk_fwd_static).

Some callers cannot allocate device memory: a runtime that owns all of it
(an inference server's arena, a plugin interface that passes only inputs and
outputs) or code that must not allocate once it is running.  For them the
library has an entry point that uses its own fixed 8 MiB device array as the
workspace.  These tests call it through the C ABI and check it against
gdn_chunk_fwd, which takes a caller workspace, on two calls in a row (the
array keeps the previous call's contents, so the second call would show any
stale state), and check that a plan needing more than the array is refused.
The file name makes pytest collect it last.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

from tests import util

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU, skipped there
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from gated_deltanet_linear_fwd_gb300 import _lib as L  # noqa: E402
from gated_deltanet_linear_fwd_gb300 import gdn_chunk_fwd, gdn_cp_plan  # noqa: E402
from gated_deltanet_linear_fwd_gb300.inputs import make_inputs, workload  # noqa: E402

DEV = "cuda:0"


def _static_call(d, plan, out, hT):
    """gdn_chunk_fwd_static through the C ABI with caller-allocated outputs."""
    dims = L.gdn_dims(1, d.T, d.h_qk, d.h_v, 128, 128, plan.raw.n_seqs, 0.0, L.GDN_BF16)
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    st = L.load().gdn_chunk_fwd_static(p(d.q), p(d.k), p(d.v), p(d.g), p(d.beta), p(d.h0), p(d.cu_seqlens),
                                       p(out), p(hT), ctypes.byref(dims), ctypes.byref(plan.raw),
                                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st


def _agree(a, b, tol):
    """max |a - b| beyond one bf16 ulp, relative to RMS(b)."""
    a, b = util.to64(a), util.to64(b)
    ulp = 2 * util.bf16_half_ulp(np.maximum(np.abs(a), np.abs(b)))
    return np.maximum(np.abs(a - b) - ulp, 0).max() <= tol * np.sqrt(np.mean(b ** 2))


def test_static_workspace_matches_caller_workspace_twice():
    cases = [(workload("tiny_T512_h2x4"), "auto"),
             (make_inputs(cu_seqlens=[0, 1, 65, 200, 200, 391, 1000], h_qk=2, h_v=6, seed=7, with_h0=True), "off")]
    for w, mode in cases:  # two calls in a row, different shapes and modes
        d = w.to(DEV)
        plan = gdn_cp_plan(T=w.T, h_qk=w.h_qk, h_v=w.h_v, cu_seqlens=w.cu_seqlens, mode=mode)
        assert plan.workspace_bytes <= 8 << 20
        o_ref, h_ref = gdn_chunk_fwd(d.q, d.k, d.v, d.g, d.beta, d.h0, d.cu_seqlens, plan=plan)
        out = torch.full_like(d.v, float("nan"))
        hT = torch.full((w.n_seqs, w.h_v, 128, 128), float("nan"), device=DEV)
        assert _static_call(d, plan, out, hT) == L.GDN_OK
        torch.cuda.synchronize()
        assert _agree(out, o_ref, util.TOL_BF16)
        assert util.parity_f32(hT, util.to64(h_ref)) <= util.TOL_STATE


def test_static_workspace_refuses_plans_above_its_size():
    w = make_inputs(32768, h_qk=2, h_v=8, seed=1)
    plan = gdn_cp_plan(T=w.T, h_qk=w.h_qk, h_v=w.h_v, mode="exact")
    assert plan.workspace_bytes > 8 << 20
    d = w.to(DEV)
    out = torch.empty_like(d.v)
    assert _static_call(d, plan, out, None) == L.GDN_ERR_WORKSPACE
