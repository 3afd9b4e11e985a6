"""The device status word: values outside the fp16 range of the MMA
operands are reported (status 7, detail 5) rather than silently rounded to
inf, ordinary inputs report nothing, and a bounded wait that runs out (the
test hook's wait on a barrier nothing arrives on) ends the call through its
timeout path (status 5) without disturbing the next call."""
from __future__ import annotations

import dataclasses

import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU, skipped there
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle  # noqa: E402
from gated_deltanet_linear_fwd_gb300 import (describe_device_status, gdn_chunk_fwd, gdn_cp_plan,  # noqa: E402
                                             gdn_debug_stall_ns, gdn_get_device_status)
from tests import util  # noqa: E402
from gated_deltanet_linear_fwd_gb300.inputs import make_inputs  # noqa: E402

DEVICE_CHECK, FP16_RANGE = 7, 5


def _status(w, mode="exact"):
    d = w.to("cuda:0")
    plan = gdn_cp_plan(T=w.T, h_qk=w.h_qk, h_v=w.h_v, cu_seqlens=w.cu_seqlens, mode=mode, lambda_=0.5)
    ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device="cuda:0")
    gdn_chunk_fwd(d.q, d.k, d.v, d.g, d.beta, d.h0, d.cu_seqlens, plan=plan, workspace=ws)
    return gdn_get_device_status(ws)


@pytest.mark.parametrize("mode", ["off", "exact"])
def test_ordinary_inputs_report_nothing(mode):
    assert _status(make_inputs(700, h_qk=2, h_v=4, seed=3, with_h0=True), mode) == (0, 0)


@pytest.mark.parametrize("mode", ["off", "exact"])
def test_values_past_fp16_range_are_reported(mode):
    w = make_inputs(700, h_qk=2, h_v=4, seed=3)
    w = dataclasses.replace(w, v=(w.v.float() * 1e6).to(torch.bfloat16))  # U = A diag(beta) V far beyond 65504
    assert _status(w, mode) == (DEVICE_CHECK, FP16_RANGE)


def test_state_past_fp16_range_is_reported():
    w = make_inputs(700, h_qk=2, h_v=4, seed=3, with_h0=True, g_kind="zero")
    w = dataclasses.replace(w, h0=w.h0 * 1e7)  # the state's fp16 operand copy overflows
    assert _status(w, "off") == (DEVICE_CHECK, FP16_RANGE)


@pytest.mark.parametrize("mode", ["off", "exact"])
def test_query_past_fp16_range_is_reported(mode):
    w = make_inputs(700, h_qk=2, h_v=4, seed=3)
    w = dataclasses.replace(w, q=(w.q.float() * 1e6).to(torch.bfloat16))  # q itself has no fp16 image
    assert _status(w, mode) == (DEVICE_CHECK, FP16_RANGE)


@pytest.mark.parametrize("mode", ["off", "exact"])
def test_timeout_path_reports_and_the_next_call_is_clean(mode):
    """The chunk-local kernel's blocks wait on an mbarrier nothing arrives on,
    20 us at most: the wait runs out, the status word reads (5, 6), the
    kernels after it do no work (o and the final state stay NaN), and the next
    ordinary call on the same workspace matches the oracle."""
    w = make_inputs(700, h_qk=2, h_v=4, seed=3, with_h0=True)
    d = w.to("cuda:0")
    plan = gdn_cp_plan(T=w.T, h_qk=w.h_qk, h_v=w.h_v, mode=mode, lambda_=0.5)
    ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device="cuda:0")
    out = torch.full_like(d.v, float("nan"))
    hT = torch.full((1, w.h_v, 128, 128), float("nan"), device="cuda:0")
    try:
        gdn_debug_stall_ns(20000)
        gdn_chunk_fwd(d.q, d.k, d.v, d.g, d.beta, d.h0, plan=plan, out=out, final_state=hT, workspace=ws)
        status = gdn_get_device_status(ws)
    finally:
        gdn_debug_stall_ns(0)
    assert status == (5, 6), describe_device_status(*status)
    assert torch.isnan(out).all() and torch.isnan(hT).all()
    o, h = gdn_chunk_fwd(d.q, d.k, d.v, d.g, d.beta, d.h0, plan=plan, workspace=ws)
    assert gdn_get_device_status(ws) == (0, 0)
    f = util.to64
    ro, rh = oracle.recurrence(f(w.q), f(w.k), f(w.v), f(w.g), f(w.beta), f(w.h0))
    assert util.parity_bf16(o, ro)[0] <= util.TOL_BF16 and util.parity_f32(h, rh) <= util.TOL_STATE


def test_bwd_values_past_fp16_range_are_reported():
    """An upstream gradient far beyond the fp16 range of the backward's operands."""
    from gated_deltanet_linear_fwd_gb300 import gdn_bwd_workspace_bytes, gdn_chunk_bwd
    w = make_inputs(300, h_qk=1, h_v=2, seed=5, with_h0=True)
    d = w.to("cuda:0")
    plan = gdn_cp_plan(T=w.T, h_qk=w.h_qk, h_v=w.h_v, mode="off")
    ws = torch.empty(gdn_bwd_workspace_bytes(plan), dtype=torch.uint8, device="cuda:0")
    d_out = (torch.randn(w.v.shape, generator=torch.Generator().manual_seed(6)) * 1e6).to(torch.bfloat16)
    gdn_chunk_bwd(d.q, d.k, d.v, d.g, d.beta, d_out.to("cuda:0"), d.h0, None, plan=plan, workspace=ws)
    assert gdn_get_device_status(ws) == (DEVICE_CHECK, FP16_RANGE)


@pytest.mark.parametrize("mode", ["off", "exact"])
def test_bwd_timeout_path_reports_and_the_next_call_is_clean(mode):
    """The backward's recompute meets the same hook: the status reads (5, 6), the
    backward's kernels do no work (the gradients stay NaN), and the next ordinary
    backward on the same workspace gives the same gradients as a fresh one."""
    from gated_deltanet_linear_fwd_gb300 import gdn_bwd_workspace_bytes, gdn_chunk_bwd
    from gated_deltanet_linear_fwd_gb300.inputs import make_output_grads
    w = make_inputs(700, h_qk=2, h_v=4, seed=7, with_h0=True)
    d = w.to("cuda:0")
    d_out, dhT = (x.to("cuda:0") for x in make_output_grads(w, seed=8))
    plan = gdn_cp_plan(T=w.T, h_qk=w.h_qk, h_v=w.h_v, mode=mode, lambda_=0.5)
    ws = torch.empty(gdn_bwd_workspace_bytes(plan), dtype=torch.uint8, device="cuda:0")
    nan = float("nan")
    grads = (torch.full_like(d.q, nan), torch.full_like(d.k, nan), torch.full_like(d.v, nan),
             torch.full_like(d.g, nan), torch.full_like(d.beta, nan),
             torch.full((1, w.h_v, 128, 128), nan, device="cuda:0"))
    try:
        gdn_debug_stall_ns(20000)
        gdn_chunk_bwd(d.q, d.k, d.v, d.g, d.beta, d_out, d.h0, dhT, plan=plan, grads=grads, workspace=ws)
        status = gdn_get_device_status(ws)
    finally:
        gdn_debug_stall_ns(0)
    assert status == (5, 6), describe_device_status(*status)
    assert all(torch.isnan(x).all() for x in grads)
    again = gdn_chunk_bwd(d.q, d.k, d.v, d.g, d.beta, d_out, d.h0, dhT, plan=plan, workspace=ws)
    assert gdn_get_device_status(ws) == (0, 0)
    ws2 = torch.empty_like(ws)
    fresh = gdn_chunk_bwd(d.q, d.k, d.v, d.g, d.beta, d_out, d.h0, dhT, plan=plan, workspace=ws2)
    for x, y in zip(again, fresh):
        assert torch.equal(x, y)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("mode", ["off", "exact"])
@pytest.mark.parametrize("bad", [[0, 300, 900], [0, 800, 700], [0, 300, 650]])
def test_device_offsets_that_disagree_with_the_plan_are_reported(bad, mode, dtype):
    """Device cu_seqlens other than the plan's: a sequence past T, one going back, the
    last ending before T.  The kernels check the offsets before following them: status 7
    (detail 3), no access outside the buffers, and the next call with the plan's offsets
    on the same workspace is clean and correct."""
    w = make_inputs(cu_seqlens=[0, 300, 700], h_qk=2, h_v=4, seed=5, with_h0=True, dtype=dtype)
    d = w.to("cuda:0")
    plan = gdn_cp_plan(T=w.T, h_qk=2, h_v=4, cu_seqlens=w.cu_seqlens, mode=mode, lambda_=0.5, dtype=dtype)
    ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device="cuda:0")
    cu_bad = torch.tensor(bad, dtype=torch.int32, device="cuda:0")
    gdn_chunk_fwd(d.q, d.k, d.v, d.g, d.beta, d.h0, cu_bad, plan=plan, workspace=ws)
    assert gdn_get_device_status(ws) == (DEVICE_CHECK, 3)
    o, hT = gdn_chunk_fwd(d.q, d.k, d.v, d.g, d.beta, d.h0, d.cu_seqlens, plan=plan, workspace=ws)
    assert gdn_get_device_status(ws) == (0, 0)
    f = util.to64
    ro, rh = oracle.recurrence(f(w.q), f(w.k), f(w.v), f(w.g), f(w.beta), f(w.h0), w.seq_offsets())
    if dtype == torch.float32:
        assert util.parity_f32(o, ro) <= 1e-4 and util.parity_f32(hT, rh) <= 1e-4
    else:
        assert util.parity_bf16(o, ro)[0] <= util.TOL_BF16 and util.parity_f32(hT, rh) <= util.TOL_STATE
