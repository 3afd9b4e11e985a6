"""CUDA-graph capture of the public calls.

A serving or training loop replays a captured step instead of launching its
kernels one by one.  The calls put only stream-ordered work on the caller's
stream (the status word's memset, kernels with programmatic dependent launch,
device-to-device copies), so a call captured once and replayed on new inputs
placed in the same buffers must give the eager call's results bit for bit:
the kernels are deterministic.
"""
from __future__ import annotations

import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU, skipped there
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from gated_deltanet_linear_fwd_gb300 import (gdn_chunk_bwd, gdn_chunk_fwd, gdn_cp_plan,  # noqa: E402
                                             gdn_decode_step, gdn_get_device_status)
from gated_deltanet_linear_fwd_gb300.api import gdn_bwd_workspace_bytes  # noqa: E402
from gated_deltanet_linear_fwd_gb300.inputs import make_inputs, make_output_grads  # noqa: E402

DEV = "cuda:0"
CU = [0, 700, 2500, 6000]  # three sequences, partial last chunks


def _capture(fn):
    """Warm up on a side stream (one-time set-up stays out of the graph), then capture."""
    side = torch.cuda.Stream(DEV)
    side.wait_stream(torch.cuda.current_stream(DEV))
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream(DEV).wait_stream(side)
    torch.cuda.synchronize(DEV)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fn()
    return graph


def _load(static, w):
    for name in ("q", "k", "v", "g", "beta", "h0"):
        getattr(static, name).copy_(getattr(w, name))


@pytest.mark.parametrize("mode", ["off", "exact", "auto"])
def test_forward_graph_replay_equals_eager(mode):
    wa = make_inputs(cu_seqlens=CU, h_qk=2, h_v=8, seed=61, with_h0=True)
    wb = make_inputs(cu_seqlens=CU, h_qk=2, h_v=8, seed=62, with_h0=True)
    s = wa.to(DEV)  # the static buffers the graph reads
    plan = gdn_cp_plan(T=wa.T, h_qk=2, h_v=8, cu_seqlens=wa.cu_seqlens, mode=mode, lambda_=0.5)
    if mode != "off":
        assert plan.n_seg_total > 3
    ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device=DEV)
    out = torch.empty_like(s.v)
    hT = torch.empty(3, 8, 128, 128, dtype=torch.float32, device=DEV)
    run = lambda: gdn_chunk_fwd(s.q, s.k, s.v, s.g, s.beta, s.h0, s.cu_seqlens, plan=plan, out=out,
                                final_state=hT, workspace=ws)
    graph = _capture(run)
    for w in (wb, wa):
        _load(s, w)
        graph.replay()
        torch.cuda.synchronize()
        o_g, h_g = out.clone(), hT.clone()
        assert gdn_get_device_status(ws) == (0, 0)
        d = w.to(DEV)
        o_e, h_e = gdn_chunk_fwd(d.q, d.k, d.v, d.g, d.beta, d.h0, d.cu_seqlens, plan=plan)
        torch.cuda.synchronize()
        assert torch.equal(o_g, o_e) and torch.equal(h_g, h_e), mode


def test_backward_graph_replay_equals_eager():
    wa = make_inputs(cu_seqlens=CU, h_qk=2, h_v=8, seed=63, with_h0=True)
    wb = make_inputs(cu_seqlens=CU, h_qk=2, h_v=8, seed=64, with_h0=True)
    s = wa.to(DEV)
    do_a, dhT_a = make_output_grads(wa, seed=65)
    do_b, dhT_b = make_output_grads(wb, seed=66)
    d_out, dhT = do_a.to(DEV), dhT_a.to(DEV)
    plan = gdn_cp_plan(T=wa.T, h_qk=2, h_v=8, cu_seqlens=wa.cu_seqlens, mode="auto", lambda_=0.5)
    ws = torch.empty(gdn_bwd_workspace_bytes(plan), dtype=torch.uint8, device=DEV)
    grads = (torch.empty_like(s.q), torch.empty_like(s.k), torch.empty_like(s.v), torch.empty_like(s.g),
             torch.empty_like(s.beta), torch.empty(3, 8, 128, 128, dtype=torch.float32, device=DEV))
    run = lambda: gdn_chunk_bwd(s.q, s.k, s.v, s.g, s.beta, d_out, s.h0, dhT, s.cu_seqlens, plan=plan,
                                grads=grads, workspace=ws)
    graph = _capture(run)
    for w, do_, dh_ in ((wb, do_b, dhT_b), (wa, do_a, dhT_a)):
        _load(s, w)
        d_out.copy_(do_)
        dhT.copy_(dh_)
        graph.replay()
        torch.cuda.synchronize()
        got = [t.clone() for t in grads]
        assert gdn_get_device_status(ws) == (0, 0)
        d = w.to(DEV)
        ref = gdn_chunk_bwd(d.q, d.k, d.v, d.g, d.beta, do_.to(DEV), d.h0, dh_.to(DEV), d.cu_seqlens, plan=plan)
        torch.cuda.synchronize()
        for name, a, b in zip(("dq", "dk", "dv", "dg", "dbeta", "dh0"), got, ref):
            assert torch.equal(a, b), name


def test_training_step_graph_replay_equals_eager():
    """The training forward and the backward that reuses its state, captured as one step."""
    wa = make_inputs(cu_seqlens=CU, h_qk=2, h_v=8, seed=67, with_h0=True)
    s = wa.to(DEV)
    do_a, dhT_a = make_output_grads(wa, seed=68)
    d_out, dhT = do_a.to(DEV), dhT_a.to(DEV)
    plan = gdn_cp_plan(T=wa.T, h_qk=2, h_v=8, cu_seqlens=wa.cu_seqlens, mode="auto", lambda_=0.5)
    ws = torch.empty(gdn_bwd_workspace_bytes(plan), dtype=torch.uint8, device=DEV)
    out = torch.empty_like(s.v)
    hT = torch.empty(3, 8, 128, 128, dtype=torch.float32, device=DEV)
    grads = (torch.empty_like(s.q), torch.empty_like(s.k), torch.empty_like(s.v), torch.empty_like(s.g),
             torch.empty_like(s.beta), torch.empty(3, 8, 128, 128, dtype=torch.float32, device=DEV))

    def step():
        gdn_chunk_fwd(s.q, s.k, s.v, s.g, s.beta, s.h0, s.cu_seqlens, plan=plan, out=out, final_state=hT,
                      workspace=ws, for_backward=True)
        gdn_chunk_bwd(s.q, s.k, s.v, s.g, s.beta, d_out, s.h0, dhT, s.cu_seqlens, plan=plan, grads=grads,
                      workspace=ws, reuse_forward=True)

    graph = _capture(step)
    graph.replay()
    torch.cuda.synchronize()
    got = [out.clone(), hT.clone()] + [t.clone() for t in grads]
    assert gdn_get_device_status(ws) == (0, 0)
    ws2 = torch.empty_like(ws)  # the same step, eager, on a workspace of its own
    ref_o, ref_h = gdn_chunk_fwd(s.q, s.k, s.v, s.g, s.beta, s.h0, s.cu_seqlens, plan=plan, workspace=ws2,
                                 for_backward=True)
    ref_g = gdn_chunk_bwd(s.q, s.k, s.v, s.g, s.beta, d_out, s.h0, dhT, s.cu_seqlens, plan=plan, workspace=ws2,
                          reuse_forward=True)
    torch.cuda.synchronize()
    for name, a, b in zip(("o", "h_T", "dq", "dk", "dv", "dg", "dbeta", "dh0"), got, [ref_o, ref_h, *ref_g]):
        assert torch.equal(a, b), name


def test_decode_steps_graph_replay_equals_eager():
    """Eight decode steps captured as one graph, the state updated in place."""
    B, h_qk, h_v, n = 16, 2, 8, 8
    toks = [make_inputs(cu_seqlens=list(range(B + 1)), h_qk=h_qk, h_v=h_v, seed=70 + i, with_h0=(i == 0))
            for i in range(n)]
    dev = [w.to(DEV) for w in toks]
    state0 = dev[0].h0.clone()
    state = state0.clone()
    outs = [torch.empty_like(d.v) for d in dev]

    def steps():
        for d, o in zip(dev, outs):
            gdn_decode_step(d.q, d.k, d.v, d.g, d.beta, state, out=o)

    graph = _capture(steps)  # (the warm-up advanced the state: start again)
    state.copy_(state0)
    graph.replay()
    torch.cuda.synchronize()
    got_o, got_s = [o.clone() for o in outs], state.clone()
    ref_s = state0.clone()
    ref_o = [gdn_decode_step(d.q, d.k, d.v, d.g, d.beta, ref_s) for d in dev]
    torch.cuda.synchronize()
    assert torch.equal(got_s, ref_s)
    for a, b in zip(got_o, ref_o):
        assert torch.equal(a, b)
