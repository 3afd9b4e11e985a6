"""GPU parity of the backward (gdn_chunk_bwd) against the float64 oracle gradients.

The oracle is ``oracle.backward``: the autograd definition on small cases and
the chunk-level derivation (pinned to it on the CPU) on the larger ones, both
on the exact bf16/fp32 values the GPU receives.  Bar, per gradient tensor:
max|diff| <= 2e-2 * RMS(ref), the forward's bf16 rule; dq, dk and dv are bf16
outputs, so their half-ulp rounding is allowed on top, as for o.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle import backward as OB
from tests import util

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU, skipped there
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from gated_deltanet_linear_fwd_gb300 import gdn_chunk_bwd, gdn_cp_plan, gdn_get_device_status  # noqa: E402
from gated_deltanet_linear_fwd_gb300.api import gdn_bwd_workspace_bytes  # noqa: E402
from gated_deltanet_linear_fwd_gb300.inputs import make_inputs, make_output_grads, workload  # noqa: E402

DEV = "cuda:0"
NAMES = ("dq", "dk", "dv", "dg", "dbeta", "dh0")
TOL = 2e-2


def run_bwd(w, d_out, dhT, mode="off", h0=True):
    d = w.to(DEV)
    plan = gdn_cp_plan(T=w.T, h_qk=w.h_qk, h_v=w.h_v, cu_seqlens=w.cu_seqlens, mode=mode)
    ws = torch.empty(gdn_bwd_workspace_bytes(plan), dtype=torch.uint8, device=DEV)
    grads = gdn_chunk_bwd(d.q, d.k, d.v, d.g, d.beta, d_out.to(DEV), d.h0 if h0 else None,
                          None if dhT is None else dhT.to(DEV), d.cu_seqlens, plan=plan, workspace=ws)
    code, detail = gdn_get_device_status(ws)
    assert code == 0, f"device status {code} detail {detail}"
    return dict(zip(NAMES, grads)), plan


def ref_grads(w, d_out, dhT, h0=True, fn=OB.grad_chunked, heads=None):
    f = util.to64
    kw = {} if heads is None else {"heads": heads}
    return dict(zip(NAMES, fn(f(w.q), f(w.k), f(w.v), f(w.g), f(w.beta), f(w.h0) if h0 else None,
                              w.seq_offsets(), f(d_out), None if dhT is None else f(dhT), **kw)))


def check(got, ref, names=NAMES, tol=TOL):
    worst = {}
    for n in names:
        r = ref[n]
        x = got[n].double().cpu().numpy()
        rms = float(np.sqrt(np.mean(r * r)))
        err = np.abs(x - r)
        if n in ("dq", "dk", "dv"):
            err = np.maximum(err - util.bf16_half_ulp(r), 0.0)
        worst[n] = float(err.max()) / max(rms, 1e-30)
    bad = {n: e for n, e in worst.items() if not e <= tol}
    assert not bad, f"over {tol}: {bad} (all: {worst})"
    return worst


@pytest.mark.parametrize("mode", ["off", "auto"])
def test_bwd_small_against_definition(mode):
    """Several chunks and a partial one, h0 and dhT given; the autograd oracle."""
    w = make_inputs(200, h_qk=1, h_v=2, seed=21, with_h0=True)
    d_out, dhT = make_output_grads(w, seed=22)
    got, _ = run_bwd(w, d_out, dhT, mode=mode)
    check(got, ref_grads(w, d_out, dhT, fn=OB.grad_recurrence))


@pytest.mark.parametrize("mode", ["off", "exact", "auto"])
def test_bwd_varlen_gqa(mode):
    """Varlen with a one-token and an exactly-one-chunk sequence, GQA 2/4, CP modes."""
    w = make_inputs(cu_seqlens=[0, 70, 330, 394, 395, 700], h_qk=2, h_v=4, seed=23, with_h0=True)
    d_out, dhT = make_output_grads(w, seed=24)
    got, _ = run_bwd(w, d_out, dhT, mode=mode)
    check(got, ref_grads(w, d_out, dhT))


def test_bwd_without_h0_or_dhT():
    w = make_inputs(300, h_qk=2, h_v=2, seed=25)
    d_out, _ = make_output_grads(w, seed=26, with_dhT=False)
    got, _ = run_bwd(w, d_out, None, h0=False)
    check(got, ref_grads(w, d_out, None, h0=False))


def test_bwd_batch_rows():
    """B fixed-length rows (no cu_seqlens) of a partial last chunk."""
    w = make_inputs(2 * 150, h_qk=1, h_v=3, seed=27, with_h0=True)
    d = w.to(DEV)
    B, T = 2, 150
    q, k, v = (t.view(B, T, *t.shape[1:]) for t in (d.q, d.k, d.v))
    g, beta = d.g.view(B, T, -1), d.beta.view(B, T, -1)
    h0 = d.h0.repeat(2, 1, 1, 1).contiguous()
    d_out, dhT = make_output_grads(w, seed=28)
    dhT = dhT.repeat(2, 1, 1, 1).contiguous()
    plan = gdn_cp_plan(T=T, h_qk=1, h_v=3, B=B, mode="off")
    ws = torch.empty(gdn_bwd_workspace_bytes(plan), dtype=torch.uint8, device=DEV)
    grads = gdn_chunk_bwd(q, k, v, g, beta, d_out.to(DEV).view(B, T, 3, 128), h0, dhT.to(DEV), plan=plan,
                          workspace=ws)
    assert gdn_get_device_status(ws)[0] == 0
    got = {n: x.reshape(-1, *x.shape[2:]) if n != "dh0" else x for n, x in zip(NAMES, grads)}
    f = util.to64
    h0_np = np.concatenate([f(w.h0)] * 2)
    ref = dict(zip(NAMES, OB.grad_chunked(f(w.q), f(w.k), f(w.v), f(w.g), f(w.beta), h0_np, [0, 150, 300],
                                          f(d_out), f(dhT))))
    check(got, ref)


def test_bwd_more_qk_heads_than_value_heads():
    """h_qk 4 / h_v 2: q/k heads 1 and 3 feed no value head; their gradients are zero."""
    w = make_inputs(130, h_qk=4, h_v=2, seed=29, with_h0=True)
    d_out, dhT = make_output_grads(w, seed=30)
    got, _ = run_bwd(w, d_out, dhT)
    check(got, ref_grads(w, d_out, dhT))
    for n in ("dq", "dk"):
        assert float(got[n][:, 1::2].abs().max()) == 0.0


def test_bwd_no_tokens():
    """T = 0: the gradient of h0 is that of h_T."""
    d = make_inputs(64, h_qk=1, h_v=2, seed=31, with_h0=True).to(DEV)
    e = lambda t: t[:0].contiguous()
    plan = gdn_cp_plan(T=0, h_qk=1, h_v=2, mode="off")
    dhT = torch.randn(1, 2, 128, 128, device=DEV)
    ws = torch.empty(max(gdn_bwd_workspace_bytes(plan), 256), dtype=torch.uint8, device=DEV)
    grads = gdn_chunk_bwd(e(d.q), e(d.k), e(d.v), e(d.g), e(d.beta), e(d.v), d.h0, dhT, plan=plan, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(grads[5], dhT)


def test_bwd_strong_decay():
    """g about -3 a token: exp(G) underflows in fp32 within a chunk."""
    w = make_inputs(cu_seqlens=[0, 70, 333], h_qk=1, h_v=2, seed=32, with_h0=True)
    gen = torch.Generator().manual_seed(33)
    w.g = (-3.0 + 0.5 * torch.randn(w.g.shape, generator=gen)).float()
    d_out, dhT = make_output_grads(w, seed=34)
    got, _ = run_bwd(w, d_out, dhT)
    check(got, ref_grads(w, d_out, dhT))


@pytest.mark.parametrize("kind", ["beta_zero", "no_decay"])
@pytest.mark.parametrize("mode", ["off", "exact"])
def test_bwd_degenerate_gates(kind, mode):
    """beta = 0 (the state only decays: k and v never reach o or h_T, so dk and dv are
    exactly zero) and g = 0 (alpha = 1, no decay at all), with and without context
    parallelism (lambda 0.5: several segments)."""
    w = make_inputs(cu_seqlens=[0, 200, 517], h_qk=1, h_v=2, seed=36, with_h0=True,
                    g_kind="zero" if kind == "no_decay" else "mix")
    if kind == "beta_zero":
        w.beta = torch.zeros_like(w.beta)
    d_out, dhT = make_output_grads(w, seed=37)
    d = w.to(DEV)
    plan = gdn_cp_plan(T=w.T, h_qk=1, h_v=2, cu_seqlens=w.cu_seqlens, mode=mode, lambda_=0.5)
    if mode == "exact":
        assert plan.n_seg_total > 2
    ws = torch.empty(gdn_bwd_workspace_bytes(plan), dtype=torch.uint8, device=DEV)
    grads = gdn_chunk_bwd(d.q, d.k, d.v, d.g, d.beta, d_out.to(DEV), d.h0, dhT.to(DEV), d.cu_seqlens, plan=plan,
                          workspace=ws)
    assert gdn_get_device_status(ws) == (0, 0)
    got = dict(zip(NAMES, grads))
    if kind == "beta_zero":
        assert float(got["dk"].abs().max()) == 0.0 and float(got["dv"].abs().max()) == 0.0
        check(got, ref_grads(w, d_out, dhT), names=("dq", "dg", "dbeta", "dh0"))
    else:
        check(got, ref_grads(w, d_out, dhT))


def test_bwd_million_token_sequence():
    """One sequence of 2^20 tokens (16384 chunks), the largest the forward's tests
    run, in the bench's launch configuration (auto plan); every gradient of both
    value heads element by element against the float64 chunk-level oracle."""
    w = make_inputs(1 << 20, h_qk=1, h_v=2, seed=38, with_h0=True)
    d_out, dhT = make_output_grads(w, seed=39)
    got, plan = run_bwd(w, d_out, dhT, mode="auto")
    assert plan.n_seg_total > 16
    worst = check(got, ref_grads(w, d_out, dhT))
    print(f"bwd 2^20 tokens, {plan.n_seg_total} segments: {worst}")


@pytest.mark.parametrize("name,heads", [("T32768_h2x8", None), ("T32768_h16x16", [0, 7, 15]),
                                        ("T32768_h8x24_h0", [0, 11, 23]), ("varlen4_T348160_h2x8", [1, 6]),
                                        ("batch8_T4096_h8x32", [0, 13, 31])])
def test_bwd_full_size(name, heads):
    """The benchmark's 1 x 32768 workloads at full size, in the bench's launch
    configuration (auto plan); every head, or a sample of heads, element by element."""
    w = workload(name)
    d_out, dhT = make_output_grads(w, seed=35)
    got, plan = run_bwd(w, d_out, dhT, mode="auto", h0=w.h0 is not None)
    ref = ref_grads(w, d_out, dhT, h0=w.h0 is not None, heads=heads)
    if heads is None:
        check(got, ref)
    else:  # the sampled heads' own gradients (dq and dk sum over every head of a group)
        names = ("dv", "dg", "dbeta", "dh0")
        check({n: got[n][:, heads] for n in names}, {n: ref[n][:, heads] for n in names}, names=names)


@pytest.mark.parametrize("mode", ["off", "auto"])
def test_bwd_after_training_forward(mode):
    """gdn_chunk_fwd(for_backward=True) then gdn_chunk_bwd(reuse_forward=True): the same
    gradients, bit for bit, as a backward that recomputes the forward itself, and the
    training forward's o and final state meet the forward's bar against the oracle."""
    from gated_deltanet_linear_fwd_gb300 import gdn_chunk_fwd
    import oracle
    w = make_inputs(cu_seqlens=[0, 300, 700], h_qk=2, h_v=4, seed=41, with_h0=True)
    d_out, dhT = make_output_grads(w, seed=42)
    d = w.to(DEV)
    plan = gdn_cp_plan(T=w.T, h_qk=w.h_qk, h_v=w.h_v, cu_seqlens=w.cu_seqlens, mode=mode)
    ws = torch.empty(gdn_bwd_workspace_bytes(plan), dtype=torch.uint8, device=DEV)
    o, hT = gdn_chunk_fwd(d.q, d.k, d.v, d.g, d.beta, d.h0, d.cu_seqlens, plan=plan, workspace=ws, for_backward=True)
    reused = gdn_chunk_bwd(d.q, d.k, d.v, d.g, d.beta, d_out.to(DEV), d.h0, dhT.to(DEV), d.cu_seqlens, plan=plan,
                           workspace=ws, reuse_forward=True)
    assert gdn_get_device_status(ws)[0] == 0
    fresh, _ = run_bwd(w, d_out, dhT, mode=mode)
    for n, x in zip(NAMES, reused):
        assert torch.equal(x, fresh[n]), n
    f = util.to64
    ro, rh = oracle.recurrence(f(w.q), f(w.k), f(w.v), f(w.g), f(w.beta), f(w.h0), w.seq_offsets())
    excess, _ = util.parity_bf16(o, ro)
    assert excess <= 2e-2
    err = np.abs(hT.double().cpu().numpy() - rh).max() / np.sqrt(np.mean(rh * rh))
    assert err < 2e-2


def test_bwd_empty_sequence_and_uneven_gqa():
    """A varlen batch with an empty sequence (its dh0 is its dh_T), and h_v not a
    multiple of h_qk (q/k head 0 feeds value heads 0 and 1, heads 1 and 2 one each)."""
    w = make_inputs(cu_seqlens=[0, 130, 130, 330], h_qk=3, h_v=4, seed=43, with_h0=True)
    d_out, dhT = make_output_grads(w, seed=44)
    got, _ = run_bwd(w, d_out, dhT, mode="auto")
    check(got, ref_grads(w, d_out, dhT))
    assert torch.equal(got["dh0"][1].cpu(), dhT[1])
