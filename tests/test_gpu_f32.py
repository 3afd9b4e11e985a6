"""GPU parity of the fp32 path (q, k, v, o in fp32) against the float64
oracle: max|diff| <= 1e-4 * RMS(ref) for o and for the final state, on small
ragged cases in every context-parallel mode (the fp32 path combines segments
exactly in all of them) and on the 1 x 32768, h 2/8 workload at full size."""
from __future__ import annotations

import pytest
import torch

import oracle
from tests import util

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU, skipped there
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from gated_deltanet_linear_fwd_gb300 import gdn_chunk_fwd, gdn_cp_plan, gdn_get_device_status  # noqa: E402
from gated_deltanet_linear_fwd_gb300.inputs import make_inputs, workload  # noqa: E402

TOL_F32 = 1e-4

CASES = {
    "tiny": lambda: workload("tiny_T512_h2x4", dtype=torch.float32),
    "ragged_gqa3_h0": lambda: make_inputs(cu_seqlens=[0, 1, 65, 200, 200, 391, 1000], h_qk=2, h_v=6, seed=7,
                                          with_h0=True, dtype=torch.float32),
    "long_mix_h0": lambda: make_inputs(8192 + 5, h_qk=2, h_v=8, seed=13, with_h0=True, dtype=torch.float32),
    "many_short": lambda: make_inputs(cu_seqlens=[0, 5, 5, 70, 200, 201, 330, 640, 641, 700], h_qk=1, h_v=2, seed=19,
                                      with_h0=True, dtype=torch.float32),
}


@pytest.mark.parametrize("key", sorted(CASES))
@pytest.mark.parametrize("mode", ["off", "exact", "auto"])
def test_f32_parity(key, mode):
    w = CASES[key]()
    d = w.to("cuda:0")
    plan = gdn_cp_plan(T=w.T, h_qk=w.h_qk, h_v=w.h_v, cu_seqlens=w.cu_seqlens, dtype=torch.float32, mode=mode)
    ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device="cuda:0")
    o, hT = gdn_chunk_fwd(d.q, d.k, d.v, d.g, d.beta, d.h0, d.cu_seqlens, plan=plan, workspace=ws)
    assert gdn_get_device_status(ws)[0] == 0
    f = util.to64
    ro, rh = oracle.recurrence(f(w.q), f(w.k), f(w.v), f(w.g), f(w.beta), f(w.h0), w.seq_offsets())
    eo, eh = util.parity_f32(o, ro), util.parity_f32(hT, rh)
    print(f"f32 {key}/{mode}: o {eo:.2e}  hT {eh:.2e}")
    assert o.dtype == torch.float32
    assert eo <= TOL_F32 and eh <= TOL_F32


def test_f32_parity_full_size():
    """The 1 x 32768, h 2/8 workload in fp32 with the planner's defaults."""
    w = workload("T32768_h2x8", dtype=torch.float32)
    d = w.to("cuda:0")
    plan = gdn_cp_plan(T=w.T, h_qk=w.h_qk, h_v=w.h_v, dtype=torch.float32)
    ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device="cuda:0")
    o, hT = gdn_chunk_fwd(d.q, d.k, d.v, d.g, d.beta, None, plan=plan, workspace=ws)
    assert gdn_get_device_status(ws)[0] == 0
    f = util.to64
    ro, rh = oracle.recurrence(f(w.q), f(w.k), f(w.v), f(w.g), f(w.beta), None)
    eo, eh = util.parity_f32(o, ro), util.parity_f32(hT, rh)
    print(f"f32 full size ({plan.n_seg_total} segments): o {eo:.2e}  hT {eh:.2e}")
    assert eo <= TOL_F32 and eh <= TOL_F32


@pytest.mark.parametrize("kind", ["no_decay", "decay_30", "decay_100", "beta_zero"])
@pytest.mark.parametrize("mode", ["off", "exact"])
def test_f32_degenerate_gates(kind, mode):
    """The kernel keeps S as one scale times a matrix and folds the scale in when it
    leaves [2^-60, 2^60]: no decay (the scale stays 1), a decay of e^-30 a token (a
    fold every other token), e^-100 (exp(g) subnormal or zero: each token restarts
    the state), and beta = 0 (the state only decays)."""
    w = make_inputs(cu_seqlens=[0, 150, 600], h_qk=1, h_v=2, seed=23, with_h0=True, dtype=torch.float32,
                    g_kind="zero" if kind == "no_decay" else "mix")
    if kind.startswith("decay_"):
        w.g = torch.full_like(w.g, -float(kind.split("_")[1]))
    if kind == "beta_zero":
        w.beta = torch.zeros_like(w.beta)
    d = w.to("cuda:0")
    plan = gdn_cp_plan(T=w.T, h_qk=1, h_v=2, cu_seqlens=w.cu_seqlens, dtype=torch.float32, mode=mode,
                       lambda_=0.5)
    ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device="cuda:0")
    o, hT = gdn_chunk_fwd(d.q, d.k, d.v, d.g, d.beta, d.h0, d.cu_seqlens, plan=plan, workspace=ws)
    assert gdn_get_device_status(ws)[0] == 0
    f = util.to64
    ro, rh = oracle.recurrence(f(w.q), f(w.k), f(w.v), f(w.g), f(w.beta), f(w.h0), w.seq_offsets())
    eo, eh = util.parity_f32(o, ro), util.parity_f32(hT, rh)
    print(f"f32 {kind}/{mode}: o {eo:.2e}  hT {eh:.2e}")
    assert torch.isfinite(o).all() and torch.isfinite(hT).all()
    assert eo <= TOL_F32 and eh <= TOL_F32
