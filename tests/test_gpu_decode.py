"""The one-token step (gdn_decode_step) against the float64 oracle.

The oracle's recurrence over one token per sequence, started from the given
state, is the step's definition; a prefill followed by decode steps must also
equal the oracle over the longer sequence (the step continues a prefill's
final state).  fp32 I/O is held to 1e-4 * RMS; bf16 I/O to the prefill's
tolerance reading.
"""
from __future__ import annotations

import pytest
import torch

import oracle
from tests import util

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU, skipped there
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from gated_deltanet_linear_fwd_gb300 import gdn_chunk_fwd, gdn_decode_step  # noqa: E402
from gated_deltanet_linear_fwd_gb300.inputs import make_inputs  # noqa: E402

TOL_F32 = 1e-4
f = util.to64


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("B,h_qk,h_v", [(1, 1, 1), (5, 2, 8), (33, 4, 4), (7, 8, 24)])
def test_decode_step_matches_oracle(B, h_qk, h_v, dtype):
    # B sequences of one token each, started from a random state
    w = make_inputs(cu_seqlens=list(range(B + 1)), h_qk=h_qk, h_v=h_v, seed=100 + B, with_h0=True, dtype=dtype)
    ro, rh = oracle.recurrence(f(w.q), f(w.k), f(w.v), f(w.g), f(w.beta), f(w.h0), w.seq_offsets())
    d = w.to("cuda:0")
    state = d.h0.clone()
    o = gdn_decode_step(d.q, d.k, d.v, d.g, d.beta, state)
    torch.cuda.synchronize()
    assert o.dtype == dtype
    eh = util.parity_f32(state, rh)
    if dtype == torch.float32:
        eo = util.parity_f32(o, ro)
        print(f"decode f32 B={B} {h_qk}/{h_v}: o {eo:.2e}  state {eh:.2e}")
        assert eo <= TOL_F32 and eh <= TOL_F32
    else:
        excess, raw = util.parity_bf16(o, ro)
        print(f"decode bf16 B={B} {h_qk}/{h_v}: o excess {excess:.2e} (raw {raw:.2e})  state {eh:.2e}")
        assert excess <= util.TOL_BF16 and eh <= util.TOL_STATE


def test_prefill_then_decode_continues_the_sequence():
    # a prefill of T tokens, then 3 steps == the oracle over T + 3 tokens
    T, extra = 200, 3
    w = make_inputs(T + extra, h_qk=2, h_v=4, seed=21, with_h0=True)
    ro, rh = oracle.recurrence(f(w.q), f(w.k), f(w.v), f(w.g), f(w.beta), f(w.h0), w.seq_offsets())
    d = w.to("cuda:0")
    cut = lambda t, a, b: t[a:b].contiguous()
    o_pre, state = gdn_chunk_fwd(cut(d.q, 0, T), cut(d.k, 0, T), cut(d.v, 0, T), cut(d.g, 0, T),
                                 cut(d.beta, 0, T), d.h0)
    outs = [o_pre]
    for t in range(T, T + extra):
        outs.append(gdn_decode_step(cut(d.q, t, t + 1), cut(d.k, t, t + 1), cut(d.v, t, t + 1),
                                    cut(d.g, t, t + 1), cut(d.beta, t, t + 1), state))
    torch.cuda.synchronize()
    excess, raw = util.parity_bf16(torch.cat(outs), ro)
    eh = util.parity_f32(state, rh)
    print(f"prefill + decode: o excess {excess:.2e} (raw {raw:.2e})  state {eh:.2e}")
    assert excess <= util.TOL_BF16 and eh <= util.TOL_STATE
