"""CPU pins of the float64 backward oracle (module ``oracle.backward``).

The gradients are pinned by central finite differences of the C token
recurrence (which the backward oracle does not use), by a closed form at
beta = 0, and the chunk-level derivation against the autograd definition,
at two chunk sizes.  Planted mistakes in the chunk-level derivation must
fail the comparison.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from oracle import backward as B
from tests.oracle_pins import rand_case

NAMES = ("q", "k", "v", "g", "beta", "h0")


def _case(T_list, h_qk, h_v, d, seed, with_h0=True):
    c = rand_case(T_list, h_qk, h_v, d=d, seed=seed, with_h0=with_h0)
    r = np.random.default_rng(seed + 100)
    T = int(sum(T_list))
    c["do"] = r.standard_normal((T, h_v, d))
    c["dhT"] = 0.3 * r.standard_normal((len(T_list), h_v, d, d))
    return c


def _loss(c, scale=None):
    o, hT = oracle.recurrence(c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"], c["cu"],
                              scale=scale, n_threads=2)
    return float(np.sum(o * c["do"]) + np.sum(hT * c["dhT"]))


def _grads(c, fn=B.grad_recurrence, **kw):
    return dict(zip(NAMES, fn(c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"], c["cu"],
                              c["do"], c["dhT"], **kw)))


@pytest.mark.parametrize("T_list,h_qk,h_v", [([90], 1, 2), ([40, 75], 2, 4)])
def test_grad_recurrence_matches_finite_differences(T_list, h_qk, h_v):
    """Directional derivatives along a random direction per input, by central
    differences of the C oracle's loss, equal <gradient, direction>."""
    c = _case(T_list, h_qk, h_v, d=16, seed=7)
    gr = _grads(c, block=32)
    r = np.random.default_rng(11)
    eps = 1e-5
    for name in NAMES:
        x = c[name]
        direction = r.standard_normal(x.shape)
        cp, cm = dict(c), dict(c)
        cp[name], cm[name] = x + eps * direction, x - eps * direction
        fd = (_loss(cp) - _loss(cm)) / (2 * eps)
        an = float(np.sum(gr[name] * direction))
        assert abs(fd - an) <= 1e-7 * max(1.0, abs(an)), (name, fd, an)


def test_grad_single_coordinates():
    """A few single coordinates of each gradient, by central differences."""
    c = _case([70], 1, 2, d=8, seed=3)
    gr = _grads(c)
    eps = 1e-6
    picks = {"q": (65, 0, 3), "k": (10, 0, 5), "v": (64, 1, 2), "g": (63, 1), "beta": (0, 0),
             "h0": (0, 1, 4, 6)}
    for name, idx in picks.items():
        cp, cm = dict(c), dict(c)
        cp[name], cm[name] = c[name].copy(), c[name].copy()
        cp[name][idx] += eps
        cm[name][idx] -= eps
        fd = (_loss(cp) - _loss(cm)) / (2 * eps)
        assert abs(fd - gr[name][idx]) <= 1e-7 * max(1.0, abs(fd)), (name, fd, gr[name][idx])


def test_grad_beta_zero_closed_form():
    """beta = 0: the state only decays, H_t = exp(G_t) H0, so
    dq_t = scale exp(G_t) H0 do_t, dk = dv = 0,
    dh0 = sum_t scale exp(G_t) q_t do_t^T + exp(G_T) dhT, and
    dg_s = sum_{t >= s} [scale exp(G_t) q_t^T H0 do_t] + exp(G_T) <H0, dhT>."""
    c = _case([100], 1, 1, d=8, seed=5)
    c["beta"] = np.zeros_like(c["beta"])
    gr = _grads(c)
    scale = 1.0 / np.sqrt(8)
    G = np.cumsum(c["g"][:, 0])
    H0, q, do, dhT = c["h0"][0, 0], c["q"][:, 0], c["do"][:, 0], c["dhT"][0, 0]
    dq = scale * np.exp(G)[:, None] * (do @ H0.T)
    dh0 = scale * (np.exp(G)[:, None] * q).T @ do + np.exp(G[-1]) * dhT
    per_t = scale * np.exp(G) * np.einsum("tk,kv,tv->t", q, H0, do)
    per_t[-1] += np.exp(G[-1]) * np.sum(H0 * dhT)
    dg = np.cumsum(per_t[::-1])[::-1]
    np.testing.assert_allclose(gr["q"][:, 0], dq, rtol=0, atol=1e-12)
    np.testing.assert_allclose(gr["h0"][0, 0], dh0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(gr["g"][:, 0], dg, rtol=0, atol=1e-11)
    assert np.abs(gr["k"]).max() == 0 and np.abs(gr["v"]).max() == 0


@pytest.mark.parametrize("C", [16, 64])
def test_chunked_backward_matches_definition(C):
    """The chunk-level derivation equals the autograd definition (several chunks,
    partial chunks, varlen, GQA, h0 and dhT given), at two chunk sizes."""
    c = _case([70, 130], 2, 4, d=32, seed=9)
    ref = _grads(c)
    got = _grads(c, fn=B.grad_chunked, C=C)
    for name in NAMES:
        err = np.abs(got[name] - ref[name]).max() / np.abs(ref[name]).max()
        assert err < 1e-11, (name, err)


def test_chunked_backward_without_h0():
    c = _case([150], 1, 2, d=16, seed=4, with_h0=False)
    c["dhT"] = np.zeros_like(c["dhT"])
    ref, got = _grads(c), _grads(c, fn=B.grad_chunked)
    for name in ("q", "k", "v", "g", "beta", "h0"):
        err = np.abs(got[name] - ref[name]).max() / max(np.abs(ref[name]).max(), 1e-300)
        assert err < 1e-11, (name, err)


# Plausible mistakes in the chunk-level derivation, planted in a copy of the
# oracle's source; each must make the comparison with the definition fail.
MUTANTS = {
    "dprev_undecayed": ("D_prev = gamma_C * D +", "D_prev = D +"),
    "dg_not_cumulated": ("dg = np.cumsum(dG[::-1])[::-1]", "dg = dG"),
    "dv_without_beta": ("dv = bc[:, None] * YU", "dv = YU"),
    "dL_without_A": ("dL = np.tril(-A.T @ (dVp @ Vp.T), -1)", "dL = np.tril(-(dVp @ Vp.T), -1)"),
    "dKK_not_symmetrised": ("dk += (dKK + dKK.T) @ kc", "dk += dKK @ kc"),
    "chunk_end_decay_dropped": ("dG[-1] += dgamma_C * gamma_C + np.sum(ddec * dec)",
                                "dG[-1] += dgamma_C * gamma_C"),
    "YW_sign": ("YW = -YU @ H.T", "YW = YU @ H.T"),
    "dq_state_undecayed": ("dq = gamma[:, None] * dQs +", "dq = dQs +"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name):
    import importlib.util
    import sys
    old, new = MUTANTS[name]
    src = open(B.__file__).read()
    assert src.count(old) == 1, name
    spec = importlib.util.spec_from_loader("oracle._mutant_backward", loader=None)
    mod = importlib.util.module_from_spec(spec)
    mod.__package__ = "oracle"
    sys.modules[spec.name] = mod
    try:
        exec(compile(src.replace(old, new), spec.name, "exec"), mod.__dict__)
        c = _case([100], 1, 2, d=16, seed=12)
        ref = _grads(c)
        got = _grads(c, fn=mod.grad_chunked)
    finally:
        del sys.modules[spec.name]
    worst = max(np.abs(got[n] - ref[n]).max() / np.abs(ref[n]).max() for n in NAMES)
    assert worst > 1e-6, (name, worst)
