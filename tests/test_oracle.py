"""CPU tests of the float64 oracle: pins, planted mistakes, and the chunked/CP form."""
from __future__ import annotations

import os
import shutil

import numpy as np
import pytest

import oracle
from oracle import chunked
from tests import oracle_pins as P

ORACLE_SRC = os.path.join(os.path.dirname(oracle.__file__), "gdn_oracle.c")


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    assert pin(oracle.load()) < P.TOL


# Plausible mistakes, planted in a copy of the oracle source.  Each must make
# at least one pin fail, so the pins are strong enough to trust the oracle.
MUTANTS = {
    "erase_not_decayed": ("alpha * (s - b * Sk[a] * kt[c]) + b * vt[a] * kt[c]",
                          "alpha * s - b * Sk[a] * kt[c] + b * vt[a] * kt[c]"),
    "erase_sign": ("alpha * (s - b * Sk[a] * kt[c])", "alpha * (s + b * Sk[a] * kt[c])"),
    "write_without_beta": ("+ b * vt[a] * kt[c]", "+ vt[a] * kt[c]"),
    "erase_without_beta": ("(s - b * Sk[a] * kt[c])", "(s - Sk[a] * kt[c])"),
    "head_map_modulo": ("(int)(((int64_t)j * hqk) / hv)", "(int)(j % hqk)"),
    "output_transposed": ("acc += S[(size_t)a * dk + c] * qt[c];",
                          "acc += S[(size_t)c * dk + a] * qt[c];"),
    "output_unscaled": ("ot[a] = J->scale * acc;", "ot[a] = acc;"),
    "h0_not_transposed": ("H0[(size_t)c * dv + a]", "H0[(size_t)a * dv + c]"),
    "hT_not_transposed": ("HT[(size_t)c * dv + a] = S[(size_t)a * dk + c]",
                          "HT[(size_t)c * dv + a] = S[(size_t)c * dk + a]"),
    "gate_linear": ("exp(J->g[(size_t)t * hv + j])", "(1.0 + J->g[(size_t)t * hv + j])"),
    "k_uses_q": ("const double *kt = J->k +", "const double *kt = J->q +"),
}


@pytest.fixture(scope="module")
def mutant_dir(tmp_path_factory):
    d = tmp_path_factory.mktemp("mutants")
    yield d
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, mutant_dir):
    src = open(ORACLE_SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    path = mutant_dir / f"{name}.c"
    path.write_text(src.replace(old, new))
    lib = oracle.load(oracle.build(str(path), str(mutant_dir / f"lib{name}.so")))
    fails = []
    for pin in P.ALL_PINS:
        try:
            err = pin(lib)
        except Exception:  # a crash or shape error also counts as caught
            err = np.inf
        if not err < P.TOL:
            fails.append(pin.__name__)
    assert fails, f"no pin catches the planted mistake {name}"


def test_oracle_rejects_bad_args():
    q = np.zeros((4, 1, 2))
    with pytest.raises(ValueError):
        oracle.recurrence(q, q, q, np.zeros((4, 1)), np.zeros((4, 1)), None, [0, 3, 2])


def test_head_subset_matches_full():
    c = P.rand_case([50], h_qk=2, h_v=4, d=8, seed=11)
    o, hT = oracle.recurrence(c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"], c["cu"])
    o1, hT1 = oracle.recurrence(c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"], c["cu"],
                                heads=[2])
    assert np.abs(o1[:, 2] - o[:, 2]).max() == 0 and np.abs(o1[:, [0, 1, 3]]).max() == 0
    assert np.abs(hT1[:, 2] - hT[:, 2]).max() == 0


# ---- the chunked form's context-parallel pieces (pages, section "AutoCP") ----

def _case(seed=21, T_list=(300, 129), d=16):
    return P.rand_case(list(T_list), h_qk=1, h_v=2, d=d, seed=seed)


def test_cp_exact_equals_single_segment():
    c = _case()
    segs = [[(0, 1), (1, 3), (3, 5)], [(0, 2), (2, 3)]]
    args = (c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"], c["cu"])
    o0, h0 = chunked.gdn_fwd_chunked(*args)
    o1, h1 = chunked.gdn_fwd_chunked(*args, segments=segs)
    o2, h2 = oracle.recurrence(*args)
    assert np.abs(o0 - o1).max() < 1e-12 and np.abs(h0 - h1).max() < 1e-12
    assert np.abs(o1 - o2).max() < 1e-12 and np.abs(h1 - h2).max() < 1e-12


def test_segment_transition_is_affine_map():
    """M and H_loc reproduce the scan from two different start states."""
    c = _case(seed=22)
    a, b = c["cu"][0], c["cu"][1]
    ks, vs, gs, bs, qs = (c[x][a:b, 0 if x in ("q", "k") else 1] for x in ("k", "v", "g", "beta", "q"))
    M, Hloc = chunked.segment_transition(ks, vs, gs, bs, (1, 4))
    r = np.random.default_rng(0)
    for _ in range(2):
        H0 = r.standard_normal((16, 16))
        H = chunked.scan_head(qs, ks, vs, gs, bs, H0, 0.25, chunk_range=(1, 4))
        assert np.abs(H - (M @ H0 + Hloc)).max() < 1e-12


def test_warmup_covering_prefix_is_exact():
    """A warmup restart that reaches back to the sequence start is exact."""
    c = _case(seed=23)
    segs = [[(0, 2), (2, 5)], [(0, 1), (1, 3)]]
    args = (c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"], c["cu"])
    o0, h0 = chunked.gdn_fwd_chunked(*args)
    o1, h1 = chunked.gdn_fwd_chunked(*args, segments=segs, warmup_chunks=8)
    assert np.abs(o0 - o1).max() < 1e-12 and np.abs(h0 - h1).max() < 1e-12


def test_warmup_error_within_gate_bound():
    """Warmup start-state error <= exp(sum of g over the window) * ||H(start - w)||
    for unit keys and beta in [0, 1] (each token map has spectral norm <= alpha)."""
    c = _case(seed=24, T_list=(640,), d=16)
    q, k, v, g, beta = (c[x][:, 0] if x in ("q", "k") else c[x][:, 0] for x in ("q", "k", "v", "g", "beta"))
    for w in (1, 2, 4):
        cb = 6
        H_exact_early = chunked.scan_head(q, k, v, g, beta, c["h0"][0, 0], 0.25, chunk_range=(0, cb - w))
        H_exact = chunked.scan_head(q, k, v, g, beta, c["h0"][0, 0], 0.25, chunk_range=(0, cb))
        H_warm = chunked.scan_head(q, k, v, g, beta, np.zeros((16, 16)), 0.25, chunk_range=(cb - w, cb))
        bound = np.exp(g[(cb - w) * 64: cb * 64].sum()) * np.linalg.norm(H_exact_early, 2)
        assert np.linalg.norm(H_exact - H_warm, 2) <= bound * (1 + 1e-9)
