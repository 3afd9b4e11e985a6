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


# ---- the warmup restart branch of the chunked form (pages, section "AutoCP":
#      a segment restarts from a zero state a few chunks before its start) ----
#
# Pinned against the token recurrence, which knows nothing of chunks or
# segments: a warm segment [cb, ce) must equal the recurrence run from a zero
# state over the tokens [(cb - w) * 64, ce * 64) (from h0 over [0, ce * 64)
# when the window reaches the sequence start), read from chunk cb on.

WARM_SEGS = [[(0, 3), (3, 7), (7, 10), (10, 15)]]
WARM_T = 64 * 14 + 23  # 15 chunks, the last one partial
WARM_DEPTHS = [
    2,  # one depth for every segment: windows start at chunks 1, 5, 8 (none clipped)
    {(0, 0, 1): 3, (0, 0, 2): 1, (0, 0, 3): 4,    # head 0: clipped exactly at chunk 0, then 6, 6
     (0, 1, 1): 1, (0, 1, 2): 5, (0, 1, 3): 2},   # head 1: 2, 2, 8
]


def _depth(wc, n, j, s):
    if s == 0:
        return 0  # the first segment starts from h0 at the sequence start
    return wc[(n, j, s)] if isinstance(wc, dict) else wc


def _warm_case(seed, zero_before_windows=None):
    # slow decay (g in [-0.01, 0]): a window's history stays far above rounding
    c = P.rand_case([WARM_T], h_qk=1, h_v=2, d=16, seed=seed, g_scale=0.01)
    if zero_before_windows is not None:
        # alpha = 0 and beta = 0 at the last token before every window: the
        # state entering the window is exactly zero, so nothing is dropped
        for j, starts in zero_before_windows.items():
            for st in starts:
                t = st * 64 - 1
                c["g"][t, j] = -800.0  # exp(-800) is 0 in float64
                c["beta"][t, j] = 0.0
    return c


def _warm_violation(mod, c, wc):
    """Largest |chunked warmup - recurrence on the restarted slice| over the
    warm segments of both heads (o of every segment, the final state)."""
    args = (c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"], c["cu"])
    o, hT = mod.gdn_fwd_chunked(*args, segments=WARM_SEGS, warmup_chunks=wc)
    worst = 0.0
    for j in range(2):
        for si, (cb, ce) in enumerate(WARM_SEGS[0]):
            wd = _depth(wc, 0, j, si)
            start = 0 if si == 0 or cb - wd <= 0 else cb - wd
            a, b = start * 64, min(ce * 64, WARM_T)
            h_init = np.zeros_like(c["h0"]) if start > 0 else c["h0"]
            ro, rh = oracle.recurrence(c["q"][a:b], c["k"][a:b], c["v"][a:b], c["g"][a:b], c["beta"][a:b],
                                       h_init, [0, b - a], heads=[j], n_threads=2)
            worst = max(worst, np.abs(o[cb * 64:b, j] - ro[(cb - start) * 64:, j]).max())
            if si == len(WARM_SEGS[0]) - 1:
                worst = max(worst, np.abs(hT[0, j] - rh[0, j]).max())
    return worst


@pytest.mark.parametrize("wc", WARM_DEPTHS, ids=["int", "per-segment"])
def test_warmup_branch_equals_restarted_recurrence(wc):
    assert _warm_violation(chunked, _warm_case(31), wc) < 1e-11


@pytest.mark.parametrize("wc", WARM_DEPTHS, ids=["int", "per-segment"])
def test_warmup_is_exact_when_history_before_window_is_zero(wc):
    """With the state wiped (alpha = beta = 0) at the token before every
    window, the warmup result is the full recurrence itself."""
    starts = {j: [cb - _depth(wc, 0, j, si) for si, (cb, _) in enumerate(WARM_SEGS[0])
                  if si > 0 and cb - _depth(wc, 0, j, si) > 0] for j in range(2)}
    c = _warm_case(32, starts)
    args = (c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"], c["cu"])
    o, hT = chunked.gdn_fwd_chunked(*args, segments=WARM_SEGS, warmup_chunks=wc)
    ro, rh = oracle.recurrence(*args, n_threads=2)
    assert np.abs(o - ro).max() < 1e-11 and np.abs(hT - rh).max() < 1e-11
    # and without the wipe the same windows do drop history (the pin is not vacuous)
    c2 = _warm_case(32)
    o2, _ = chunked.gdn_fwd_chunked(c2["q"], c2["k"], c2["v"], c2["g"], c2["beta"], c2["h0"], c2["cu"],
                                    segments=WARM_SEGS, warmup_chunks=wc)
    ro2, _ = oracle.recurrence(c2["q"], c2["k"], c2["v"], c2["g"], c2["beta"], c2["h0"], c2["cu"], n_threads=2)
    assert np.abs(o2 - ro2).max() > 1e-6


# Off-by-one windows planted in a copy of the chunked form: each must break the pin.
WARM_MUTANTS = {
    "window_one_late": ("(cb - wd, cb))", "(cb - wd + 1, cb))"),
    "window_one_early": ("(cb - wd, cb))", "(cb - wd - 1, cb))"),
    "clip_strict": ("cb - wd <= 0", "cb - wd < 0"),
    "depth_of_next_segment": ("warmup_chunks[(n, j, si)]", "warmup_chunks.get((n, j, si + 1), 1)"),
}


@pytest.mark.parametrize("name", sorted(WARM_MUTANTS))
def test_planted_warmup_mistake_is_caught(name):
    import types
    src = open(chunked.__file__).read()
    old, new = WARM_MUTANTS[name]
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mod = types.ModuleType(f"chunked_{name}")
    exec(compile(src.replace(old, new), f"<{name}>", "exec"), mod.__dict__)
    worst = max(_warm_violation(mod, _warm_case(31), wc) for wc in WARM_DEPTHS)
    assert not worst < 1e-11, f"the warmup pin misses the planted mistake {name}"
