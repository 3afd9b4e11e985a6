"""Pins of the float64 oracle against facts that do not come from the oracle itself.

Each ``pin_*`` function runs the token recurrence (through a given oracle
library handle, so that planted-mistake builds can be checked too) and
returns the largest violation it saw.  A pin passes when that number is below
``TOL``.  The pins are closed forms and special cases of the gated delta rule
(Gated Delta Networks, ICLR 2025, section "Gated delta rule"), invariants that
follow from it, a hand-worked example, and the independent chunked closed form
(oracle/chunked.py), which takes the FlashQLA pages' chunked-prefill route
(section "Optimising GDN chunked prefill") to the same result.
"""
from __future__ import annotations

import json
import os

import numpy as np

import oracle
from oracle import chunked

TOL = 1e-10
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def rand_case(T_list, h_qk, h_v, d=8, seed=0, with_h0=True, unit_k=True, g_scale=0.3):
    """Random float64 inputs; T_list = sequence lengths (varlen)."""
    r = _rng(seed)
    T = int(sum(T_list))
    cu = np.concatenate([[0], np.cumsum(T_list)]).astype(np.int64)
    q = r.standard_normal((T, h_qk, d))
    k = r.standard_normal((T, h_qk, d))
    if unit_k:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
    v = r.standard_normal((T, h_v, d))
    g = -g_scale * r.random((T, h_v))
    beta = r.random((T, h_v))
    h0 = r.standard_normal((len(T_list), h_v, d, d)) if with_h0 else None
    return dict(q=q, k=k, v=v, g=g, beta=beta, h0=h0, cu=cu)


def _rec(lib, c, **kw):
    return oracle.recurrence(c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"], c["cu"],
                             lib=lib, n_threads=2, **kw)


def pin_hand_example(lib):
    """Hand-worked d=2, T=2 example (tests/golden/hand_d2_T2.json)."""
    with open(os.path.join(GOLDEN, "hand_d2_T2.json")) as f:
        e = json.load(f)
    q = np.array(e["q"])[:, None, :]
    k = np.array(e["k"])[:, None, :]
    v = np.array(e["v"])[:, None, :]
    g = np.log(np.array(e["alpha"]))[:, None]
    beta = np.array(e["beta"])[:, None]
    o, hT = oracle.recurrence(q, k, v, g, beta, None, [0, 2], scale=e["scale"], lib=lib)
    return max(np.abs(o[:, 0] - np.array(e["o"])).max(),
               np.abs(hT[0, 0] - np.array(e["H_final"])).max())


def pin_chunked_form(lib, seed=1):
    """Recurrence == chunked closed form (varlen, partial/empty chunks, GQA, h0)."""
    c = rand_case([70, 1, 0, 200, 64], h_qk=2, h_v=6, d=16, seed=seed)
    o, hT = _rec(lib, c)
    worst = 0.0
    for C in (1, 16, 64):
        o2, hT2 = chunked.gdn_fwd_chunked(c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"],
                                          c["cu"], C=C)
        worst = max(worst, np.abs(o - o2).max(), np.abs(hT - hT2).max())
    return worst


def pin_beta_zero(lib, seed=2):
    """beta = 0: no writes; S_t = exp(G_t) S_0, o_t = scale exp(G_t) S_0 q_t."""
    c = rand_case([50, 33], h_qk=1, h_v=2, d=8, seed=seed)
    c["beta"] = np.zeros_like(c["beta"])
    o, hT = _rec(lib, c)
    worst = 0.0
    scale = 1 / np.sqrt(8)
    for n in range(2):
        a, b = c["cu"][n], c["cu"][n + 1]
        for j in range(2):
            G = np.cumsum(c["g"][a:b, j])
            S0 = c["h0"][n, j].T
            ref_o = scale * np.exp(G)[:, None] * (c["q"][a:b, 0] @ S0.T)
            worst = max(worst, np.abs(o[a:b, j] - ref_o).max(),
                        np.abs(hT[n, j] - np.exp(G[-1]) * c["h0"][n, j]).max())
    return worst


def _orthonormal_keys(T, d, r):
    Qm, _ = np.linalg.qr(r.standard_normal((d, d)))
    return Qm[:T]


def pin_orthonormal_linear_attention(lib, seed=3):
    """Orthonormal keys, S_0 = 0: S_{t-1} k_t = 0, so the layer is decayed
    linear attention o_t = scale sum_{s<=t} exp(G_t - G_s) beta_s (k_s.q_t) v_s."""
    r = _rng(seed)
    d, T = 16, 16
    k = _orthonormal_keys(T, d, r)[:, None, :]
    q = r.standard_normal((T, 1, d))
    v = r.standard_normal((T, 2, d))
    g = -0.5 * r.random((T, 2))
    beta = r.random((T, 2))
    c = dict(q=q, k=k, v=v, g=g, beta=beta, h0=None, cu=np.array([0, T]))
    o, hT = _rec(lib, c)
    scale = 1 / np.sqrt(d)
    worst = 0.0
    for j in range(2):
        G = np.cumsum(g[:, j])
        D = np.tril(np.exp(G[:, None] - G[None, :]))
        att = D * (q[:, 0] @ k[:, 0].T) * beta[None, :, j]
        worst = max(worst, np.abs(o[:, j] - scale * att @ v[:, j]).max())
        # final state of linear attention: H = sum_s exp(G_T - G_s) beta_s k_s v_s^T
        Href = (k[:, 0] * (np.exp(G[-1] - G) * beta[:, j])[:, None]).T @ v[:, j]
        worst = max(worst, np.abs(hT[0, j] - Href).max())
    return worst


def pin_overwrite(lib, seed=4):
    """alpha = 1, beta = 1, orthonormal keys: each write overwrites, S_t k_s = v_s
    for s <= t, and S_T = S_0 (I - sum k k^T) + sum v k^T."""
    r = _rng(seed)
    d, T = 16, 12
    k = _orthonormal_keys(T, d, r)[:, None, :]
    q = k.copy()  # o_t = scale S_t k_t = scale v_t
    v = r.standard_normal((T, 1, d))
    g = np.zeros((T, 1))
    beta = np.ones((T, 1))
    h0 = r.standard_normal((1, 1, d, d))
    c = dict(q=q, k=k, v=v, g=g, beta=beta, h0=h0, cu=np.array([0, T]))
    o, hT = _rec(lib, c)
    scale = 1 / np.sqrt(d)
    kk = k[:, 0]
    S0 = h0[0, 0].T
    S_T = S0 @ (np.eye(d) - kk.T @ kk) + v[:, 0].T @ kk
    worst = max(np.abs(o[:, 0] - scale * v[:, 0]).max(), np.abs(hT[0, 0].T - S_T).max())
    # every earlier key still reads back its value
    worst = max(worst, np.abs(hT[0, 0].T @ kk.T - v[:, 0].T).max())
    return worst


def pin_gqa_mapping(lib, seed=5):
    """Grouped heads: h_qk = h_v with duplicated q/k heads equals the grouped call;
    value head j reads q/k head floor(j h_qk / h_v) (h_qk=2, h_v=3: 0, 0, 1)."""
    c = rand_case([40, 30], h_qk=2, h_v=3, d=8, seed=seed)
    o, hT = _rec(lib, c)
    idx = [(j * 2) // 3 for j in range(3)]
    assert idx == [0, 0, 1]
    c2 = dict(c)
    c2["q"] = c["q"][:, idx]
    c2["k"] = c["k"][:, idx]
    o2, hT2 = _rec(lib, c2)
    return max(np.abs(o - o2).max(), np.abs(hT - hT2).max())


def pin_varlen_resume(lib, seed=6):
    """Packed sequences equal separate calls; a split call resumed from the
    first part's final state equals one call."""
    c = rand_case([37, 90], h_qk=1, h_v=2, d=8, seed=seed)
    o, hT = _rec(lib, c)
    worst = 0.0
    for n in range(2):
        a, b = c["cu"][n], c["cu"][n + 1]
        cn = {kk: (vv[a:b] if kk in ("q", "k", "v", "g", "beta") else vv) for kk, vv in c.items()}
        cn["h0"] = c["h0"][n:n + 1]
        cn["cu"] = np.array([0, b - a])
        on, hTn = _rec(lib, cn)
        worst = max(worst, np.abs(on - o[a:b]).max(), np.abs(hTn[0] - hT[n]).max())
        # resume at token m
        m = (b - a) // 3
        c1 = {kk: (vv[:m] if kk in ("q", "k", "v", "g", "beta") else vv) for kk, vv in cn.items()}
        c1["cu"] = np.array([0, m])
        o1, hT1 = _rec(lib, c1)
        c2 = {kk: (vv[m:] if kk in ("q", "k", "v", "g", "beta") else vv) for kk, vv in cn.items()}
        c2["cu"] = np.array([0, b - a - m])
        c2["h0"] = hT1
        o2, hT2 = _rec(lib, c2)
        worst = max(worst, np.abs(np.concatenate([o1, o2]) - on).max(), np.abs(hT2 - hTn).max())
    return worst


def pin_write_identity_and_contraction(lib, seed=7):
    """For unit k_t: S_t k_t = alpha_t (1 - beta_t) S_{t-1} k_t + beta_t v_t, and
    ||S_t||_F <= alpha_t ||S_{t-1}||_F + beta_t ||v_t|| (||I - b k k^T||_2 <= 1).
    Returns the worst identity error plus any contraction excess."""
    c = rand_case([24], h_qk=1, h_v=1, d=8, seed=seed)
    worst = 0.0
    prev = c["h0"][0, 0].T
    for t in range(1, 25):
        ct = {kk: (vv[:t] if kk in ("q", "k", "v", "g", "beta") else vv) for kk, vv in c.items()}
        ct["cu"] = np.array([0, t])
        _, hT = _rec(lib, ct)
        S = hT[0, 0].T
        kt = c["k"][t - 1, 0]
        a = np.exp(c["g"][t - 1, 0])
        b = c["beta"][t - 1, 0]
        vt = c["v"][t - 1, 0]
        worst = max(worst, np.abs(S @ kt - (a * (1 - b) * (prev @ kt) + b * vt)).max())
        excess = np.linalg.norm(S) - (a * np.linalg.norm(prev) + b * np.linalg.norm(vt))
        worst = max(worst, excess)
        prev = S
    return worst


ALL_PINS = [pin_hand_example, pin_chunked_form, pin_beta_zero, pin_orthonormal_linear_attention,
            pin_overwrite, pin_gqa_mapping, pin_varlen_resume, pin_write_identity_and_contraction]
