"""float64 CPU gradients of the GDN forward.  TEST INFRASTRUCTURE ONLY.

Only tests/, ``__graft_entry__.smoke()`` and bench.py's cpu_baseline leg may use
this module.  It shares no code with the CUDA path.

The FlashQLA pages name a fused backward (section "TileLang warp-specialised
kernels", the backward-pass bullet: the dv, dh, dq/dk/dw/dg and WY gradient
steps in one kernel) but give no gradient formulas.  The gradient of a scalar
loss  sum(o * do) + sum(h_T * dh_T)  with respect to every input is fixed by
the forward alone, so two implementations are given here:

* ``grad_recurrence`` -- the definition: reverse-mode differentiation
  (torch.autograd, float64, CPU) of the token-by-token recurrence
      H_t = a_t (I - b_t k_t k_t^T) H_{t-1} + b_t k_t v_t^T,  o_t = scale H_t^T q_t
  (H = S^T, d_k x d_v; a_t = exp(g_t)), run over blocks of tokens in reverse
  with the state gradient handed from block to block (gradient
  checkpointing; the chain rule across a block boundary is that hand-over).
* ``grad_chunked`` -- the same gradients through the chunked WY form of the
  chunked oracle (module ``chunked``), derived by hand step by step; it is the
  algorithm the GPU backward follows and is pinned against ``grad_recurrence``.

Both are pinned by central finite differences of the C token recurrence
(module ``recurrence``), which neither of them uses.

Chunk-level derivation (one chunk, C' rows, chunk-start state H, gradient D of
the chunk-end state; notation of module ``chunked``; P = (Q K^T) * Gam):
  forward      V' = U - W H,  O = scale (diag(gamma) Q H + P V'),
               H_next = gamma_C H + Ktil^T V'
  dV'          = scale P^T dO + Ktil D
  dP           = scale dO V'^T                (lower triangle incl. diagonal)
  dQ           = scale diag(gamma) dO H^T + (dP * Gam) K
  dK           = (dP * Gam)^T Q + diag(dec) V' D^T + diag(beta gamma) Y_W
                 + (dKK + dKK^T) K
  Y_U = A^T dV',  Y_W = A^T dW = -Y_U H^T      (dU = dV', dW = -dV' H^T)
  dV           = diag(beta) Y_U
  dL           = -A^T dV' V'^T                (strict lower triangle; uses
                 dA A^T = dU U^T + dW W^T = dV' V'^T)
  dbeta_r      = <Y_U[r], V[r]> + gamma_r <Y_W[r], K[r]> + sum_s dL_rs KK_rs Gam_rs
  dKK          = dL * beta[:, None] * Gam,   dGam = dP * (Q K^T) + dL * beta[:, None] * KK
  dgamma_r     = <Q[r], scale (dO H^T)[r]> + beta_r <Y_W[r], K[r]>
  ddec_r       = <K[r], (V' D^T)[r]>,   dgamma_C = <D, H>
  dG_r         = dgamma_r gamma_r + sum_s dGam_rs Gam_rs - sum_s dGam_sr Gam_sr
                 - ddec_r dec_r  (+ dgamma_C gamma_C + sum_s ddec_s dec_s at r = C'-1)
  dg_s         = sum_{r >= s} dG_r
  D_prev       = gamma_C D + scale (diag(gamma) Q)^T dO - W^T dV'
with dec = exp(G_{C'-1} - G).  dQ and dK sum over the value heads that share
a q/k head; D_prev of a sequence's first chunk is the gradient of h0.
"""
from __future__ import annotations

import numpy as np

from .chunked import CHUNK, chunk_bounds, chunk_step


def _torch():
    import torch
    return torch


def grad_recurrence(q, k, v, g, beta, h0, cu_seqlens, do, dhT=None, scale=None, block=64,
                    heads=None):
    """Gradients of sum(o * do) + sum(h_T * dh_T) by autograd of the token recurrence.

    q,k [T, h_qk, d_k]; v, do [T, h_v, d_v]; g, beta [T, h_v]; h0, dhT [N, h_v, d_k, d_v]
    or None.  heads: value heads to differentiate (None: all); dq and dk then hold only
    those heads' contributions and the other heads' dv, dg, dbeta, dh0 stay 0.
    Returns float64 numpy (dq, dk, dv, dg, dbeta, dh0); dh0 is returned even when h0 is
    None (the gradient with respect to a zero initial state).
    """
    torch = _torch()
    f64 = lambda a: torch.as_tensor(np.asarray(a, dtype=np.float64))
    q, k, v, g, beta, do = map(f64, (q, k, v, g, beta, do))
    T, h_qk, d_k = q.shape
    h_v, d_v = v.shape[1], v.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(d_k)
    if cu_seqlens is None:
        cu_seqlens = [0, T]
    n_seqs = len(cu_seqlens) - 1
    hs = list(range(h_v)) if heads is None else sorted(heads)
    hidx = torch.tensor(hs, dtype=torch.long)
    imap = torch.tensor([(j * h_qk) // h_v for j in hs], dtype=torch.long)
    dq, dk = torch.zeros_like(q), torch.zeros_like(k)
    dv, dg, dbeta = torch.zeros_like(v), torch.zeros_like(g), torch.zeros_like(beta)
    dh0 = torch.zeros((n_seqs, h_v, d_k, d_v), dtype=torch.float64)

    def run(H, qb, kb, vb, gb, bb):
        """Recurrence over one block for the selected heads.  Returns (o, H_end)."""
        outs = []
        for t in range(qb.shape[0]):
            kt = kb[t, imap]                    # [h, d_k]
            a = torch.exp(gb[t, hidx])[:, None, None]
            b = bb[t, hidx][:, None, None]
            kH = torch.einsum("hk,hkv->hv", kt, H)
            H = a * H - a * b * kt[:, :, None] * kH[:, None, :] + b * kt[:, :, None] * vb[t, hidx][:, None, :]
            outs.append(scale * torch.einsum("hk,hkv->hv", qb[t, imap], H))
        return torch.stack(outs), H

    for n in range(n_seqs):
        bos, eos = int(cu_seqlens[n]), int(cu_seqlens[n + 1])
        H = (torch.zeros((len(hs), d_k, d_v), dtype=torch.float64) if h0 is None
             else f64(h0)[n, hidx].clone())
        starts, ckpt = list(range(bos, eos, block)), []
        with torch.no_grad():  # block-start states
            for a0 in starts:
                ckpt.append(H)
                a1 = min(a0 + block, eos)
                _, H = run(H, q[a0:a1], k[a0:a1], v[a0:a1], g[a0:a1], beta[a0:a1])
        dH = (torch.zeros((len(hs), d_k, d_v), dtype=torch.float64) if dhT is None
              else f64(dhT)[n, hidx].clone())
        for a0, Hs in zip(reversed(starts), reversed(ckpt)):
            a1 = min(a0 + block, eos)
            leaves = [Hs.clone().requires_grad_(True)] + [
                x[a0:a1].clone().requires_grad_(True) for x in (q, k, v, g, beta)]
            o_b, H_end = run(*leaves)
            loss = (o_b * do[a0:a1, hidx]).sum() + (H_end * dH).sum()
            grads = torch.autograd.grad(loss, leaves, allow_unused=True)
            dH = grads[0]
            for acc, gr in zip((dq, dk, dv, dg, dbeta), grads[1:]):
                if gr is not None:
                    acc[a0:a1] += gr
        dh0[n, hidx] = dH
    return tuple(x.numpy() for x in (dq, dk, dv, dg, dbeta, dh0))


def chunk_backward(H, D, qc, kc, vc, gc, bc, doc, scale):
    """Gradients of one chunk, one value head (the derivation in the module docstring).

    H, D [d_k, d_v]: chunk-start state and the gradient of the chunk-end state.
    Returns (dq, dk, dv, dg, dbeta, D_prev).
    """
    cp = gc.shape[0]
    G = np.cumsum(gc)
    gamma = np.exp(G)
    gamma_C = np.exp(G[-1])
    dec = np.exp(G[-1] - G)
    lower_incl = np.tril(np.ones((cp, cp), dtype=bool))
    Gam = np.where(lower_incl, np.exp(np.where(lower_incl, G[:, None] - G[None, :], 0.0)), 0.0)
    KK = kc @ kc.T
    A = np.linalg.inv(np.eye(cp) + np.tril(bc[:, None] * KK * Gam, -1))
    W = A @ ((bc * gamma)[:, None] * kc)
    U = A @ (bc[:, None] * vc)
    Ktil = dec[:, None] * kc
    Vp = U - W @ H
    QK = qc @ kc.T
    P = QK * Gam

    dVp = scale * P.T @ doc + Ktil @ D
    dP = np.where(lower_incl, scale * doc @ Vp.T, 0.0)
    dQs = scale * doc @ H.T
    dgamma = np.sum(qc * dQs, axis=1)
    dq = gamma[:, None] * dQs + (dP * Gam) @ kc
    dk = (dP * Gam).T @ qc
    Z = Vp @ D.T
    dk += dec[:, None] * Z
    ddec = np.sum(kc * Z, axis=1)
    dgamma_C = np.sum(D * H)
    dGam = dP * QK
    YU = A.T @ dVp
    YW = -YU @ H.T
    dv = bc[:, None] * YU
    dk += (bc * gamma)[:, None] * YW
    t2 = np.sum(YW * kc, axis=1)
    dbeta = np.sum(YU * vc, axis=1) + gamma * t2
    dgamma += bc * t2
    dL = np.tril(-A.T @ (dVp @ Vp.T), -1)
    dbeta += np.sum(dL * KK * Gam, axis=1)
    dKK = dL * bc[:, None] * Gam
    dk += (dKK + dKK.T) @ kc
    dGam += dL * bc[:, None] * KK
    E = dGam * Gam
    dG = dgamma * gamma + E.sum(axis=1) - E.sum(axis=0) - ddec * dec
    dG[-1] += dgamma_C * gamma_C + np.sum(ddec * dec)
    dg = np.cumsum(dG[::-1])[::-1]
    D_prev = gamma_C * D + scale * (gamma[:, None] * qc).T @ doc - W.T @ dVp
    return dq, dk, dv, dg, dbeta, D_prev


def grad_chunked(q, k, v, g, beta, h0, cu_seqlens, do, dhT=None, scale=None, C=CHUNK, heads=None):
    """Gradients of sum(o * do) + sum(h_T * dh_T) through the chunked form.

    Same arguments and results as ``grad_recurrence`` (heads: the value heads
    to differentiate, None: all).  Per sequence and value
    head: a forward pass of the chunked scan keeps every chunk-start state, then
    the chunks are differentiated in reverse with ``chunk_backward``.
    """
    q, k, v, g, beta, do = (np.asarray(a, dtype=np.float64) for a in (q, k, v, g, beta, do))
    T, h_qk, d_k = q.shape
    h_v, d_v = v.shape[1], v.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(d_k)
    if cu_seqlens is None:
        cu_seqlens = [0, T]
    n_seqs = len(cu_seqlens) - 1
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    dg, dbeta = np.zeros_like(g), np.zeros_like(beta)
    dh0 = np.zeros((n_seqs, h_v, d_k, d_v))
    for n in range(n_seqs):
        bos, eos = int(cu_seqlens[n]), int(cu_seqlens[n + 1])
        bounds = [(a + bos, b + bos) for a, b in chunk_bounds(eos - bos, C)]
        for j in (range(h_v) if heads is None else sorted(heads)):
            i = (j * h_qk) // h_v
            H = np.zeros((d_k, d_v)) if h0 is None else np.asarray(h0, dtype=np.float64)[n, j].copy()
            states = []
            for a, b in bounds:
                states.append(H)
                _, H = chunk_step(H, q[a:b, i], k[a:b, i], v[a:b, j], g[a:b, j], beta[a:b, j],
                                  scale, want_out=False)
            D = np.zeros((d_k, d_v)) if dhT is None else np.asarray(dhT, dtype=np.float64)[n, j].copy()
            for (a, b), Hs in zip(reversed(bounds), reversed(states)):
                gq, gk, gv, gg, gb, D = chunk_backward(Hs, D, q[a:b, i], k[a:b, i], v[a:b, j],
                                                       g[a:b, j], beta[a:b, j], do[a:b, j], scale)
                dq[a:b, i] += gq
                dk[a:b, i] += gk
                dv[a:b, j] = gv
                dg[a:b, j] = gg
                dbeta[a:b, j] = gb
            dh0[n, j] = D
    return dq, dk, dv, dg, dbeta, dh0
