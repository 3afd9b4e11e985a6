"""Chunked closed form of the GDN forward, float64 numpy.  TEST INFRASTRUCTURE ONLY.

Only tests/, ``__graft_entry__.smoke()`` and bench.py's cpu_baseline leg may use
this module.  It shares no code with the CUDA path.

This is the second CPU implementation: the same layer evaluated chunk by
chunk, step by step in the order the FlashQLA pages describe the chunked
prefill flow (FlashQLA pages, section "Optimising GDN chunked prefill": the
flow works through per-chunk intermediates W, U and the chunk-boundary state
S; section "AutoCP": a sequence is split into segments whose start states are
combined exactly through a correction term M, or approximated by a warmup
restart).  The per-chunk algebra is the WY representation of the gated delta
rule (Yang, Kautz and Hatamizadeh, "Gated Delta Networks", ICLR 2025, section
"Chunkwise parallel form"; Yang et al., "Parallelizing Linear Transformers
with the Delta Rule over Sequence Length", NeurIPS 2024, section "WY
representation").  Library primitives (matmul, a triangular inverse, cumsum)
serve as steps; nothing is blocked, fused or reordered beyond those
equations.

State orientation: H = S^T, d_k x d_v, the stored layout [n_seqs, h_v, d_k, d_v].

Per chunk of C' <= C rows (row r = token chunk_start + r):
  G_r      = sum_{s<=r} g_s                    (inclusive cumulative gate)
  gamma_r  = exp(G_r),  gamma_C = exp(G_{C'-1})
  Gam_rs   = exp(G_r - G_s) for s <= r, else 0  (inclusive decay mask)
  L        = strict_lower(diag(beta) (K K^T) * Gam)
  A        = (I + L)^{-1}
  W        = A diag(beta * gamma) K,   U = A diag(beta) V
  V'       = U - W H
  O        = scale * (diag(gamma) Q H + (Q K^T * Gam) V')
  H_next   = gamma_C H + Ktil^T V',   Ktil = diag(exp(G_{C'-1} - G)) K

The row scaling Ktil is what the exact chunk update needs (each token's key is
decayed from its own position to the chunk end); it follows from unrolling
the recurrence over the chunk and is pinned against the token recurrence.

Segment transition (exact context parallelism): over a run of chunks the map
H_start -> H_end is affine, H_end = M H_start + H_loc.  Running the chunk
update on the augmented state X = [M | H_loc], started from [I | 0] with the
value part [0 | U], yields both (each chunk: X <- gamma_C X + Ktil^T([0|U] - W X)).
"""
from __future__ import annotations

import numpy as np

CHUNK = 64


def chunk_local(kc: np.ndarray, vc: np.ndarray, gc: np.ndarray, bc: np.ndarray):
    """Gate cumsum and WY form of one chunk (the chunk-local steps).

    kc [C', d_k], vc [C', d_v], gc/bc [C'] float64.
    Returns G, gamma, Gam (inclusive decay mask), W, U, Ktil.
    """
    cp = gc.shape[0]
    G = np.cumsum(gc)
    gamma = np.exp(G)
    lower_incl = np.tril(np.ones((cp, cp), dtype=bool))
    diff = np.where(lower_incl, G[:, None] - G[None, :], 0.0)
    Gam = np.where(lower_incl, np.exp(diff), 0.0)
    L = np.tril(bc[:, None] * (kc @ kc.T) * Gam, -1)
    A = np.linalg.inv(np.eye(cp) + L)
    W = A @ ((bc * gamma)[:, None] * kc)
    U = A @ (bc[:, None] * vc)
    Ktil = np.exp(G[-1] - G)[:, None] * kc
    return G, gamma, Gam, W, U, Ktil


def chunk_step(H, qc, kc, vc, gc, bc, scale, want_out=True):
    """One chunk of the state scan with its output.  Returns (O or None, H_next)."""
    G, gamma, Gam, W, U, Ktil = chunk_local(kc, vc, gc, bc)
    Vp = U - W @ H
    O = None
    if want_out:
        O = scale * ((gamma[:, None] * qc) @ H + ((qc @ kc.T) * Gam) @ Vp)
    H_next = np.exp(G[-1]) * H + Ktil.T @ Vp
    return O, H_next


def chunk_bounds(n_tokens: int, C: int = CHUNK):
    """Chunks start at the sequence start; the last one may be partial."""
    return [(s, min(s + C, n_tokens)) for s in range(0, n_tokens, C)]


def scan_head(q, k, v, g, beta, H0, scale, C=CHUNK, chunk_range=None, out=None, out_from=None):
    """Chunked scan for one sequence and one value head.

    q,k [T, d_k]; v [T, d_v]; g,beta [T]; H0 [d_k, d_v].
    chunk_range: (c_begin, c_end) chunk indices to run (default: all).
    Outputs of chunks with index >= out_from (default c_begin) are written
    into out [T, d_v] when out is given.  Returns the state after c_end.
    """
    bounds = chunk_bounds(q.shape[0], C)
    cb, ce = (0, len(bounds)) if chunk_range is None else chunk_range
    if out_from is None:
        out_from = cb
    H = H0.copy()
    for c in range(cb, ce):
        a, b = bounds[c]
        want = out is not None and c >= out_from
        O, H = chunk_step(H, q[a:b], k[a:b], v[a:b], g[a:b], beta[a:b], scale, want)
        if want:
            out[a:b] = O
    return H


def segment_transition(k, v, g, beta, chunk_range, C=CHUNK):
    """(M, H_loc) of a run of chunks: H_end = M @ H_start + H_loc."""
    d_k, d_v = k.shape[1], v.shape[1]
    bounds = chunk_bounds(k.shape[0], C)
    X = np.concatenate([np.eye(d_k), np.zeros((d_k, d_v))], axis=1)
    for c in range(*chunk_range):
        a, b = bounds[c]
        G, gamma, Gam, W, U, Ktil = chunk_local(k[a:b], v[a:b], g[a:b], beta[a:b])
        Uaug = np.concatenate([np.zeros((b - a, d_k)), U], axis=1)
        X = np.exp(G[-1]) * X + Ktil.T @ (Uaug - W @ X)
    return X[:, :d_k], X[:, d_k:]


def gdn_fwd_chunked(q, k, v, g, beta, h0, cu_seqlens, scale=None, C=CHUNK,
                    segments=None, warmup_chunks=None, warmup_heads=None):
    """Whole forward in the chunked form, optionally context-parallel.

    q,k [T, h_qk, d_k]; v [T, h_v, d_v]; g,beta [T, h_v]; h0 [N, h_v, d_k, d_v] or None.
    segments: per sequence, a list of (c_begin, c_end) chunk ranges covering
      the sequence in order (None: one segment per sequence).
    warmup_chunks / warmup_heads: segments after the first of a head in
      warmup_heads (a set of (seq, head) or of head indices; None: all heads)
      restart from a zero state warmup_chunks chunks before their start
      instead of taking the exactly combined start state.  warmup_chunks is
      an int, or a dict {(seq, head, segment): depth} giving each segment its
      own depth.  A restart clipped at the sequence start runs exactly from h0.
    Returns (o [T, h_v, d_v], hT [N, h_v, d_k, d_v]).
    """
    T, h_qk, d_k = q.shape
    h_v, d_v = v.shape[1], v.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(d_k)
    n_seqs = len(cu_seqlens) - 1
    o = np.zeros((T, h_v, d_v))
    hT = np.zeros((n_seqs, h_v, d_k, d_v))
    for n in range(n_seqs):
        bos, eos = int(cu_seqlens[n]), int(cu_seqlens[n + 1])
        n_chunks = len(chunk_bounds(eos - bos, C))
        segs = [(0, n_chunks)] if segments is None else list(segments[n])
        for j in range(h_v):
            i = (j * h_qk) // h_v
            qs, ks = q[bos:eos, i], k[bos:eos, i]
            vs, gs, bs = v[bos:eos, j], g[bos:eos, j], beta[bos:eos, j]
            H0 = np.zeros((d_k, d_v)) if h0 is None else h0[n, j]
            out = np.zeros((eos - bos, d_v))
            use_warm = warmup_chunks is not None and (
                warmup_heads is None or j in warmup_heads or (n, j) in warmup_heads)
            if use_warm:
                H = H0
                for si, (cb, ce) in enumerate(segs):
                    wd = (warmup_chunks[(n, j, si)] if isinstance(warmup_chunks, dict) and si > 0
                          else warmup_chunks)
                    if si == 0 or cb - wd <= 0:
                        Hs = scan_head(qs, ks, vs, gs, bs, H0, scale, C, (0, cb)) if cb > 0 else H0
                    else:
                        Hs = scan_head(qs, ks, vs, gs, bs, np.zeros((d_k, d_v)), scale, C,
                                       (cb - wd, cb))
                    H = scan_head(qs, ks, vs, gs, bs, Hs, scale, C, (cb, ce), out=out)
            else:
                # exact: local transitions, exact combine, then the scan per segment
                trans = [segment_transition(ks, vs, gs, bs, sr, C) for sr in segs]
                starts = [H0]
                for (M, Hloc) in trans[:-1]:
                    starts.append(M @ starts[-1] + Hloc)
                for (sr, Hs) in zip(segs, starts):
                    H = scan_head(qs, ks, vs, gs, bs, Hs, scale, C, sr, out=out)
            o[bos:eos, j] = out
            hT[n, j] = H
    return o, hT
