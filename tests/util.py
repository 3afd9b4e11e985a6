"""Helpers shared by the tests: the parity comparator and the CP segmentation rule.

The segmentation rule is restated here from its documented definition (the
header's gdn_cp_plan comment), independently of the library, so tests can
check the planner and build oracle expectations for warmup mode.
"""
from __future__ import annotations

import math

import numpy as np
import torch

TOL_BF16 = 2e-2   # max|diff| <= 2e-2 * RMS(ref), on top of the bf16 store's half ulp
TOL_STATE = 2e-2  # final state (fp32 output) of the bf16 path


def isqrt(x: int) -> int:
    return math.isqrt(x)


def seg_count(n_chunks: int, lambda_q8: int, cp_off: bool) -> int:
    if cp_off or n_chunks <= 1:
        return 1
    L = max(1, (isqrt(lambda_q8 * lambda_q8 * n_chunks) + 128) // 256)
    return max(1, -(-n_chunks // L))


def segments(n_tokens: int, lambda_q8: int, cp_off: bool):
    N = -(-n_tokens // 64)
    ns = seg_count(N, lambda_q8, cp_off)
    return [((s * N) // ns, ((s + 1) * N) // ns) for s in range(ns)]


def bf16_half_ulp(x: np.ndarray) -> np.ndarray:
    """Half the spacing of bf16 numbers at |x| (8 significant bits)."""
    a = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    return np.exp2(np.floor(np.log2(a)) - 8)


def parity_bf16(out_gpu: torch.Tensor, ref: np.ndarray):
    """(excess over the bf16 rounding allowance, raw max|diff|) / RMS(ref)."""
    g = out_gpu.detach().double().cpu().numpy()
    rms = float(np.sqrt(np.mean(ref ** 2)))
    diff = np.abs(g - ref)
    allowance = bf16_half_ulp(np.maximum(np.abs(ref), np.abs(g)))
    excess = float(np.maximum(diff - allowance, 0.0).max()) / rms
    return excess, float(diff.max()) / rms


def parity_f32(out_gpu: torch.Tensor, ref: np.ndarray) -> float:
    g = out_gpu.detach().double().cpu().numpy()
    rms = float(np.sqrt(np.mean(ref ** 2)))
    return float(np.abs(g - ref).max()) / max(rms, 1e-300)


def to64(t):
    return None if t is None else t.detach().double().cpu().numpy()


def warmup_depths(w, lambda_q8, wmax, tol, rule="fixed"):
    """Per (seq, head, segment) warmup depth by the documented rule: the
    smallest w <= wmax with sum over the w chunks before the segment of
    g + log max(1, |1 - beta ||k||^2|) <= log(the segment's tolerance); a
    window reaching the sequence start runs exactly; None when no depth
    qualifies.  The tolerance is tol ("fixed"), or ("noise") the larger of
    tol and 2^-11 (1 + sum over m = 1..min(wmax, 8, chunks before) of
    min(1, exp(sum over the last m chunks)))."""
    f = to64
    g, beta, k = f(w.g), f(w.beta), f(w.k)
    offs = w.seq_offsets()
    out = {}
    for n in range(len(offs) - 1):
        bos, eos = offs[n], offs[n + 1]
        segs = segments(eos - bos, lambda_q8, False)
        for j in range(w.h_v):
            i = (j * w.h_qk) // w.h_v
            kk = (k[bos:eos, i] ** 2).sum(-1)
            term = g[bos:eos, j] + np.log(np.maximum(1.0, np.abs(1.0 - beta[bos:eos, j] * kk)))
            chunk = lambda c: term[c * 64:(c + 1) * 64].sum()
            for si, (cb, _) in enumerate(segs):
                if si == 0:
                    continue
                thr = math.log(tol)
                if rule == "noise":
                    acc, fl = 0.0, 1.0
                    for m in range(1, min(wmax, 8, cb) + 1):
                        acc += chunk(cb - m)
                        fl += min(1.0, math.exp(acc))
                    thr = max(thr, math.log(fl) - 11 * math.log(2.0))
                acc, wsel = 0.0, None
                for wd in range(1, min(wmax, cb) + 1):
                    acc += chunk(cb - wd)
                    if cb - wd == 0 or acc <= thr:
                        wsel = wd
                        break
                out[(n, j, si)] = wsel
    return out


def auto_lambda_q8(T_list, h_v, sm_count, overhead=3, combine=True):
    """The planner's automatic lambda, restated from its documented rule:
    among lambda = k/8 (k = 1..128) take the smallest (2 x finish of the list
    schedule of the scan's CTAs + 2 x the largest segment count of a sequence:
    a combine step costs about a chunk-time),
    ties to fewer segments.  The schedule: launch order (the segments of every
    sequence, head after head), each CTA taking segment chunks + overhead on
    the first of sm_count slots to free up.  The fp32 path: 2 x SMs slots, no
    overhead, no combine term."""
    best = None
    for q8 in range(32, 4097, 32):
        seglists = [segments(n_tok, q8, False) for n_tok in T_list]
        free = [0] * sm_count
        for _ in range(h_v):
            for sg in seglists:
                for a, b in sg:
                    i = min(range(sm_count), key=free.__getitem__)
                    free[i] += b - a + overhead
        comb = 2 * max(len(sg) for sg in seglists) if combine else 0
        key = (2 * max(free) + comb, sum(len(sg) for sg in seglists))
        if best is None or key < best[0]:
            best = (key, q8)
    return best[1]
