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
