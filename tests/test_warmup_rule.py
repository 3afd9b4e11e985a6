"""The restated warmup-depth rule (the tests' expectation for the kernels'
head modes) against hand arithmetic.

With unit keys and beta in (0, 1) the bound of a chunk is exp(sum of its g).
A constant g = -0.02 gives -1.28 a chunk, so w chunks bound the dropped
history by exp(-1.28 w):
  fixed 1e-4 (log -9.210): w = 8 (-10.24; w = 7 gives -8.96);
  noise floor with a 6-chunk window: 2^-11 (1 + sum_{m=1..6} exp(-1.28 m))
    = 2^-11 * 1.3849 = 6.762e-4 (log -7.299): w = 6 (-7.68; w = 5 gives -6.40);
  with an 8-chunk window the floor hardly moves (1.3851): w = 6 again.
Segments whose first chunk is closer than that to the sequence start restart
from the start (exact, depth = chunks before them).
"""
from __future__ import annotations

import dataclasses
import math

import torch

from gated_deltanet_linear_fwd_gb300.inputs import make_inputs
from tests import util


def _case():
    base = make_inputs(64 * 40 + 9, h_qk=1, h_v=2, seed=12)
    return dataclasses.replace(base, g=torch.full_like(base.g, -0.02))


def test_noise_floor_by_hand():
    fl = 1 + sum(math.exp(-1.28 * m) for m in range(1, 7))
    assert abs(fl - 1.3849) < 1e-4
    assert abs(math.log(fl * 2.0 ** -11) - (-7.299)) < 1e-3


def test_depths_follow_the_hand_values():
    w = _case()
    q8 = 128  # lambda 0.5: 41 chunks -> L = round(0.5 sqrt(41)) = 3, 14 segments
    segs = util.segments(w.T, q8, False)
    assert len(segs) == 14
    for wmax, rule, depth in ((8, "fixed", 8), (6, "fixed", None), (6, "noise", 6), (8, "noise", 6),
                              (5, "noise", None)):
        d = util.warmup_depths(w, q8, wmax, 1e-4, rule)
        for (n, j, s), got in d.items():
            cb = segs[s][0]
            if cb <= (depth if depth is not None else wmax):
                assert got == cb, (wmax, rule, s, got)  # the window reaches the sequence start
            else:
                assert got == depth, (wmax, rule, s, got)
