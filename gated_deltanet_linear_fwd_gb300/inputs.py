"""Seeded synthetic GDN inputs shared by the CUDA path's tests/bench and the oracle.

This module holds no arithmetic of the method: it only draws tensors with the
shapes and value distributions of the FlashQLA pages' forward benchmark
(pages, section "Benchmarks": batch x seqlen = 1 x 32768 with the (h_qk, h_v)
head sweep of the table) and of the tiny and long varlen cases.  All draws
come from one CPU ``torch.Generator`` per workload, so the same seed gives the
same tensors on any host.

Recipe (per workload):
  q, k  ~ N(0, 1) fp32, L2-normalised over d_k, then cast (bf16 by default)
  v     ~ N(0, 1), cast
  beta  = sigmoid(N(0, 1)) fp32                       [T, h_v]
  g     tiny:  logsigmoid(N(3, 1))                    [T, h_v]
        mix:   a seeded permutation picks round(0.7 h_v) fast-decay heads,
               g = logsigmoid(N(1, 0.5)) there and logsigmoid(N(6, 0.5))
               on the other heads (pages: on 60-80 % of heads old tokens
               fade quickly)
  h0    optional: bf16(0.1 * N(0, 1)) stored fp32     [N, h_v, d_k, d_v]
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import torch
import torch.nn.functional as F

D_K = 128
D_V = 128


@dataclasses.dataclass
class Workload:
    name: str
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    g: torch.Tensor
    beta: torch.Tensor
    h0: Optional[torch.Tensor]
    cu_seqlens: Optional[torch.Tensor]  # int32 [N+1] or None (one sequence)
    h_qk: int
    h_v: int
    fast_heads: Sequence[int]

    @property
    def T(self) -> int:
        return self.q.shape[0]

    @property
    def n_seqs(self) -> int:
        return 1 if self.cu_seqlens is None else self.cu_seqlens.numel() - 1

    def seq_offsets(self):
        if self.cu_seqlens is None:
            return [0, self.T]
        return [int(x) for x in self.cu_seqlens.tolist()]

    def to(self, device) -> "Workload":
        mv = lambda t: None if t is None else t.to(device)
        return dataclasses.replace(self, q=mv(self.q), k=mv(self.k), v=mv(self.v), g=mv(self.g),
                                   beta=mv(self.beta), h0=mv(self.h0),
                                   cu_seqlens=mv(self.cu_seqlens))


def make_inputs(n_tokens: int | None = None, h_qk: int = 2, h_v: int = 4, seed: int = 0,
                g_kind: str = "mix", with_h0: bool = False, cu_seqlens: Sequence[int] | None = None,
                dtype: torch.dtype = torch.bfloat16, name: str = "custom", d_k: int = D_K,
                d_v: int = D_V, h0_std: float = 0.1) -> Workload:
    """Draw one workload.  Either n_tokens (one sequence) or cu_seqlens (varlen)."""
    if cu_seqlens is not None:
        cu = [int(x) for x in cu_seqlens]
        T = cu[-1]
        n_seqs = len(cu) - 1
    else:
        T = int(n_tokens)
        cu = None
        n_seqs = 1
    gen = torch.Generator().manual_seed(seed)
    q = torch.randn(T, h_qk, d_k, generator=gen)
    k = torch.randn(T, h_qk, d_k, generator=gen)
    q = F.normalize(q, dim=-1).to(dtype)
    k = F.normalize(k, dim=-1).to(dtype)
    v = torch.randn(T, h_v, d_v, generator=gen).to(dtype)
    beta = torch.sigmoid(torch.randn(T, h_v, generator=gen))
    fast: list[int] = []
    if g_kind == "tiny":
        g = F.logsigmoid(torch.randn(T, h_v, generator=gen) + 3.0)
    elif g_kind == "mix":
        perm = torch.randperm(h_v, generator=gen)
        fast = sorted(int(x) for x in perm[: round(0.7 * h_v)])
        mean = torch.full((h_v,), 6.0)
        mean[fast] = 1.0
        g = F.logsigmoid(mean[None, :] + 0.5 * torch.randn(T, h_v, generator=gen))
    elif g_kind == "zero":  # alpha = 1
        g = torch.zeros(T, h_v)
    else:
        raise ValueError(f"unknown g_kind {g_kind}")
    h0 = None
    if with_h0:
        h0 = (h0_std * torch.randn(n_seqs, h_v, d_k, d_v, generator=gen)).to(torch.bfloat16).float()
    cu_t = None if cu is None else torch.tensor(cu, dtype=torch.int32)
    return Workload(name, q, k, v, g.float().contiguous(), beta.float().contiguous(), h0, cu_t,
                    h_qk, h_v, fast)


# The standard workloads: the tiny parity case, the three 1 x 32768 rows of
# the pages' benchmark table, a long packed varlen batch, and a batch of 8
# sequences x 32 value heads that fills the GPU without context parallelism.
WORKLOADS = {
    "tiny_T512_h2x4": dict(n_tokens=512, h_qk=2, h_v=4, seed=0, g_kind="tiny"),
    "T32768_h2x8": dict(n_tokens=32768, h_qk=2, h_v=8, seed=1, g_kind="mix"),
    "T32768_h8x24_h0": dict(n_tokens=32768, h_qk=8, h_v=24, seed=2, g_kind="mix", with_h0=True),
    "T32768_h16x16": dict(n_tokens=32768, h_qk=16, h_v=16, seed=3, g_kind="mix"),
    "varlen4_T348160_h2x8": dict(cu_seqlens=[0, 262144, 327680, 344064, 348160], h_qk=2, h_v=8,
                                 seed=4, g_kind="mix"),
    # a batch wide enough to fill the GPU without context parallelism (8 x 32 = 256 chains)
    "batch8_T4096_h8x32": dict(cu_seqlens=[4096 * i for i in range(9)], h_qk=8, h_v=32, seed=5, g_kind="mix"),
}


def workload(name: str, dtype: torch.dtype = torch.bfloat16) -> Workload:
    return make_inputs(name=name, dtype=dtype, **WORKLOADS[name])


def make_output_grads(w: Workload, seed: int = 100, with_dhT: bool = True, dhT_std: float = 0.1,
                      dtype: torch.dtype = torch.bfloat16):
    """Seeded upstream gradients for the backward: d_out ~ N(0, 1) like v (cast),
    d_final_state ~ dhT_std * N(0, 1) fp32 [N, h_v, d_k, d_v] (or None)."""
    gen = torch.Generator().manual_seed(seed)
    d_out = torch.randn(w.v.shape, generator=gen).to(dtype)
    dhT = None
    if with_dhT:
        dhT = dhT_std * torch.randn(w.n_seqs, w.h_v, w.q.shape[-1], w.v.shape[-1], generator=gen)
    return d_out, dhT
