"""Seeded synthetic inputs for the gated delta rule workloads.

This module only draws random numbers and lays them out; it contains none of
the method's arithmetic, so both the CUDA path and the CPU oracle can be fed
from it.

Distributions (the workloads' stated recipe):
  q, k   ~ N(0, 1), L2-normalised over d_k per (token, head) in fp32, then
           cast to the io dtype (the cast values are what every consumer sees)
  v      ~ N(0, 1), cast to the io dtype
  g      ~ -U(0.001, 0.1)  (log-gate, alpha = exp(g)), fp32
  beta   = sigmoid(N(0, 1)), fp32
  dO     ~ N(0, 1), fp32 (upstream gradient)
  h0     ~ N(0, h0_std^2), fp32 (zero when h0_std == 0)
  varlen lengths: integers ~ U[lo, hi] inclusive, seeded.
All draws come from one CPU ``torch.Generator`` seeded with ``seed``.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional, Sequence

import torch


@dataclass
class GdnInputs:
    q: torch.Tensor            # [n_tok, H, d_k] io dtype
    k: torch.Tensor            # [n_tok, H, d_k] io dtype
    v: torch.Tensor            # [n_tok, H, d_v] io dtype
    g: torch.Tensor            # [n_tok, H] fp32
    beta: torch.Tensor         # [n_tok, H] fp32
    cu_seqlens: torch.Tensor   # [n_seq + 1] int32
    h0: Optional[torch.Tensor]  # [n_seq, H, d_k, d_v] fp32 or None
    dO: Optional[torch.Tensor]  # [n_tok, H, d_v] fp32 or None

    @property
    def seqlens(self):
        cu = self.cu_seqlens.tolist()
        return [cu[i + 1] - cu[i] for i in range(len(cu) - 1)]

    def to(self, device):
        f = lambda t: None if t is None else t.to(device)
        return GdnInputs(f(self.q), f(self.k), f(self.v), f(self.g), f(self.beta),
                         f(self.cu_seqlens), f(self.h0), f(self.dO))


def varlen_lengths(n_seq: int, lo: int, hi: int, seed: int = 0) -> list[int]:
    gen = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, (n_seq,), generator=gen).tolist()


def make_inputs(seqlens: Sequence[int], H: int, dk: int, dv: int,
                io_dtype: torch.dtype = torch.bfloat16, seed: int = 0,
                h0_std: float = 0.0, with_grad: bool = False,
                g_range=(0.001, 0.1)) -> GdnInputs:
    gen = torch.Generator().manual_seed(seed)
    n_tok = int(sum(seqlens))
    n_seq = len(seqlens)
    q = torch.randn(n_tok, H, dk, generator=gen)
    k = torch.randn(n_tok, H, dk, generator=gen)
    q = q / q.norm(dim=-1, keepdim=True).clamp_min(1e-30)
    k = k / k.norm(dim=-1, keepdim=True).clamp_min(1e-30)
    v = torch.randn(n_tok, H, dv, generator=gen)
    lo, hi = g_range
    g = -(torch.rand(n_tok, H, generator=gen) * (hi - lo) + lo)
    beta = torch.sigmoid(torch.randn(n_tok, H, generator=gen))
    h0 = None
    if h0_std > 0:
        h0 = torch.randn(n_seq, H, dk, dv, generator=gen) * h0_std
    dO = torch.randn(n_tok, H, dv, generator=gen) if with_grad else None
    cu = torch.zeros(n_seq + 1, dtype=torch.int32)
    if n_seq:
        cu[1:] = torch.cumsum(torch.tensor(list(seqlens), dtype=torch.int64), 0).to(torch.int32)
    return GdnInputs(q.to(io_dtype).contiguous(), k.to(io_dtype).contiguous(),
                     v.to(io_dtype).contiguous(), g.contiguous().float(),
                     beta.contiguous().float(), cu, h0, dO)


def make_decode_tokens(n_seq: int, H: int, dk: int, dv: int, n_steps: int,
                       io_dtype: torch.dtype = torch.bfloat16, seed: int = 1) -> GdnInputs:
    """Tokens for `n_steps` decode steps, laid out [n_steps * n_seq, H, ...]
    (step-major), with the same distributions."""
    return make_inputs([1] * (n_steps * n_seq), H, dk, dv, io_dtype=io_dtype, seed=seed)
