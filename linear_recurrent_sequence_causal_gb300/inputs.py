"""Seeded synthetic inputs for the PRISM mixer forward pass.

This module only draws random numbers and shapes them: it holds none of the
method's arithmetic (no anchor, no refinement, no recurrence).  Both the CUDA
path (tests, bench) and the CPU oracle read their inputs from here, so the two
see exactly the same values.

Workload recipe (the pages give no sizes; these are the five workloads this
library is measured and checked on):

  q, k ~ N(0, 1), each token's vector L2-normalised over d_k in fp32, then cast
  v    ~ N(0, 1)
  log_alpha = -softplus(N(0, 1)) / 8        (fp32, forget gate alpha = exp(.))
  beta      = sigmoid(N(0, 1))              (fp32, delta-rule strength in (0,1))
  conv_w ~ N(0, 0.5)   (variance 0.5)       [H, w, d_v]; tap j-1 multiplies v_{t-j}
  Wk ~ N(0, 1/d_v)  [H, L, d_k, d_v];  Wp ~ N(0, 1/d_v) [H, L, d_v, d_v]
  wbeta ~ N(0, 1/d_v) [H, L, d_v]
  seq_lens (ragged workload only): integers uniform in [20, 200]

"N(0, x)" is read as variance x.  On bf16 workloads the fp32 parameters
(conv_w, Wk, Wp, wbeta) are rounded to bf16-representable values before either
side sees them, so staging them as bf16 on the GPU is exact.  The draw order is
q, k, v, log_alpha, beta, conv_w, Wk, Wp, wbeta, seq_lens from one torch CPU
generator seeded with the workload's seed.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    dtype: str          # "f32" or "bf16": the I/O type of q, k, v and out
    B: int
    T: int
    H: int
    dk: int
    dv: int
    L: int
    w: int
    chunk: int
    seed: int
    ragged: bool = False
    note: str = ""

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    @property
    def tokens(self) -> int:
        return self.B * self.T


WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", "f32", B=1, T=64, H=1, dk=16, dv=16, L=2, w=4,
                         chunk=16, seed=0, note="tiny fp32 reference case"),
    "lsweep_bf16": Workload("lsweep_bf16", "bf16", B=4, T=1024, H=4, dk=64, dv=64, L=2,
                            w=4, chunk=64, seed=1,
                            note="L sweep {0,1,2,4}; L=0 must equal gated delta rule"),
    "recsys_bf16": Workload("recsys_bf16", "bf16", B=512, T=200, H=2, dk=32, dv=32, L=3,
                            w=4, chunk=32, seed=2, ragged=True,
                            note="recommendation-shaped, right-padded, lengths U[20,200]"),
    "lm_bf16": Workload("lm_bf16", "bf16", B=8, T=4096, H=16, dk=128, dv=128, L=2, w=4,
                        chunk=64, seed=3, note="LM-shaped"),
    "longctx_bf16": Workload("longctx_bf16", "bf16", B=1, T=65536, H=32, dk=128, dv=128,
                             L=4, w=4, chunk=64, seed=4, note="long context"),
    "longctx_h4_bf16": Workload("longctx_h4_bf16", "bf16", B=1, T=65536, H=4, dk=128, dv=128,
                                L=4, w=4, chunk=64, seed=5,
                                note="long context with few heads (the sequence-split scan)"),
}


def get_workload(name: str) -> Workload:
    return WORKLOADS[name]


def _round_to(x: torch.Tensor, dtype: torch.dtype) -> torch.Tensor:
    return x.to(dtype).to(torch.float32)


def generate(wl: Workload, *, L: Optional[int] = None, seed: Optional[int] = None) -> dict:
    """Draw one workload's inputs on the host (torch CPU tensors).

    Returns a dict with q, k, v ([B,T,H,d], the workload's I/O dtype),
    log_alpha, beta ([B,T,H] fp32), conv_w, Wk, Wp, wbeta (fp32) and seq_lens
    ([B] int32, or None when every sequence has length T).
    """
    L = wl.L if L is None else L
    g = torch.Generator().manual_seed(wl.seed if seed is None else seed)
    B, T, H, dk, dv, w = wl.B, wl.T, wl.H, wl.dk, wl.dv, wl.w
    io = wl.torch_dtype

    def unit(shape):
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        x = x / x.norm(dim=-1, keepdim=True).clamp_min(1e-30)
        return x.to(io)

    q = unit((B, T, H, dk))
    k = unit((B, T, H, dk))
    v = torch.randn((B, T, H, dv), generator=g, dtype=torch.float32).to(io)
    log_alpha = -torch.nn.functional.softplus(
        torch.randn((B, T, H), generator=g, dtype=torch.float32)) / 8.0
    beta = torch.sigmoid(torch.randn((B, T, H), generator=g, dtype=torch.float32))
    conv_w = torch.randn((H, w, dv), generator=g, dtype=torch.float32) * (0.5 ** 0.5)
    std = dv ** -0.5
    Wk = torch.randn((H, L, dk, dv), generator=g, dtype=torch.float32) * std
    Wp = torch.randn((H, L, dv, dv), generator=g, dtype=torch.float32) * std
    wbeta = torch.randn((H, L, dv), generator=g, dtype=torch.float32) * std
    if wl.dtype == "bf16":
        conv_w, Wk, Wp, wbeta = (_round_to(t, torch.bfloat16) for t in (conv_w, Wk, Wp, wbeta))
    seq_lens = None
    if wl.ragged:
        lo, hi = min(20, T), T
        seq_lens = torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int32)
    return dict(q=q, k=k, v=v, log_alpha=log_alpha, beta=beta, conv_w=conv_w,
                Wk=Wk, Wp=Wp, wbeta=wbeta, seq_lens=seq_lens)


def random_small(B, T, H, dk, dv, L, w, *, seed=0, dtype=torch.float64, ragged=False,
                 alpha_scale=1.0 / 8.0) -> dict:
    """Small random inputs of any shape (d_k may differ from d_v), for oracle pins.

    Same distributions as the workloads; fp64 by default.
    """
    g = torch.Generator().manual_seed(seed)

    def n(*shape):
        return torch.randn(shape, generator=g, dtype=torch.float64)

    q = n(B, T, H, dk); q = q / q.norm(dim=-1, keepdim=True)
    k = n(B, T, H, dk); k = k / k.norm(dim=-1, keepdim=True)
    v = n(B, T, H, dv)
    log_alpha = -torch.nn.functional.softplus(n(B, T, H)) * alpha_scale
    beta = torch.sigmoid(n(B, T, H))
    conv_w = n(H, w, dv) * 0.5 ** 0.5
    Wk = n(H, L, dk, dv) * dv ** -0.5
    Wp = n(H, L, dv, dv) * dv ** -0.5
    wbeta = n(H, L, dv) * dv ** -0.5
    seq_lens = None
    if ragged:
        seq_lens = torch.randint(1, T + 1, (B,), generator=g, dtype=torch.int32)
    out = dict(q=q, k=k, v=v, log_alpha=log_alpha, beta=beta, conv_w=conv_w, Wk=Wk,
               Wp=Wp, wbeta=wbeta, seq_lens=seq_lens)
    return {key: (val.to(dtype) if val is not None and val.is_floating_point() else val)
            for key, val in out.items()}
