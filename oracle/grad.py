"""Gradients of the PRISM mixer forward pass (fp64, CPU), the reference for the GPU
backward pass.

TEST INFRASTRUCTURE ONLY: the tests and the benchmark's CPU-baseline leg are the only
callers.  The CUDA path never imports or runs anything here.

``forward_torch`` restates the token-by-token recurrence of "Technical Summary: PRISM
(Parallel Residual Iterative Sequence Model)", §2.1 (the causal ShortConv anchor) and
§2.2 (the L-step input-anchored refinement, the rank-L write and the gated delta-rule
state update S_t = S_(t-1) A_t + B_t with o_t = S_t q_t), with the readings the C oracle
uses (the Gated DeltaNet base write beta v k^T kept in B_t, r^(1) = v - u, beta^(l) =
sigmoid(w_beta^(l) . u), k^(l) normalised, exact erf GELU), in differentiable torch fp64
operations, vectorised over (b, h) and looping over tokens.  ``backward`` differentiates
the scalar  sum(out * d_out) + sum(final_state * d_final_state)  with torch.autograd (a
library primitive applied to that definition).

Pins (``tests/oracle_pins.py``): ``forward_torch`` equals the C oracle's forward to
rounding; every gradient equals central finite differences of the C oracle (an
independent implementation) along random directions; dq_t = S_t^T do_t with S_t taken
from prefix runs of the C oracle.
"""
from __future__ import annotations

import math

import numpy as np
import torch

NORM_EPS = 1e-6
GRAD_KEYS = ("q", "k", "v", "log_alpha", "beta", "conv_w", "Wk", "Wp", "wbeta")


def _t64(x):
    if x is None:
        return None
    if isinstance(x, torch.Tensor):
        return x.detach().to("cpu", torch.float64)
    return torch.as_tensor(np.asarray(x, dtype=np.float64))


def forward_torch(p: dict, L: int, *, seq_lens=None, identity_act: bool = False):
    """out [B,T,H,dv] and final_state [B,H,dv,dk] from fp64 tensors in ``p`` (keys as
    ``GRAD_KEYS``); padding tokens (t >= seq_lens[b]) leave the state unchanged and
    output zero (selected, not multiplied)."""
    q, k, v = p["q"], p["k"], p["v"]
    la, be = p["log_alpha"], p["beta"]
    conv_w, Wk, Wp, wb = p["conv_w"], p["Wk"][:, :L], p["Wp"][:, :L], p["wbeta"][:, :L]
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    w = conv_w.shape[1]
    lens = torch.full((B,), T, dtype=torch.int64) if seq_lens is None else \
        torch.as_tensor(np.asarray(seq_lens), dtype=torch.int64).clamp(0, T)
    S = torch.zeros((B, H, dv, dk), dtype=torch.float64)
    eye = torch.eye(dk, dtype=torch.float64)
    outs = []
    for t in range(T):
        live = (t < lens).view(B, 1, 1, 1)
        vt, kt, qt = v[:, t], k[:, t], q[:, t]                  # [B,H,d]
        # causal ShortConv anchor: u_t = sum_{j=1..w} c_j (.) v_(t-j), zero before t = 0
        u = torch.zeros((B, H, dv), dtype=torch.float64)
        for j in range(1, w + 1):
            if t - j >= 0:
                u = u + conv_w[:, j - 1].unsqueeze(0) * v[:, t - j]
        r = vt - u
        Bw = be[:, t].view(B, H, 1, 1) * vt.unsqueeze(-1) * kt.unsqueeze(-2)
        for l in range(L):
            kh = torch.einsum("hab,xhb->xha", Wk[:, l], u)
            kl = kh / torch.sqrt((kh * kh).sum(-1, keepdim=True) + NORM_EPS)
            pl = torch.einsum("hab,xhb->xha", Wp[:, l], u)
            bl = torch.sigmoid((wb[:, l].unsqueeze(0) * u).sum(-1))
            x = pl * r
            d = x if identity_act else 0.5 * x * (1.0 + torch.erf(x / math.sqrt(2.0)))
            r = r - d
            Bw = Bw + bl.view(B, H, 1, 1) * d.unsqueeze(-1) * kl.unsqueeze(-2)
        A = torch.exp(la[:, t]).view(B, H, 1, 1) * (
            eye - be[:, t].view(B, H, 1, 1) * kt.unsqueeze(-1) * kt.unsqueeze(-2))
        S_new = S @ A + Bw
        S = torch.where(live, S_new, S)
        o = torch.einsum("xhab,xhb->xha", S, qt)
        outs.append(torch.where(live[..., 0], o, torch.zeros_like(o)))
    return torch.stack(outs, dim=1), S


def backward(inp: dict, d_out, d_final_state=None, *, L: int | None = None,
             identity_act: bool = False):
    """Gradients (fp64 numpy, same shapes as the inputs) of
    sum(out * d_out) + sum(final_state * d_final_state) with respect to every input in
    ``GRAD_KEYS``."""
    p = {n: _t64(inp[n]).clone().requires_grad_(True) for n in GRAD_KEYS}
    if L is None:
        L = p["Wk"].shape[1]
    out, S = forward_torch(p, L, seq_lens=inp.get("seq_lens"), identity_act=identity_act)
    loss = (out * _t64(d_out)).sum()
    if d_final_state is not None:
        loss = loss + (S * _t64(d_final_state)).sum()
    grads = torch.autograd.grad(loss, [p[n] for n in GRAD_KEYS], allow_unused=True)
    res = {}
    for n, g in zip(GRAD_KEYS, grads):
        res[n] = np.zeros(tuple(p[n].shape)) if g is None else g.numpy()
    return res
