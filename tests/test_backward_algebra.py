"""The adjoint recursion that the CUDA backward kernels evaluate, restated in fp64 numpy
and checked against the autograd gradient oracle (CPU only).

This freezes the backward kernels' algebra before any GPU code runs.  It is a test
artefact: the CUDA path does not use it.

Forward, per live token ("Technical Summary: PRISM", §2.1 and §2.2, with the readings of
the oracle): u = sum_j c_j (.) v_(t-j); r_1 = v - u; per step l: k^_l = Wk_l u,
n_l = 1/sqrt(|k^_l|^2 + 1e-6), k_l = n_l k^_l, p_l = Wp_l u, b_l = sigmoid(wb_l . u),
x_l = p_l (.) r_l, delta_l = GELU(x_l), r_(l+1) = r_l - delta_l, D_l = b_l delta_l;
z = S_(t-1) k;  S_t = alpha (S_(t-1) - beta z k^T) + beta v k^T + sum_l D_l k_l^T;
o_t = S_t q_t.

Reverse, per live token, with dS the cotangent of S_t (do_t q_t^T added first):
  y = dS k,  y_l = dS k_l
  dq  = S_t^T do
  dv  = beta y                                   (base write; the anchor adds below)
  dbeta = v . y - alpha z . y
  dlog_alpha = alpha (<S_(t-1), dS> - beta z . y)
  dk  = dS^T (beta v - alpha beta z) - alpha beta S_(t-1)^T y
  dD_l = y_l,  dk_l = dS^T D_l
  dS <- alpha (dS - beta y k^T)
then the refinement chain backwards (l = L-1 .. 0, dr = 0 entering):
  g = b_l dD_l - dr;  dx = g (.) GELU'(x_l);  dp_l = dx (.) r_l;  dr <- dr + dx (.) p_l
  dz_l = (delta_l . dD_l) b_l (1 - b_l);  dk^_l = n_l (dk_l - k_l (k_l . dk_l))
  du += Wk_l^T dk^_l + Wp_l^T dp_l + dz_l wb_l;  dWk_l += dk^_l u^T, dWp_l += dp_l u^T,
  dwb_l += dz_l u
and r_1 = v - u gives dv += dr, du -= dr; the anchor gives dc_j += du_t (.) v_(t-j) and
dv_(t-j) += c_j (.) du_t.

As in the kernels, the state forward keeps S only every ``block`` tokens and the reverse
sweep recomputes each block's states from its checkpoint; the rows of S are split into
``rs`` slices that evolve independently (a row of S_t depends only on the same row of
S_(t-1), and so does a row of the dS step), and the column sums (dq, dk, dk_l, dbeta,
dlog_alpha) are per-slice partials added in slice order.
"""
import math

import numpy as np
import pytest
import scipy.special
import scipy.stats

from linear_recurrent_sequence_causal_gb300.inputs import random_small
from oracle import grad as G

NORM_EPS = 1e-6


def _refine_forward(u, v, Wk, Wp, wb, identity_act):
    """Per-token refinement quantities for one (b, h) at one token."""
    L = Wk.shape[0]
    r = v - u
    st = []
    for l in range(L):
        kh = Wk[l] @ u
        n = 1.0 / math.sqrt(kh @ kh + NORM_EPS)
        p = Wp[l] @ u
        b = scipy.special.expit(wb[l] @ u)
        x = p * r
        d = x if identity_act else x * scipy.stats.norm.cdf(x)
        st.append(dict(kh=kh, n=n, k=kh * n, p=p, b=b, x=x, r=r, delta=d, D=b * d))
        r = r - d
    return st


def refine_backward(st, dD, dkl, u, Wk, Wp, wb, g, h, identity_act):
    """The refinement chain of one token backwards, from the cotangents dD[l] of the write
    values D_l and dkl[l] of the directions k_l.  Adds the weight gradients of head h to
    ``g`` and returns (dr_1, du): the cotangent of r^(1) and the projections' share of the
    anchor's cotangent."""
    dv = u.shape[0]
    dr = np.zeros(dv)
    du = np.zeros(dv)
    for l in range(len(st) - 1, -1, -1):
        s = st[l]
        gd = s["b"] * dD[l] - dr
        gp = np.ones(dv) if identity_act else \
            scipy.stats.norm.cdf(s["x"]) + s["x"] * scipy.stats.norm.pdf(s["x"])
        dx = gd * gp
        dp = dx * s["r"]
        dr = dr + dx * s["p"]
        dz = (s["delta"] @ dD[l]) * s["b"] * (1.0 - s["b"])
        dkh = s["n"] * (dkl[l] - s["k"] * (s["k"] @ dkl[l]))
        du += Wk[l].T @ dkh + Wp[l].T @ dp + dz * wb[l]
        g["Wk"][h, l] += np.outer(dkh, u)
        g["Wp"][h, l] += np.outer(dp, u)
        g["wbeta"][h, l] += dz * u
    return dr, du


def adjoint(inp, d_out, d_fs, *, identity_act=False, block=16, rs=1):
    f = {n: (np.asarray(inp[n], dtype=np.float64) if inp[n] is not None else None)
         for n in G.GRAD_KEYS}
    q, k, v, la, be = f["q"], f["k"], f["v"], f["log_alpha"], f["beta"]
    cw, Wk, Wp, wb = f["conv_w"], f["Wk"], f["Wp"], f["wbeta"]
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    w = cw.shape[1]
    lens = [T] * B if inp.get("seq_lens") is None else [int(x) for x in inp["seq_lens"]]
    g = {n: np.zeros_like(f[n]) for n in G.GRAD_KEYS}
    rows = np.array_split(np.arange(dv), rs)
    for b in range(B):
        n_tok = lens[b]
        for h in range(H):
            # refinement forward and per-token write terms
            u = np.zeros((n_tok, dv))
            for t in range(n_tok):
                for j in range(1, w + 1):
                    if t - j >= 0:
                        u[t] += cw[h, j - 1] * v[b, t - j, h]
            ref = [_refine_forward(u[t], v[b, t, h], Wk[h], Wp[h], wb[h], identity_act)
                   for t in range(n_tok)]
            alpha = np.exp(la[b, :, h])

            def step(S, t):
                kt = k[b, t, h]
                Sn = alpha[t] * (S - be[b, t, h] * np.outer(S @ kt, kt))
                Sn += be[b, t, h] * np.outer(v[b, t, h], kt)
                for s in ref[t]:
                    Sn += np.outer(s["D"], s["k"])
                return Sn

            # state forward with a checkpoint at the start of every block
            ckpt = {}
            S = np.zeros((dv, dk))
            for t in range(n_tok):
                if t % block == 0:
                    ckpt[t] = S.copy()
                S = step(S, t)
            dS = np.zeros((dv, dk)) if d_fs is None else np.array(d_fs[b, h], dtype=np.float64)
            du = np.zeros((n_tok, dv))
            for t0 in sorted(ckpt, reverse=True):
                t1 = min(t0 + block, n_tok)
                states = [ckpt[t0]]                 # S_(t0-1), S_t0, ..., S_(t1-1)
                for t in range(t0, t1):
                    states.append(step(states[-1], t))
                for t in range(t1 - 1, t0 - 1, -1):
                    Sp, St = states[t - t0], states[t - t0 + 1]
                    kt, qt, vt = k[b, t, h], q[b, t, h], v[b, t, h]
                    a, bt = alpha[t], be[b, t, h]
                    do = d_out[b, t, h]
                    dS = dS + np.outer(do, qt)
                    acc = dict(dq=np.zeros(dk), dk=np.zeros(dk), dbeta=0.0, dla=0.0,
                               dkl=[np.zeros(dk) for _ in ref[t]])
                    dv_t = np.zeros(dv)
                    dD = np.zeros((len(ref[t]), dv))
                    for rsl in rows:                 # one row slice at a time
                        S_r, Sp_r, dS_r = St[rsl], Sp[rsl], dS[rsl]
                        y = dS_r @ kt
                        z = Sp_r @ kt
                        acc["dq"] += S_r.T @ do[rsl]
                        dv_t[rsl] += bt * y
                        acc["dbeta"] += vt[rsl] @ y - a * (z @ y)
                        acc["dla"] += a * (np.sum(Sp_r * dS_r) - bt * (z @ y))
                        acc["dk"] += dS_r.T @ (bt * vt[rsl] - a * bt * z) - a * bt * (Sp_r.T @ y)
                        for l, s in enumerate(ref[t]):
                            dD[l, rsl] = dS_r @ s["k"]
                            acc["dkl"][l] += dS_r.T @ s["D"][rsl]
                        dS[rsl] = a * (dS_r - bt * np.outer(y, kt))
                    g["q"][b, t, h] = acc["dq"]
                    g["k"][b, t, h] = acc["dk"]
                    g["beta"][b, t, h] = acc["dbeta"]
                    g["log_alpha"][b, t, h] = acc["dla"]
                    # refinement chain backwards
                    dr, dut = refine_backward(ref[t], dD, acc["dkl"], u[t], Wk[h], Wp[h], wb[h],
                                              g, h, identity_act)
                    dv_t += dr
                    dut -= dr
                    g["v"][b, t, h] += dv_t
                    du[t] = dut
            # the anchor, transposed
            for t in range(n_tok):
                for j in range(1, w + 1):
                    if t - j >= 0:
                        g["conv_w"][h, j - 1] += du[t] * v[b, t - j, h]
                        g["v"][b, t - j, h] += cw[h, j - 1] * du[t]
    return g


CASES = [
    # B, T, H, dk, dv, L, w, ragged, identity_act, d_fs, block, rs
    (2, 37, 2, 4, 5, 2, 4, True, False, True, 16, 1),
    (1, 21, 1, 6, 6, 3, 3, False, True, False, 8, 2),
    (2, 18, 2, 5, 4, 0, 2, False, False, True, 16, 2),
    (3, 9, 1, 4, 4, 1, 1, True, False, True, 4, 4),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_adjoint_matches_autograd(case):
    B, T, H, dk, dv, L, w, ragged, ida, with_fs, block, rs = case
    inp = random_small(B, T, H, dk, dv, L, w, seed=70 + T, ragged=ragged)
    rng = np.random.default_rng(T)
    d_out = rng.standard_normal((B, T, H, dv))
    d_fs = rng.standard_normal((B, H, dv, dk)) if with_fs else None
    ref = G.backward(inp, d_out, d_fs, identity_act=ida)
    mine = adjoint({n: (inp[n].numpy() if inp[n] is not None else None) for n in inp},
                   d_out, d_fs, identity_act=ida, block=block, rs=rs)
    for n in G.GRAD_KEYS:
        assert mine[n].shape == ref[n].shape, n
        if ref[n].size == 0:                       # W_k, W_p, w_beta at L = 0
            continue
        scale = max(np.max(np.abs(ref[n])), 1e-300)
        err = np.max(np.abs(mine[n] - ref[n])) / scale
        assert err <= 1e-11, f"d{n}: {err:.3e}"
