"""The chunkwise (WY/UT) form of the backward pass, restated in fp64 numpy and checked
against the autograd gradient oracle (CPU only).

The backward kernels that run today walk the tokens one by one; this file fixes the
algebra of a chunked backward (the forward's chunk products differentiated, so that
they can run as dense contractions) before any kernel is written for it.  It is a test
artefact: the CUDA path does not use it.

Per chunk of n tokens with entering state S0 (d_v x d_k), g = in-chunk cumulative sum of
log alpha, gamma = exp(g), lambda = gamma_C / gamma, Gamma_ts = exp(g_t - g_s), the
forward ("Technical Summary: PRISM", §2.1 and §2.2, in the chunk form of the forward
scan) is
  A = strict_tril(diag(beta) K K^T (.) Gamma),  T = (I + A)^-1
  P_l = strict_tril(K K_l^T (.) Gamma),  R = sum_l P_l D_l
  W = T diag(beta gamma) K,  U = T diag(beta) (V - R),  E = U - W S0^T
  O = diag(gamma) Q S0^T + tril(Q K^T (.) Gamma) E + sum_l tril(Q K_l^T (.) Gamma) D_l
  S1 = gamma_C S0 + E^T diag(lambda) K + sum_l D_l^T diag(lambda) K_l
and its adjoint, given dO and dS1, takes the same steps in reverse:
  (S1)  dS0 = gamma_C dS1,  dE = diag(lambda) K dS1^T,  dK += diag(lambda) E dS1,
        dD_l += diag(lambda) K_l dS1^T,  dK_l += diag(lambda) D_l dS1
  (O)   dS0 += dO^T diag(gamma) Q,  dQ += diag(gamma) dO S0,  dE += tril(.)^T dO,
        dD_l += tril_l(.)^T dO, and for each masked product X = M (.) Gamma (.) (Y Z^T):
        dY += (M (.) Gamma (.) dX) Z,  dZ += (M (.) Gamma (.) dX)^T Y
  (E)   dU = dE,  dW = -dE S0,  dS0 -= dE^T W
  (U,W) dT = dU (diag(beta)(V - R))^T + dW (diag(beta gamma) K)^T,
        dV += diag(beta) T^T dU,  dR = -diag(beta) T^T dU,  dK += diag(beta gamma) T^T dW
  (R)   dD_l += P_l^T dR,  dP_l = dR D_l^T
  (T)   dA = -T^T dT T^T
and every Gamma, gamma, lambda, gamma_C factor adds to dg (for X_ts carrying
exp(g_t - g_s): dg_t += sum_s dX_ts X_ts, dg_s -= the same), with
d log alpha = the in-chunk reverse cumulative sum of dg.  Chunks run in reverse order,
dS0 of one chunk being dS1 of the chunk before it; each chunk's S0 comes from the
forward (kept per chunk).  The per-token refinement chain and the transposed anchor then
finish the gradients as in the token-sequential restatement.
"""
import numpy as np
import pytest

from linear_recurrent_sequence_causal_gb300.inputs import random_small
from oracle import grad as G
from tests.test_backward_algebra import _refine_forward, refine_backward


def _decays(la):
    n = la.shape[0]
    g = np.cumsum(la)
    t_ge_s = np.tril(np.ones((n, n), dtype=bool))
    Gm = np.exp(np.where(t_ge_s, g[:, None] - g[None, :], 0.0))
    return g, Gm * np.tril(np.ones((n, n)), -1), Gm * np.tril(np.ones((n, n)))


def chunk_forward(S0, Q, K, V, be, la, Kl, Dl):
    n, dk = K.shape
    g, GS, GI = _decays(la)
    gam = np.exp(g)
    lam = np.exp(g[-1] - g)
    KK = K @ K.T
    A = be[:, None] * KK * GS
    T = np.linalg.inv(np.eye(n) + A)
    P = [(K @ Kl[l].T) * GS for l in range(len(Kl))]
    R = sum((P[l] @ Dl[l] for l in range(len(Kl))), np.zeros_like(V))
    Kbg = (be * gam)[:, None] * K
    W = T @ Kbg
    VR = V - R
    Vb = be[:, None] * VR
    U = T @ Vb
    E = U - W @ S0.T
    QK = (Q @ K.T) * GI
    QKl = [(Q @ Kl[l].T) * GI for l in range(len(Kl))]
    O = gam[:, None] * (Q @ S0.T) + QK @ E + sum((QKl[l] @ Dl[l] for l in range(len(Kl))),
                                                  np.zeros_like(V))
    S1 = np.exp(g[-1]) * S0 + E.T @ (lam[:, None] * K)
    for l in range(len(Kl)):
        S1 = S1 + Dl[l].T @ (lam[:, None] * Kl[l])
    saved = dict(g=g, GS=GS, GI=GI, gam=gam, lam=lam, KK=KK, A=A, T=T, P=P, Kbg=Kbg, W=W,
                 VR=VR, Vb=Vb, E=E, QK=QK, QKl=QKl)
    return O, S1, saved


def chunk_backward(S0, Q, K, V, be, la, Kl, Dl, dO, dS1):
    """Cotangents of one chunk's inputs (S0, Q, K, V, beta, log alpha, K_l, D_l) from those
    of its outputs (O, S1)."""
    _, _, f = chunk_forward(S0, Q, K, V, be, la, Kl, Dl)
    L = len(Kl)
    gam, lam, GS, GI, E, T = f["gam"], f["lam"], f["GS"], f["GI"], f["E"], f["T"]
    gC = gam[-1]
    dg = np.zeros_like(la)
    dQ, dK, dV = np.zeros_like(Q), np.zeros_like(K), np.zeros_like(V)
    dbeta = np.zeros_like(be)
    dKl = [np.zeros_like(x) for x in Kl]
    dDl = [np.zeros_like(x) for x in Dl]

    def masked(dX, X, Gmask, Y, Z):           # X = Gmask (.) (Y Z^T)
        Gd = Gmask * dX
        Zp = dX * X
        dg[:] += Zp.sum(1) - Zp.sum(0)
        return Gd @ Z, Gd.T @ Y

    # S1 = gamma_C S0 + E^T diag(lambda) K + sum_l D_l^T diag(lambda) K_l
    dS0 = gC * dS1
    dg[-1] += gC * np.sum(S0 * dS1)
    dE = lam[:, None] * (K @ dS1.T)
    dK += lam[:, None] * (E @ dS1)
    dlam = np.sum((E @ dS1) * K, axis=1)
    for l in range(L):
        dDl[l] += lam[:, None] * (Kl[l] @ dS1.T)
        dKl[l] += lam[:, None] * (Dl[l] @ dS1)
        dlam += np.sum((Dl[l] @ dS1) * Kl[l], axis=1)
    dg[-1] += np.sum(dlam * lam)
    dg -= dlam * lam
    # O = diag(gamma) Q S0^T + QK E + sum_l QK_l D_l
    dS0 += dO.T @ (gam[:, None] * Q)
    dQ += gam[:, None] * (dO @ S0)
    dg += gam * np.sum(dO * (Q @ S0.T), axis=1)
    dE += f["QK"].T @ dO
    a, b = masked(dO @ E.T, f["QK"], GI, Q, K)
    dQ += a
    dK += b
    for l in range(L):
        dDl[l] += f["QKl"][l].T @ dO
        a, b = masked(dO @ Dl[l].T, f["QKl"][l], GI, Q, Kl[l])
        dQ += a
        dKl[l] += b
    # E = U - W S0^T
    dU = dE
    dW = -dE @ S0
    dS0 -= dE.T @ f["W"]
    # U = T diag(beta) (V - R),  W = T diag(beta gamma) K
    dT = dU @ f["Vb"].T + dW @ f["Kbg"].T
    dVb = T.T @ dU
    dV += be[:, None] * dVb
    dR = -be[:, None] * dVb
    dbeta += np.sum(f["VR"] * dVb, axis=1)
    dKbg = T.T @ dW
    dK += (be * gam)[:, None] * dKbg
    kd = np.sum(K * dKbg, axis=1)
    dbeta += gam * kd
    dg += be * gam * kd
    # R = sum_l P_l D_l,  P_l = strict_tril(K K_l^T (.) Gamma)
    for l in range(L):
        dDl[l] += f["P"][l].T @ dR
        a, b = masked(dR @ Dl[l].T, f["P"][l], GS, K, Kl[l])
        dK += a
        dKl[l] += b
    # T = (I + A)^-1,  A = strict_tril(diag(beta) K K^T (.) Gamma)
    dA = -T.T @ dT @ T.T
    dbeta += np.sum(dA * f["KK"] * GS, axis=1)
    Gd = GS * be[:, None] * dA
    dK += Gd @ K + Gd.T @ K
    Zp = dA * f["A"]
    dg += Zp.sum(1) - Zp.sum(0)
    dla = np.cumsum(dg[::-1])[::-1]
    return dict(S0=dS0, q=dQ, k=dK, v=dV, beta=dbeta, log_alpha=dla, Kl=dKl, Dl=dDl)


def chunked_adjoint(inp, d_out, d_fs, C, *, identity_act=False):
    f = {n: np.asarray(inp[n], dtype=np.float64) for n in G.GRAD_KEYS}
    q, k, v, la, be = f["q"], f["k"], f["v"], f["log_alpha"], f["beta"]
    cw, Wk, Wp, wb = f["conv_w"], f["Wk"], f["Wp"], f["wbeta"]
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    w = cw.shape[1]
    L = Wk.shape[1]
    lens = [T] * B if inp.get("seq_lens") is None else [int(x) for x in inp["seq_lens"]]
    g = {n: np.zeros_like(f[n]) for n in G.GRAD_KEYS}
    for b in range(B):
        n_tok = lens[b]
        for h in range(H):
            u = np.zeros((n_tok, dv))
            for t in range(n_tok):
                for j in range(1, w + 1):
                    if t - j >= 0:
                        u[t] += cw[h, j - 1] * v[b, t - j, h]
            ref = [_refine_forward(u[t], v[b, t, h], Wk[h], Wp[h], wb[h], identity_act)
                   for t in range(n_tok)]
            Kl_all = np.array([[s["k"] for s in r] for r in ref]).reshape(n_tok, L, dk)
            Dl_all = np.array([[s["D"] for s in r] for r in ref]).reshape(n_tok, L, dv)

            def chunk_args(c0, c1):
                return (q[b, c0:c1, h], k[b, c0:c1, h], v[b, c0:c1, h], be[b, c0:c1, h],
                        la[b, c0:c1, h], [Kl_all[c0:c1, l] for l in range(L)],
                        [Dl_all[c0:c1, l] for l in range(L)])

            starts = list(range(0, n_tok, C))
            S0s = []
            S = np.zeros((dv, dk))
            for c0 in starts:
                S0s.append(S)
                _, S, _ = chunk_forward(S, *chunk_args(c0, min(c0 + C, n_tok)))
            dS = np.zeros((dv, dk)) if d_fs is None else np.array(d_fs[b, h], dtype=np.float64)
            dKl = np.zeros((n_tok, L, dk))
            dDl = np.zeros((n_tok, L, dv))
            for ci in range(len(starts) - 1, -1, -1):
                c0 = starts[ci]
                c1 = min(c0 + C, n_tok)
                r = chunk_backward(S0s[ci], *chunk_args(c0, c1), d_out[b, c0:c1, h], dS)
                dS = r["S0"]
                for name in ("q", "k", "v", "beta", "log_alpha"):
                    g[name][b, c0:c1, h] += r[name]
                for l in range(L):
                    dKl[c0:c1, l] = r["Kl"][l]
                    dDl[c0:c1, l] = r["Dl"][l]
            du = np.zeros((n_tok, dv))
            for t in range(n_tok):
                dr, dut = refine_backward(ref[t], dDl[t], dKl[t], u[t], Wk[h], Wp[h], wb[h],
                                          g, h, identity_act)
                g["v"][b, t, h] += dr
                du[t] = dut - dr
            for t in range(n_tok):
                for j in range(1, w + 1):
                    if t - j >= 0:
                        g["conv_w"][h, j - 1] += du[t] * v[b, t - j, h]
                        g["v"][b, t - j, h] += cw[h, j - 1] * du[t]
    return g


CASES = [
    # B, T, H, dk, dv, L, w, ragged, identity_act, d_fs, chunk
    (2, 37, 2, 4, 5, 2, 4, True, False, True, 8),
    (1, 30, 1, 6, 6, 3, 3, False, True, False, 16),
    (2, 19, 2, 5, 4, 0, 2, False, False, True, 4),
    (3, 11, 1, 4, 4, 1, 1, True, False, True, 5),
    (1, 24, 1, 3, 3, 2, 3, False, False, True, 24),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_chunked_adjoint_matches_autograd(case):
    B, T, H, dk, dv, L, w, ragged, ida, with_fs, C = case
    inp = random_small(B, T, H, dk, dv, L, w, seed=80 + T, ragged=ragged)
    rng = np.random.default_rng(T + 1)
    d_out = rng.standard_normal((B, T, H, dv))
    d_fs = rng.standard_normal((B, H, dv, dk)) if with_fs else None
    ref = G.backward(inp, d_out, d_fs, identity_act=ida)
    mine = chunked_adjoint({n: (inp[n].numpy() if inp[n] is not None else None) for n in inp},
                           d_out, d_fs, C, identity_act=ida)
    for n in G.GRAD_KEYS:
        assert mine[n].shape == ref[n].shape, n
        if ref[n].size == 0:
            continue
        scale = max(np.max(np.abs(ref[n])), 1e-300)
        err = np.max(np.abs(mine[n] - ref[n])) / scale
        assert err <= 1e-10, f"d{n}: {err:.3e}"


def test_chunk_adjoint_dot_product():
    """<J x, y> = <x, J^T y> for one chunk with a nonzero entering state: the adjoint of
    chunk_forward's linearisation, checked by central differences along a random
    direction (all inputs, S0 included)."""
    rng = np.random.default_rng(5)
    n, dk, dv, L = 7, 4, 5, 2
    Q, K = rng.standard_normal((n, dk)), rng.standard_normal((n, dk)) / 2
    V = rng.standard_normal((n, dv))
    be = 1 / (1 + np.exp(-rng.standard_normal(n)))
    la = -np.log1p(np.exp(rng.standard_normal(n))) / 8
    Kl = [rng.standard_normal((n, dk)) / 2 for _ in range(L)]
    Dl = [rng.standard_normal((n, dv)) for _ in range(L)]
    S0 = rng.standard_normal((dv, dk))
    dO, dS1 = rng.standard_normal((n, dv)), rng.standard_normal((dv, dk))
    r = chunk_backward(S0, Q, K, V, be, la, Kl, Dl, dO, dS1)
    x = dict(S0=S0, q=Q, k=K, v=V, beta=be, log_alpha=la)
    dx = {key: rng.standard_normal(np.shape(val)) for key, val in x.items()}
    dKl = [rng.standard_normal((n, dk)) for _ in range(L)]
    dDl = [rng.standard_normal((n, dv)) for _ in range(L)]
    eps = 1e-6

    def run(sign):
        y = {key: x[key] + sign * eps * dx[key] for key in x}
        O, S1, _ = chunk_forward(y["S0"], y["q"], y["k"], y["v"], y["beta"], y["log_alpha"],
                                 [Kl[l] + sign * eps * dKl[l] for l in range(L)],
                                 [Dl[l] + sign * eps * dDl[l] for l in range(L)])
        return np.sum(O * dO) + np.sum(S1 * dS1)

    fd = (run(1) - run(-1)) / (2 * eps)
    an = sum(np.sum(r[key] * dx[key]) for key in x)
    an += sum(np.sum(r["Kl"][l] * dKl[l]) + np.sum(r["Dl"][l] * dDl[l]) for l in range(L))
    assert abs(fd - an) <= 1e-7 * max(abs(an), 1.0), (fd, an)


def test_reverse_chain_has_the_forward_scan_form():
    """The serial part of the chunked backward is the forward scan's state update run
    backwards with the same per-chunk factors: with W = T diag(beta gamma) K,
    Qt = diag(gamma) Q - tril(Q K^T (.) Gamma) W and Kt = diag(lambda) K (the factors the
    forward's prepare stage computes),
        dS0 = gamma_C dS1 - (Kt dS1^T)^T W + dO^T Qt,
    i.e. dS0 = dS1 M^T + dO^T Qt with M = gamma_C I - W^T Kt the forward chunk map.  Every
    other gradient of the chunk is then state-parallel given S0 and dS1."""
    rng = np.random.default_rng(9)
    for n, dk, dv, L in [(8, 4, 5, 2), (16, 6, 6, 0), (5, 3, 4, 3)]:
        Q, K = rng.standard_normal((n, dk)), rng.standard_normal((n, dk)) / 2
        V = rng.standard_normal((n, dv))
        be = 1 / (1 + np.exp(-rng.standard_normal(n)))
        la = -np.log1p(np.exp(rng.standard_normal(n))) / 8
        Kl = [rng.standard_normal((n, dk)) / 2 for _ in range(L)]
        Dl = [rng.standard_normal((n, dv)) for _ in range(L)]
        S0 = rng.standard_normal((dv, dk))
        dO, dS1 = rng.standard_normal((n, dv)), rng.standard_normal((dv, dk))
        r = chunk_backward(S0, Q, K, V, be, la, Kl, Dl, dO, dS1)
        _, _, f = chunk_forward(S0, Q, K, V, be, la, Kl, Dl)
        W, gam, lam = f["W"], f["gam"], f["lam"]
        Qt = gam[:, None] * Q - f["QK"] @ W
        Kt = lam[:, None] * K
        dS0 = gam[-1] * dS1 - (Kt @ dS1.T).T @ W + dO.T @ Qt
        np.testing.assert_allclose(r["S0"], dS0, rtol=0, atol=1e-12 * np.max(np.abs(dS0)))
        M = gam[-1] * np.eye(dk) - W.T @ Kt
        np.testing.assert_allclose(dS1 @ M.T + dO.T @ Qt, dS0, rtol=0, atol=1e-12 * np.max(np.abs(dS0)))
