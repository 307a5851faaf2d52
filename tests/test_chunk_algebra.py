"""The chunkwise WY/UT form that the CUDA scan kernel evaluates, restated in
fp64 numpy and checked against the token-by-token oracle (CPU only).

This freezes the kernel's algebra before any GPU code runs.  It is a test
artefact: the CUDA path does not use it.

Per chunk of C tokens with entering state S0 (d_v x d_k), g = cumulative sum of
log alpha inside the chunk, gamma = exp(g), Gamma_ts = exp(g_t - g_s):
  A  = strict_tril(diag(beta) (K K^T (.) Gamma))
  T  = (I + A)^-1
  R  = sum_l strict_tril(K K_l^T (.) Gamma) D_l
  W  = T diag(beta gamma) K,   U = T diag(beta) (V - R)
  E  = U - W S0^T                       (pseudo-values of the delta rule)
  O  = diag(gamma) Q S0^T + tril(Q K^T (.) Gamma) E + sum_l tril(Q K_l^T (.) Gamma) D_l
  S1 = gamma_C S0 + E^T diag(gamma_C/gamma) K + sum_l D_l^T diag(gamma_C/gamma) K_l
where K_l, D_l are the per-token refinement directions k^(l) and write values
beta^(l) delta^(l) ("Technical Summary: PRISM", §2.2), and the Gated DeltaNet
write beta v k^T is the E part.

S1 is affine in S0: S1 = S0 M + c with M = gamma_C I - W^T diag(gamma_C/gamma) K and
c = U^T diag(gamma_C/gamma) K + sum_l D_l^T diag(gamma_C/gamma) K_l.  Maps compose as
(M1, c1) o (M2, c2) = (M1 M2, c1 M2 + c2), which is what a sequence split into segments
scanned in parallel would exchange (the §2.1 recurrence is an affine scan); the last test
checks that combine against the oracle.
"""
import numpy as np
import pytest

import oracle
from linear_recurrent_sequence_causal_gb300.inputs import random_small


def one_chunk(S, Q, K, V, bt, la, Kl, Dl):
    """One chunk from entering state S: returns (O, S1, M, c) with S1 = S M + c."""
    n_c, dk = K.shape
    g = np.cumsum(la)
    gam = np.exp(g)
    G = np.exp(g[:, None] - g[None, :])
    low = np.tril(np.ones((n_c, n_c)), -1)
    inc = np.tril(np.ones((n_c, n_c)))
    A = bt[:, None] * (K @ K.T) * G * low
    Tm = np.linalg.inv(np.eye(n_c) + A)
    L = len(Kl)
    R = sum(((K @ Kl[l].T) * G * low) @ Dl[l] for l in range(L)) if L else 0.0
    W = Tm @ ((bt * gam)[:, None] * K)
    U = Tm @ (bt[:, None] * (V - R))
    E = U - W @ S.T
    O = gam[:, None] * (Q @ S.T) + ((Q @ K.T) * G * inc) @ E
    for l in range(L):
        O += ((Q @ Kl[l].T) * G * inc) @ Dl[l]
    dec = np.exp(g[-1] - g)
    c = U.T @ (dec[:, None] * K)
    for l in range(L):
        c += Dl[l].T @ (dec[:, None] * Kl[l])
    M = np.exp(g[-1]) * np.eye(dk) - W.T @ (dec[:, None] * K)
    return O, S @ M + c, M, c


def _chunk_inputs(inp, kl, dl, b, h, c0, c1):
    q, k, v = (inp[n].double().numpy() for n in ("q", "k", "v"))
    la, be = inp["log_alpha"].double().numpy(), inp["beta"].double().numpy()
    L = kl.shape[3]
    return (q[b, c0:c1, h], k[b, c0:c1, h], v[b, c0:c1, h], be[b, c0:c1, h], la[b, c0:c1, h],
            [np.nan_to_num(kl[b, c0:c1, h, l]) for l in range(L)],
            [np.nan_to_num(dl[b, c0:c1, h, l]) for l in range(L)])


def chunk_form(inp, kl, dl, C):
    B, T, H, dk = inp["q"].shape
    dv = inp["v"].shape[-1]
    sl = inp.get("seq_lens")
    out = np.zeros((B, T, H, dv))
    fs = np.zeros((B, H, dv, dk))
    for b in range(B):
        n = T if sl is None else int(sl[b])
        for h in range(H):
            S = np.zeros((dv, dk))
            for c0 in range(0, n, C):
                c1 = min(c0 + C, n)
                O, S, _, _ = one_chunk(S, *_chunk_inputs(inp, kl, dl, b, h, c0, c1))
                out[b, c0:c1, h] = O
            fs[b, h] = S
    return out, fs


@pytest.mark.parametrize("L,C,ragged", [(0, 8, False), (2, 8, False), (3, 16, True), (4, 5, False)])
def test_chunk_form_matches_oracle(L, C, ragged):
    inp = random_small(3, 45, 2, 6, 7, L, 4, seed=30 + L, ragged=ragged)
    out, fs, tr = oracle.forward(inp, trace=True)
    co, cs = chunk_form(inp, tr["kl"], tr["dl"], C)
    scale_o = np.max(np.abs(out))
    np.testing.assert_allclose(co, out, atol=1e-12 * scale_o, rtol=0)
    np.testing.assert_allclose(cs, fs, atol=1e-12 * np.max(np.abs(fs)), rtol=0)


@pytest.mark.parametrize("L,C,cuts", [(0, 8, (16, 40)), (2, 8, (24,)), (3, 6, (12, 18, 36))])
def test_sequence_split_affine_combine(L, C, cuts):
    """Sequence split: each segment's affine map S_end = S_start M + c is built from its own
    chunks starting from nothing; an exclusive scan with (M1, c1) o (M2, c2) =
    (M1 M2, c1 M2 + c2) gives every segment's entering state, which equals the oracle's
    state after the prefix; the segment's outputs recomputed from that state equal the
    oracle's."""
    B, T, H, dk, dv = 1, 45, 2, 6, 7
    inp = random_small(B, T, H, dk, dv, L, 4, seed=60 + L)
    out, fs, tr = oracle.forward(inp, trace=True)
    bounds = [0, *cuts, T]
    for h in range(H):
        maps = []
        for s0, s1 in zip(bounds[:-1], bounds[1:]):
            M, c = np.eye(dk), np.zeros((dv, dk))
            for c0 in range(s0, s1, C):
                _, _, Mc, cc = one_chunk(np.zeros((dv, dk)),
                                         *_chunk_inputs(inp, tr["kl"], tr["dl"], 0, h, c0,
                                                        min(c0 + C, s1)))
                M, c = M @ Mc, c @ Mc + cc
            maps.append((M, c))
        S = np.zeros((dv, dk))
        for i, (s0, s1) in enumerate(zip(bounds[:-1], bounds[1:])):
            if s0 > 0:
                pre = {n: (v[:, :s0].contiguous() if n in ("q", "k", "v", "log_alpha", "beta")
                           else v) for n, v in inp.items()}
                _, fs_pre, _ = oracle.forward(pre)
                np.testing.assert_allclose(S, fs_pre[0, h], rtol=0,
                                           atol=1e-12 * np.max(np.abs(fs_pre[0, h])))
            Sseg = S.copy()
            for c0 in range(s0, s1, C):
                c1 = min(c0 + C, s1)
                O, Sseg, _, _ = one_chunk(Sseg, *_chunk_inputs(inp, tr["kl"], tr["dl"], 0, h,
                                                               c0, c1))
                np.testing.assert_allclose(O, out[0, c0:c1, h], rtol=0,
                                           atol=1e-12 * np.max(np.abs(out)))
            M, c = maps[i]
            S = S @ M + c
            np.testing.assert_allclose(S, Sseg, rtol=0, atol=1e-12 * np.max(np.abs(Sseg)))
        np.testing.assert_allclose(S, fs[0, h], rtol=0, atol=1e-12 * np.max(np.abs(fs[0, h])))
