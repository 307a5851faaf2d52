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
"""
import numpy as np
import pytest

import oracle
from linear_recurrent_sequence_causal_gb300.inputs import random_small


def chunk_form(inp, kl, dl, C):
    q, k, v = (inp[n].double().numpy() for n in ("q", "k", "v"))
    la, be = inp["log_alpha"].double().numpy(), inp["beta"].double().numpy()
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    L = kl.shape[3]
    sl = inp.get("seq_lens")
    out = np.zeros((B, T, H, dv))
    fs = np.zeros((B, H, dv, dk))
    for b in range(B):
        n = T if sl is None else int(sl[b])
        for h in range(H):
            S = np.zeros((dv, dk))
            for c0 in range(0, n, C):
                c1 = min(c0 + C, n)
                Q, K, V = q[b, c0:c1, h], k[b, c0:c1, h], v[b, c0:c1, h]
                bt = be[b, c0:c1, h]
                g = np.cumsum(la[b, c0:c1, h])
                gam = np.exp(g)
                G = np.exp(g[:, None] - g[None, :])
                n_c = c1 - c0
                low = np.tril(np.ones((n_c, n_c)), -1)
                inc = np.tril(np.ones((n_c, n_c)))
                A = bt[:, None] * (K @ K.T) * G * low
                Tm = np.linalg.inv(np.eye(n_c) + A)
                Kl = [np.nan_to_num(kl[b, c0:c1, h, l]) for l in range(L)]
                Dl = [np.nan_to_num(dl[b, c0:c1, h, l]) for l in range(L)]
                R = sum(((K @ Kl[l].T) * G * low) @ Dl[l] for l in range(L)) if L else 0.0
                W = Tm @ ((bt * gam)[:, None] * K)
                U = Tm @ (bt[:, None] * (V - R))
                E = U - W @ S.T
                O = gam[:, None] * (Q @ S.T) + ((Q @ K.T) * G * inc) @ E
                for l in range(L):
                    O += ((Q @ Kl[l].T) * G * inc) @ Dl[l]
                dec = np.exp(g[-1] - g)
                Snew = np.exp(g[-1]) * S + E.T @ (dec[:, None] * K)
                for l in range(L):
                    Snew += Dl[l].T @ (dec[:, None] * Kl[l])
                out[b, c0:c1, h] = O
                S = Snew
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
