"""Checks that pin the CPU oracle to facts fixed by the pages and by mathematics.

Each ``pin_*`` function takes ``fwd`` (``oracle.forward`` or a build of the
oracle with a planted mistake) and raises AssertionError when the oracle
disagrees with the fact it checks.  None of them retypes the oracle's own
loop: they use an independent formulation (explicit d x d matrices, products
of explicit A_t), a library routine (numpy convolution, the normal CDF,
scipy's logistic function, SVD, cumulative sums) or a closed form.

Sources ("Technical Summary: PRISM (Parallel Residual Iterative Sequence
Model)", gist.science/paper/2602.10796):
  §2.1  S_t = S_{t-1} A_t + B_t, A_t rank-1 as in Gated DeltaNet
  §2.2  anchor u_t from a ShortConv over the input; refinement loop
        k^(l) = W_k^(l) u_t, p^(l) = W_p^(l) u_t, delta = GELU(p (.) r),
        r^(l+1) = r^(l) - delta^(l); B_t = sum_l beta^(l) delta^(l) k^(l)^T
  §3.3  at L = 0 PRISM reduces to Gated DeltaNet; the write has rank <= L
        (plus the Gated DeltaNet rank-1 base write, which is kept in B_t so that
        L = 0 gives Gated DeltaNet)
"""
from __future__ import annotations

import numpy as np
import scipy.special
import scipy.stats
import torch

from linear_recurrent_sequence_causal_gb300.inputs import random_small


def gdn_explicit(inp, T=None, S0=None):
    """Gated DeltaNet with explicit matrices: S <- S (alpha (I - beta k k^T)) + beta v k^T,
    starting from S0 [B,H,dv,dk] (zero when None).

    Independent of the oracle: forms every A_t as a d_k x d_k matrix.
    Returns out [B,T,H,dv] and final state [B,H,dv,dk].
    """
    q, k, v = (inp[n].double().numpy() for n in ("q", "k", "v"))
    la, be = inp["log_alpha"].double().numpy(), inp["beta"].double().numpy()
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    sl = inp.get("seq_lens")
    out = np.zeros((B, T, H, dv))
    fs = np.zeros((B, H, dv, dk))
    I = np.eye(dk)
    for b in range(B):
        n = T if sl is None else int(sl[b])
        for h in range(H):
            S = np.zeros((dv, dk)) if S0 is None else np.array(S0[b, h], dtype=np.float64)
            for t in range(n):
                kt = k[b, t, h]
                A = np.exp(la[b, t, h]) * (I - be[b, t, h] * np.outer(kt, kt))
                S = S @ A + be[b, t, h] * np.outer(v[b, t, h], kt)
                out[b, t, h] = S @ q[b, t, h]
            fs[b, h] = S
    return out, fs


def _close(a, b, tol, what):
    err = np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300)
    assert err <= tol, f"{what}: normwise error {err:.3e} > {tol:.1e}"


def pin_l0_is_gated_deltanet(fwd):
    """§3.3: with L = 0 the oracle must be the plain gated delta rule."""
    inp = random_small(2, 40, 2, 5, 7, 0, 3, seed=11)
    out, fs, _ = fwd(inp, L=0)
    ref_o, ref_s = gdn_explicit(inp)
    _close(out, ref_o, 1e-12, "L=0 output vs Gated DeltaNet")
    _close(fs, ref_s, 1e-12, "L=0 final state vs Gated DeltaNet")


def pin_zero_conv_is_gated_deltanet(fwd):
    """conv_w = 0 => u = 0 => p = 0 => delta = GELU(0) = 0: any L gives Gated DeltaNet."""
    inp = random_small(1, 33, 2, 6, 6, 3, 4, seed=12)
    inp["conv_w"] = torch.zeros_like(inp["conv_w"])
    out, fs, _ = fwd(inp)
    ref_o, ref_s = gdn_explicit(inp)
    _close(out, ref_o, 1e-12, "zero-conv output vs Gated DeltaNet")
    _close(fs, ref_s, 1e-12, "zero-conv final state vs Gated DeltaNet")


def pin_write_rank(fwd):
    """§3.3 rank accumulation: B_t - beta_t v_t k_t^T has rank <= L (generically = L)."""
    L = 2
    inp = random_small(1, 24, 1, 6, 8, L, 4, seed=13)
    _, _, tr = fwd(inp, trace=True)
    k, v, be = inp["k"].numpy(), inp["v"].numpy(), inp["beta"].numpy()
    for t in range(2, 24):   # from t = 2 on the anchor is non-zero
        extra = tr["Bt"][0, t, 0] - be[0, t, 0] * np.outer(v[0, t, 0], k[0, t, 0])
        s = np.linalg.svd(extra, compute_uv=False)
        assert s[L] <= 1e-12 * s[0], f"t={t}: sigma_{L + 1}/sigma_1 = {s[L] / s[0]:.2e}"
        assert s[L - 1] >= 1e-8 * s[0], f"t={t}: write rank below L"


def pin_telescoping(fwd):
    """§2.2: r^(l+1) = r^(l) - delta^(l) telescopes to r^(L+1) = r^(1) - sum_l delta^(l),
    with r^(1) = v - u."""
    inp = random_small(2, 20, 2, 5, 7, 4, 3, seed=14)
    _, _, tr = fwd(inp, trace=True)
    scale = np.max(np.abs(tr["r1"]))
    np.testing.assert_allclose(tr["r_final"], tr["r1"] - tr["delta"].sum(axis=3),
                               atol=1e-14 * scale, rtol=0)
    np.testing.assert_allclose(tr["r1"], inp["v"].numpy() - tr["u"], atol=1e-15, rtol=0)


def pin_brute_force_products(fwd):
    """§2.1 for T <= 16: S_t = sum_{s<=t} B_s prod_{j=s+1..t} A_j with explicit A_j."""
    inp = random_small(1, 16, 2, 4, 5, 2, 3, seed=15)
    out, fs, tr = fwd(inp, trace=True)
    q, k = inp["q"].numpy(), inp["k"].numpy()
    la, be = inp["log_alpha"].numpy(), inp["beta"].numpy()
    dk = k.shape[-1]
    for h in range(2):
        A = [np.exp(la[0, j, h]) * (np.eye(dk) - be[0, j, h] * np.outer(k[0, j, h], k[0, j, h]))
             for j in range(16)]
        for t in range(16):
            S = np.zeros_like(tr["Bt"][0, 0, h])
            for s in range(t + 1):
                P = np.eye(dk)
                for j in range(s + 1, t + 1):
                    P = P @ A[j]
                S += tr["Bt"][0, s, h] @ P
            np.testing.assert_allclose(out[0, t, h], S @ q[0, t, h], atol=1e-12, rtol=0)
            if t == 15:
                np.testing.assert_allclose(fs[0, h], S, atol=1e-12, rtol=0)


def pin_prefix_sum(fwd):
    """alpha = 1, beta = 0: A_t = I, so S_t is the running sum of the writes B_s."""
    inp = random_small(1, 12, 1, 4, 6, 2, 3, seed=16)
    inp["log_alpha"].zero_()
    inp["beta"].zero_()
    out, _, tr = fwd(inp, trace=True)
    S = np.cumsum(tr["Bt"][0, :, 0], axis=0)
    np.testing.assert_allclose(out[0, :, 0], np.einsum("tij,tj->ti", S, inp["q"][0, :, 0].numpy()),
                               atol=1e-12, rtol=0)


def pin_no_write_no_output(fwd):
    """L = 0 and beta = 0: nothing is ever written, so o = 0 exactly."""
    inp = random_small(2, 10, 2, 4, 4, 0, 3, seed=17)
    inp["beta"].zero_()
    out, fs, _ = fwd(inp, L=0)
    assert np.all(out == 0.0) and np.all(fs == 0.0)


def pin_shortconv(fwd):
    """§2.2 stage 1: u_t = sum_{j=1..w} c_j (.) v_{t-j} (strictly causal, zero history),
    checked against numpy's full convolution with the taps shifted by one lag."""
    w = 4
    inp = random_small(2, 19, 3, 5, 6, 1, w, seed=18)
    _, _, tr = fwd(inp, trace=True)
    v, c = inp["v"].numpy(), inp["conv_w"].numpy()
    T = v.shape[1]
    for b in range(2):
        for h in range(3):
            for i in range(6):
                taps = np.concatenate([[0.0], c[h, :, i]])   # lag 0 has no tap
                ref = np.convolve(v[b, :, h, i], taps)[:T]
                np.testing.assert_allclose(tr["u"][b, :, h, i], ref, atol=1e-14, rtol=0)


def pin_direction(fwd):
    """§2.2 direction k^(l) = normalize(W_k^(l) u): with a one-hot W_k = e_a e_c^T the
    direction is e_a g u_c / sqrt((g u_c)^2 + 1e-6).  Each head has its own (a, c, g), so
    a transposed W_k or one head's W_k used for another is caught."""
    dk, dv = 3, 5
    inp = random_small(1, 9, 2, dk, dv, 1, 2, seed=19)
    Wk = torch.zeros_like(inp["Wk"])
    per_head = [(1, 3, 1.7), (2, 0, -0.8)]   # (row a on the d_k side, column c on d_v, gain)
    for h, (a, c, g) in enumerate(per_head):
        Wk[h, 0, a, c] = g
    inp["Wk"] = Wk
    _, _, tr = fwd(inp, trace=True)
    for h, (a, c, g) in enumerate(per_head):
        x = g * tr["u"][0, :, h, c]
        exp = np.zeros((9, dk))
        exp[:, a] = x / np.sqrt(x * x + 1e-6)
        np.testing.assert_allclose(tr["kl"][0, :, h, 0], exp, atol=1e-14, rtol=0)


def pin_gain_and_gelu(fwd):
    """§2.2 delta^(1) = GELU(p (.) r^(1)) with p = W_p u.  W_p = s I gives p = s u, and
    GELU(x) = x Phi(x) with Phi the standard normal CDF (scipy).  The two heads take
    different gains s."""
    dv = 6
    inp = random_small(1, 14, 2, 4, dv, 2, 3, seed=20)
    gains = (1.9, -0.6)
    for h, s in enumerate(gains):
        inp["Wp"][h, 0] = s * torch.eye(dv, dtype=torch.float64)
    _, _, tr = fwd(inp, trace=True)
    for h, s in enumerate(gains):
        u, r1 = tr["u"][0, :, h], tr["r1"][0, :, h]
        x = s * u * r1
        np.testing.assert_allclose(tr["delta"][0, :, h, 0], x * scipy.stats.norm.cdf(x),
                                   atol=1e-14, rtol=1e-13)
        # The second step acts on the updated residual r^(2) = r^(1) - delta^(1).
        p2 = tr["pl"][0, :, h, 1]
        x2 = p2 * (r1 - tr["delta"][0, :, h, 0])
        np.testing.assert_allclose(tr["delta"][0, :, h, 1], x2 * scipy.stats.norm.cdf(x2),
                                   atol=1e-14, rtol=1e-13)


def pin_confidence_gate(fwd):
    """§2.2 confidence gate beta^(l) = sigmoid(w_beta^(l) . u): w = 0 gives exactly 1/2;
    w = s e_c gives expit(s u_c) (scipy).  The write factor is beta^(l) delta^(l).  The
    second head takes another (s, c)."""
    dv = 5
    inp = random_small(1, 11, 2, 4, dv, 2, 3, seed=21)
    inp["wbeta"].zero_()
    per_head = [(3, -2.3), (1, 1.4)]
    for h, (c, s) in enumerate(per_head):
        inp["wbeta"][h, 1, c] = s
    _, _, tr = fwd(inp, trace=True)
    assert np.all(tr["betal"][0, :, :, 0] == 0.5)
    for h, (c, s) in enumerate(per_head):
        np.testing.assert_allclose(tr["betal"][0, :, h, 1], scipy.special.expit(s * tr["u"][0, :, h, c]),
                                   atol=1e-15, rtol=1e-14)
    np.testing.assert_allclose(tr["dl"], tr["betal"][..., None] * tr["delta"], atol=1e-15, rtol=0)


def pin_gate_scales_write(fwd):
    """§2.2 final injection B_t = sum_l beta^(l) delta^(l) k^(l)^T: delta^(l) and k^(l) do
    not depend on w_beta, so the refinement part of the write the state receives, B_t minus
    the L = 0 write, scales with the gate.  At L = 1 a run with w_beta = s e_c has
    2 expit(s u_c) times the refinement write of a run with w_beta = 0 (gate 1/2)."""
    inp = random_small(1, 13, 2, 4, 5, 1, 3, seed=27)
    c, s = 2, 1.6
    half = {k: (v.clone() if v is not None else None) for k, v in inp.items()}
    half["wbeta"].zero_()
    gated = {k: (v.clone() if v is not None else None) for k, v in half.items()}
    gated["wbeta"][:, 0, c] = s
    _, _, tr0 = fwd(inp, trace=True, L=0)
    _, _, trh = fwd(half, trace=True)
    _, _, trg = fwd(gated, trace=True)
    base = tr0["Bt"]
    dh, dg = trh["Bt"] - base, trg["Bt"] - base
    assert np.max(np.abs(dh)) > 1e-3, "refinement write vanished"
    ratio = 2.0 * scipy.special.expit(s * trh["u"][..., c])       # [B, T, H]
    np.testing.assert_allclose(dg, ratio[..., None, None] * dh, atol=1e-14, rtol=1e-12)


def pin_padding(fwd):
    """Right padding: a length-n sequence padded to T gives the length-n result, zeros
    after n, and a frozen final state; NaN in the padding must not leak."""
    inp = random_small(3, 21, 2, 4, 5, 2, 3, seed=22)
    lens = torch.tensor([21, 7, 1], dtype=torch.int32)
    padded = {k: (v.clone() if v is not None else None) for k, v in inp.items()}
    padded["seq_lens"] = lens
    for b, n in enumerate(lens.tolist()):
        for name in ("q", "k", "v", "log_alpha", "beta"):
            padded[name][b, n:] = float("nan")
    out, fs, _ = fwd(padded)
    for b, n in enumerate(lens.tolist()):
        one = {k: (v[b:b + 1, :n] if k in ("q", "k", "v", "log_alpha", "beta") else v)
               for k, v in inp.items() if k != "seq_lens"}
        o1, s1, _ = fwd(one)
        np.testing.assert_allclose(out[b, :n], o1[0], atol=1e-14, rtol=0)
        assert np.all(out[b, n:] == 0.0)
        np.testing.assert_allclose(fs[b], s1[0], atol=1e-14, rtol=0)


def pin_causality(fwd):
    """Outputs before t0 do not depend on inputs at or after t0."""
    inp = random_small(1, 30, 2, 4, 4, 3, 4, seed=23)
    out1, _, _ = fwd(inp)
    other = {k: (v.clone() if v is not None else None) for k, v in inp.items()}
    g = torch.Generator().manual_seed(99)
    for name in ("q", "k", "v", "log_alpha", "beta"):
        other[name][:, 17:] = torch.randn(other[name][:, 17:].shape, generator=g,
                                          dtype=torch.float64)
    out2, _, _ = fwd(other)
    np.testing.assert_array_equal(out1[:, :17], out2[:, :17])
    assert not np.allclose(out1[:, 17:], out2[:, 17:])


def pin_identity_activation(fwd):
    """No-GELU ablation: delta^(l) = p^(l) (.) r^(l) exactly."""
    inp = random_small(1, 12, 1, 4, 4, 3, 3, seed=24)
    _, _, tr = fwd(inp, trace=True, identity_act=True)
    r = tr["r1"][0, :, 0]
    for l in range(3):
        d = tr["pl"][0, :, 0, l] * r
        np.testing.assert_allclose(tr["delta"][0, :, 0, l], d, atol=1e-15, rtol=0)
        r = r - d


def _slice_tokens(inp, t0, t1):
    out = dict(inp)
    for n in ("q", "k", "v", "log_alpha", "beta"):
        out[n] = inp[n][:, t0:t1].contiguous()
    return out


def pin_resume_is_markov(fwd):
    """The recurrence is Markov in (S, the last w values of v): running tokens
    [0, T1), then [T1, T) from the reached state and the last w rows of v, gives the
    outputs and final state of one run over [0, T) (split at several points)."""
    inp = random_small(2, 29, 2, 5, 4, 2, 3, seed=25)
    out, fs, _ = fwd(inp)
    w = inp["conv_w"].shape[1]
    for T1 in (1, 2, 11, 28):
        o1, s1, _ = fwd(_slice_tokens(inp, 0, T1))
        t0 = max(T1 - w, 0)
        hist = np.zeros((2, 2, w, 4))
        hist[:, :, w - (T1 - t0):] = inp["v"][:, t0:T1].double().numpy().transpose(0, 2, 1, 3)
        o2, s2, _ = fwd(_slice_tokens(inp, T1, 29), initial_state=s1, v_hist=hist)
        _close(o1, out[:, :T1], 1e-12, f"prefix outputs (T1={T1})")
        _close(o2, out[:, T1:], 1e-12, f"resumed outputs (T1={T1})")
        _close(s2, fs, 1e-12, f"resumed final state (T1={T1})")


def pin_initial_state_gated_deltanet(fwd):
    """L = 0 from a given state: the explicit-matrix Gated DeltaNet started at S0."""
    inp = random_small(2, 17, 2, 6, 5, 0, 3, seed=26)
    S0 = np.random.default_rng(3).standard_normal((2, 2, 5, 6))
    out, fs, _ = fwd(inp, initial_state=S0)
    ref_o, ref_s = gdn_explicit(inp, S0=S0)
    _close(out, ref_o, 1e-12, "outputs")
    _close(fs, ref_s, 1e-12, "final state")


ALL_PINS = [pin_l0_is_gated_deltanet, pin_zero_conv_is_gated_deltanet, pin_write_rank,
            pin_telescoping, pin_brute_force_products, pin_prefix_sum, pin_no_write_no_output,
            pin_shortconv, pin_direction, pin_gain_and_gelu, pin_confidence_gate,
            pin_gate_scales_write, pin_padding,
            pin_causality, pin_identity_activation, pin_resume_is_markov,
            pin_initial_state_gated_deltanet]


# ---- gradients (oracle.grad): pinned to the C oracle above, an independent implementation ----

def _grad_case(seed, L=2, ragged=True, T=13):
    inp = random_small(2, T, 2, 4, 4, L, 3, seed=seed, ragged=ragged)
    rng = np.random.default_rng(seed)
    d_out = rng.standard_normal((2, T, 2, 4))
    d_fs = rng.standard_normal((2, 2, 4, 4))
    return inp, d_out, d_fs


def pin_grad_forward_matches(fwd, grad_mod):
    """The differentiable restatement gives the C oracle's outputs and final state."""
    for seed, L, ragged, act in ((40, 2, True, False), (41, 0, False, False), (42, 3, True, True)):
        inp, _, _ = _grad_case(seed, L, ragged)
        p = {n: inp[n].double() for n in grad_mod.GRAD_KEYS}
        with torch.no_grad():
            o, s = grad_mod.forward_torch(p, L, seq_lens=inp.get("seq_lens"), identity_act=act)
        ro, rs, _ = fwd(inp, identity_act=act)
        _close(o.numpy(), ro, 1e-12, f"outputs (L={L})")
        _close(s.numpy(), rs, 1e-12, f"final state (L={L})")


def pin_grad_finite_difference(fwd, grad_mod):
    """Every gradient along a random direction equals the central difference of the
    C oracle's  sum(out * d_out) + sum(final_state * d_fs)  (step 1e-5, fp64)."""
    for seed, L, act in ((43, 2, False), (44, 3, True)):
        inp, d_out, d_fs = _grad_case(seed, L)
        g = grad_mod.backward(inp, d_out, d_fs, identity_act=act)

        def f(x):
            o, s, _ = fwd(x, identity_act=act)
            return float(np.sum(o * d_out) + np.sum(s * d_fs))
        rng = np.random.default_rng(seed + 100)
        eps = 1e-5
        for n in grad_mod.GRAD_KEYS:
            base = inp[n].double()
            delta = torch.from_numpy(rng.standard_normal(tuple(base.shape)))
            xp, xm = dict(inp), dict(inp)
            xp[n] = base + eps * delta
            xm[n] = base - eps * delta
            fd = (f(xp) - f(xm)) / (2 * eps)
            an = float(np.sum(g[n] * delta.numpy()))
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), f"d/d{n} (L={L}): fd {fd:.9e} vs {an:.9e}"


def pin_grad_dq_closed_form(fwd, grad_mod):
    """o_t = S_t q_t, so dq_t = S_t^T do_t, with S_t the final state of the C oracle run
    on tokens [0, t] (zero for padding tokens, whose output is fixed at 0)."""
    inp, d_out, _ = _grad_case(45, 2, True, T=9)
    g = grad_mod.backward(inp, d_out, None)
    lens = inp["seq_lens"].numpy()
    for t in range(9):
        _, s, _ = fwd(_slice_tokens(inp, 0, t + 1))
        for b in range(2):
            for h in range(2):
                if t < lens[b]:
                    _close(g["q"][b, t, h], s[b, h].T @ d_out[b, t, h], 1e-12, f"dq (t={t})")
                else:
                    assert not np.any(g["q"][b, t, h]), f"dq of a padding token (t={t})"


GRAD_PINS = [pin_grad_forward_matches, pin_grad_finite_difference, pin_grad_dq_closed_form]
