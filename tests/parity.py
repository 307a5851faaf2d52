"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI,
run the oracle on the same host inputs, and compare with the specified tolerances
(fp32: normwise 1e-4; bf16: max|d| <= 2e-2 RMS(o_ref) and relative Frobenius error
of the final state <= 1e-2; padding exactly 0)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from linear_recurrent_sequence_causal_gb300 import prism

F32_TOL = 1e-4
BF16_OUT_TOL = 2e-2
BF16_STATE_TOL = 1e-2


def gpu_forward(inp: dict, L: int, chunk: int, *, no_gelu=False, want_state=True):
    d = prism.inputs_to_device(inp)
    out, fs = prism.forward_inputs(d, L, chunk, no_gelu=no_gelu, want_state=want_state)
    torch.cuda.synchronize()
    return out, fs


def to64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def check(out_gpu, fs_gpu, out_ref, fs_ref, dtype: str, *, bh=None, seq_lens=None, what=""):
    """Compare GPU results with the oracle's. ``bh`` restricts to (b, h) pairs;
    ``seq_lens`` adds the exact-zero check on padding. Returns the error dict."""
    o = to64(out_gpu) if torch.is_tensor(out_gpu) else out_gpu
    s = to64(fs_gpu) if (fs_gpu is not None and torch.is_tensor(fs_gpu)) else fs_gpu
    if bh is not None:
        bi = np.array([b for b, _ in bh]); hi = np.array([h for _, h in bh])
        o_g, o_r = o[bi, :, hi], out_ref[bi, :, hi]
        s_g = s[bi, hi] if s is not None else None
        s_r = fs_ref[bi, hi]
    else:
        o_g, o_r, s_g, s_r = o, out_ref, s, fs_ref
    assert np.all(np.isfinite(o_g)), f"{what}: non-finite output"
    err = {}
    if dtype == "f32":
        err["out"] = np.max(np.abs(o_g - o_r)) / max(np.max(np.abs(o_r)), 1e-30)
        assert err["out"] <= F32_TOL, f"{what}: fp32 output error {err['out']:.3e}"
        if s_g is not None:
            err["state"] = np.max(np.abs(s_g - s_r)) / max(np.max(np.abs(s_r)), 1e-30)
            assert err["state"] <= F32_TOL, f"{what}: fp32 state error {err['state']:.3e}"
    else:
        rms = np.sqrt(np.mean(o_r ** 2))
        err["out"] = np.max(np.abs(o_g - o_r)) / rms
        assert err["out"] <= BF16_OUT_TOL, f"{what}: bf16 output error {err['out']:.3e} x RMS"
        if s_g is not None:
            err["state"] = np.linalg.norm(s_g - s_r) / max(np.linalg.norm(s_r), 1e-30)
            assert err["state"] <= BF16_STATE_TOL, f"{what}: bf16 state error {err['state']:.3e}"
    if seq_lens is not None:
        lens = np.asarray(seq_lens)
        for b, n in enumerate(lens.tolist()):
            assert np.all(o[b, n:] == 0.0), f"{what}: padding of sequence {b} not zero"
    return err


def chunk_maps(inp, kl, dl, C):
    """fp64 reference of what the bf16 prepare stage writes per chunk:
    W, Kt, Qt, U, O_intra ([B,H,NC,C,D]), N ([B,H,NC,D,D]) and gamma_C ([B,H,NC]),
    from the inputs and the oracle's per-token factors k^(l), beta^(l) delta^(l)."""
    q, k, v = (inp[n].double().numpy() for n in ("q", "k", "v"))
    la, be = inp["log_alpha"].double().numpy(), inp["beta"].double().numpy()
    B, T, H, D = q.shape
    L = kl.shape[3]
    NC = (T + C - 1) // C
    sl = inp.get("seq_lens")
    names = ("W", "Kt", "Qt", "U", "Oi")
    res = {n: np.zeros((B, H, NC, C, D)) for n in names}
    res["N"] = np.zeros((B, H, NC, D, D))
    res["gC"] = np.ones((B, H, NC))
    for b in range(B):
        n_len = T if sl is None else int(sl[b])
        for h in range(H):
            for c in range(NC):
                t0 = c * C
                nv = min(C, n_len - t0)
                if nv <= 0:
                    continue
                def pad(x):
                    y = np.zeros((C,) + x.shape[1:])
                    y[:nv] = x[:nv]
                    return y
                Q, K, V = (pad(a[b, t0:t0 + C, h]) for a in (q, k, v))
                bt = pad(be[b, t0:t0 + C, h])
                g = np.cumsum(pad(la[b, t0:t0 + C, h]))
                gam = np.exp(g)
                G = np.exp(np.minimum(g[:, None] - g[None, :], 0.0))
                low, inc = np.tril(np.ones((C, C)), -1), np.tril(np.ones((C, C)))
                Kl = [np.nan_to_num(pad(kl[b, t0:t0 + C, h, l])) for l in range(L)]
                Dl = [np.nan_to_num(pad(dl[b, t0:t0 + C, h, l])) for l in range(L)]
                dec = np.exp(g[-1] - g)
                R = sum(((K @ Kl[l].T) * G * low) @ Dl[l] for l in range(L)) if L else 0.0
                Ol = sum(((Q @ Kl[l].T) * G * inc) @ Dl[l] for l in range(L)) if L else 0.0
                A = bt[:, None] * (K @ K.T) * G * low
                Tm = np.linalg.inv(np.eye(C) + A)
                P = (Q @ K.T) * G * inc
                W = Tm @ ((bt * gam)[:, None] * K)
                U = Tm @ (bt[:, None] * (V - R))
                res["W"][b, h, c] = W
                res["Kt"][b, h, c] = dec[:, None] * K
                res["Qt"][b, h, c] = gam[:, None] * Q - P @ W
                res["U"][b, h, c] = U
                res["Oi"][b, h, c] = P @ U + Ol
                if L:
                    res["N"][b, h, c] = sum((dec[:, None] * Dl[l]).T @ Kl[l] for l in range(L))
                res["gC"][b, h, c] = np.exp(g[-1])
    return res


def read_pair(ws, layout, name, shape):
    """An interleaved fp16 region (two [..., C, F] maps sharing 16-byte column pieces:
    in each piece the C rows of the first map, then the C rows of the second) as two
    CPU fp64 numpy arrays in plain [..., C, F] order."""
    off = layout[name]
    C, F = shape[-2], shape[-1]
    n = int(np.prod(shape)) * 2 * 2
    flat = ws[off:off + n].view(torch.float16).double().cpu().numpy()
    x = flat.reshape(tuple(shape[:-2]) + (F // 8, 2, C, 8))
    first, second = x[..., 0, :, :], x[..., 1, :, :]
    return (np.moveaxis(first, -3, -2).reshape(shape), np.moveaxis(second, -3, -2).reshape(shape))


def read_region(ws, layout, name, dtype, shape, piece_major=True):
    """One workspace region as a CPU fp64 numpy array.  Per-chunk arrays
    (shape [..., R, F]) are stored piece-major: 16-byte column pieces, rows
    contiguous inside a piece; they are returned in plain [..., R, F] order."""
    off = layout[name]
    esz = torch.tensor([], dtype=dtype).element_size()
    n = int(np.prod(shape)) * esz
    flat = ws[off:off + n].view(dtype).double().cpu().numpy()
    if len(shape) < 2 or not piece_major:
        return flat.reshape(shape)
    R, F = shape[-2], shape[-1]
    V = 16 // esz
    x = flat.reshape(shape[:-2] + (F // V, R, V))
    return np.moveaxis(x, -3, -2).reshape(shape)
