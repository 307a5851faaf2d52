"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI,
run the oracle on the same host inputs, and compare with the tolerances of the
design notes (fp32: normwise 1e-4; bf16: max|d| <= 2e-2 RMS(o_ref) and
relative Frobenius error of the final state <= 1e-2; padding exactly 0)."""
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
