"""GPU parity of the resumed forward pass (initial state + v history) and of the
single-token decode step, against the fp64 oracle run on the whole sequence."""
import numpy as np
import pytest
import torch

import oracle
from linear_recurrent_sequence_causal_gb300 import inputs as I
from linear_recurrent_sequence_causal_gb300 import prism
from tests.parity import check

pytestmark = pytest.mark.gpu

TOKEN_KEYS = ("q", "k", "v", "log_alpha", "beta")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("CUDA GPU required for -m gpu tests")
    prism.load()


def _tokens(d, t0, t1):
    """Tokens [t0, t1) of a device input dict (contiguous copies)."""
    out = dict(d)
    for n in TOKEN_KEYS:
        out[n] = d[n][:, t0:t1].contiguous()
    out["seq_lens"] = None
    return out


def _run(d, L, chunk, **kw):
    return prism.prism_forward_from(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["conv_w"],
                                    d["Wk"], d["Wp"], d["wbeta"], L, chunk, **kw)


@pytest.mark.parametrize("dtype,D,chunk,L,T1", [("bf16", 128, 64, 2, 69), ("bf16", 32, 32, 3, 40),
                                                ("f32", 32, 16, 2, 21), ("bf16", 128, 32, 1, 3),
                                                ("bf16", 64, 64, 0, 64)])
def test_split_sequence_matches_one_run(dtype, D, chunk, L, T1):
    """Run [0, T1), then [T1, T) from its final state and last w v rows: the outputs and
    final state of the oracle's single run over [0, T)."""
    wl = I.Workload("case", dtype, 2, 3 * chunk + 11, 2, D, D, L, 4, chunk, seed=60 + D + L)
    inp = I.generate(wl)
    ro, rs, _ = oracle.forward(inp)
    d = prism.inputs_to_device(inp)
    out1, s1 = _run(_tokens(d, 0, T1), L, chunk)
    hist = prism.v_history(d["v"], wl.w, T1)
    out2, s2 = _run(_tokens(d, T1, wl.T), L, chunk, initial_state=s1, v_hist=hist)
    torch.cuda.synchronize()
    check(torch.cat([out1, out2], dim=1), s2, ro, rs, dtype, what=f"split at {T1}")


@pytest.mark.parametrize("dtype,D,chunk,L", [("bf16", 128, 64, 4), ("f32", 16, 16, 1), ("bf16", 64, 32, 2)])
def test_forward_from_given_state_and_history(dtype, D, chunk, L):
    """A given entering state and history against the oracle started from the same."""
    wl = I.Workload("case", dtype, 2, 2 * chunk + 7, 2, D, D, L, 4, chunk, seed=70 + D)
    inp = I.generate(wl)
    warm = I.generate(I.Workload("w", dtype, 2, 50, 2, D, D, L, 4, chunk, seed=71 + D))
    for key in ("conv_w", "Wk", "Wp", "wbeta"):            # same layer, different earlier tokens
        warm[key] = inp[key]
    _, s0, _ = oracle.forward(warm)                         # a realistic entering state
    hist = warm["v"][:, -wl.w:].permute(0, 2, 1, 3).contiguous()
    ro, rs, _ = oracle.forward(inp, initial_state=s0, v_hist=hist)
    d = prism.inputs_to_device(inp)
    out, fs = _run(d, L, chunk, initial_state=torch.tensor(s0, dtype=torch.float32, device="cuda"),
                   v_hist=hist.to("cuda"))
    torch.cuda.synchronize()
    check(out, fs, ro, rs, dtype, what="given state")


@pytest.mark.parametrize("dtype,D,L,no_gelu,B,H,T0,n", [
    ("bf16", 128, 2, False, 2, 3, 37, 6), ("bf16", 64, 4, False, 2, 3, 37, 6),
    ("f32", 32, 2, False, 2, 3, 37, 6), ("bf16", 16, 0, False, 2, 3, 37, 6),
    ("bf16", 32, 3, True, 2, 3, 37, 6),
    # an odd batch (sequences are grouped in pairs per CTA), a single sequence
    ("bf16", 128, 2, False, 3, 2, 21, 3), ("bf16", 128, 4, False, 1, 2, 21, 3),
    # enough CTAs that the weight ring holds fewer slices than the 2L of a step
    ("bf16", 128, 8, False, 48, 8, 5, 2), ("f32", 64, 8, True, 96, 8, 5, 2)])
def test_decode_steps_match_oracle(dtype, D, L, no_gelu, B, H, T0, n):
    """A chunked prefix, then one token at a time: outputs and state of the oracle's
    single run over all tokens."""
    chunk = 16
    wl = I.Workload("case", dtype, B, T0 + n, H, D, D, L, 4, chunk, seed=80 + D + L + B)
    inp = I.generate(wl)
    ro, rs, _ = oracle.forward(inp, identity_act=no_gelu)
    d = prism.inputs_to_device(inp)
    out0, state = _run(_tokens(d, 0, T0), L, chunk, no_gelu=no_gelu)
    hist = prism.v_history(d["v"], wl.w, T0)
    outs = [out0]
    for t in range(T0, T0 + n):
        tok = {k: d[k][:, t].clone() for k in TOKEN_KEYS}   # own storage: 16-byte aligned
        o = prism.prism_decode_step(tok["q"], tok["k"], tok["v"], tok["log_alpha"], tok["beta"],
                                    d["conv_w"], d["Wk"], d["Wp"], d["wbeta"], L, state, hist,
                                    no_gelu=no_gelu)
        outs.append(o[:, None])
    torch.cuda.synchronize()
    check(torch.cat(outs, dim=1), state, ro, rs, dtype, what="decode")
    # the history now holds the last w tokens
    np.testing.assert_array_equal(hist.float().cpu().numpy(),
                                  prism.v_history(d["v"], wl.w).float().cpu().numpy())


def _random_decode_cases(n, seed):
    import random
    rnd = random.Random(seed)
    out = []
    for _ in range(n):
        dtype = rnd.choice(["bf16", "bf16", "f32"])
        D = rnd.choice([16, 32, 64] if dtype == "f32" else [16, 32, 64, 128])
        w = rnd.randint(1, 8)
        out.append((dtype, D, rnd.randint(0, 8), w, rnd.randint(1, 9), rnd.randint(1, 4), rnd.randint(w, 60),
                    rnd.randint(1, 5), rnd.random() < 0.2))
    return out


@pytest.mark.parametrize("dtype,D,L,w,B,H,T0,n,no_gelu", _random_decode_cases(12, 5))
def test_decode_random_shapes(dtype, D, L, w, B, H, T0, n, no_gelu):
    """Seeded random shapes (conv widths 1..8 included): a chunked prefix, then decode
    steps, against the oracle's single run."""
    chunk = 16
    wl = I.Workload("case", dtype, B, T0 + n, H, D, D, L, w, chunk, seed=900 + T0 + D + L + w)
    inp = I.generate(wl)
    ro, rs, _ = oracle.forward(inp, identity_act=no_gelu)
    d = prism.inputs_to_device(inp)
    out0, state = _run(_tokens(d, 0, T0), L, chunk, no_gelu=no_gelu)
    hist = prism.v_history(d["v"], w, T0)
    outs = [out0]
    for t in range(T0, T0 + n):
        tok = {k: d[k][:, t].clone() for k in TOKEN_KEYS}
        o = prism.prism_decode_step(tok["q"], tok["k"], tok["v"], tok["log_alpha"], tok["beta"],
                                    d["conv_w"], d["Wk"], d["Wp"], d["wbeta"], L, state, hist,
                                    no_gelu=no_gelu)
        outs.append(o[:, None])
    torch.cuda.synchronize()
    check(torch.cat(outs, dim=1), state, ro, rs, dtype, what="decode, random shape")
