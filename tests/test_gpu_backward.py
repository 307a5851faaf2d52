"""GPU parity of the backward pass (prism_backward) against the gradient oracle
(oracle/grad.py: autograd of the fp64 token recurrence, pinned to the C oracle by finite
differences).

Tolerance: the GPU computes every gradient in fp32 from the same (bf16-exact or fp32)
inputs, so the gap to the fp64 reference is fp32 rounding carried through the backward
recurrence and the token sums of the weight gradients.  Each gradient tensor is compared
normwise, max|g_gpu - g_ref| / max|g_ref| <= 2e-4 (the forward's fp32 bound of 1e-4,
doubled for the second pass over the same operations); padding tokens' gradients are
exactly zero.
"""
import numpy as np
import pytest
import torch

from linear_recurrent_sequence_causal_gb300 import inputs as I
from linear_recurrent_sequence_causal_gb300 import prism
from oracle import grad as G

pytestmark = pytest.mark.gpu

GRAD_TOL = 2e-4


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("CUDA GPU required for -m gpu tests")
    prism.load()


def _run(dtype, D, L, T, B, H, w, ragged, no_gelu, with_fs, seed):
    wl = I.Workload("bwd", dtype, B, T, H, D, D, L, w, 16, seed=seed, ragged=ragged)
    inp = I.generate(wl)
    if ragged:                                   # lengths over the whole range, one full
        g = torch.Generator().manual_seed(seed)
        lens = torch.randint(1, T + 1, (B,), generator=g, dtype=torch.int32)
        lens[0] = T
        inp["seq_lens"] = lens
    rng = np.random.default_rng(seed)
    d_out = rng.standard_normal((B, T, H, D)).astype(np.float32)
    d_fs = rng.standard_normal((B, H, D, D)).astype(np.float32) if with_fs else None
    ref = G.backward(inp, d_out.astype(np.float64), None if d_fs is None else d_fs.astype(np.float64),
                     identity_act=no_gelu)
    d = prism.inputs_to_device(inp)
    gg = prism.prism_backward(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["conv_w"],
                              d["Wk"], d["Wp"], d["wbeta"], L, torch.from_numpy(d_out).cuda(),
                              d_final_state=None if d_fs is None else torch.from_numpy(d_fs).cuda(),
                              seq_lens=d.get("seq_lens"), no_gelu=no_gelu)
    torch.cuda.synchronize()
    return inp, ref, gg


CASES = [
    # dtype, D, L, T, B, H, w, ragged, no_gelu, d_final_state
    ("f32", 16, 2, 37, 2, 2, 4, True, False, True),
    ("bf16", 32, 3, 50, 2, 2, 3, True, True, False),
    ("bf16", 64, 0, 33, 1, 2, 4, False, False, True),
    ("bf16", 128, 2, 40, 1, 2, 4, False, False, True),
    ("f32", 64, 4, 21, 2, 1, 8, True, False, False),
    ("bf16", 128, 1, 17, 1, 1, 1, False, False, False),
    ("bf16", 16, 1, 20, 20, 8, 4, True, False, True),     # 160 sequences: one CTA per (b, h)
    ("f32", 32, 2, 24, 10, 10, 3, False, False, True),    # 100 sequences: two row slices
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_backward_matches_oracle(case):
    dtype, D, L, T, B, H, w, ragged, no_gelu, with_fs = case
    inp, ref, gg = _run(dtype, D, L, T, B, H, w, ragged, no_gelu, with_fs, seed=90 + D + L + T)
    errs = {}
    for n in G.GRAD_KEYS:
        if L == 0 and n in ("Wk", "Wp", "wbeta"):
            continue
        gpu = gg[n].double().cpu().numpy()
        r = ref[n]
        if n in ("Wk", "Wp", "wbeta"):
            r = r[:, :L]
        assert np.all(np.isfinite(gpu)), f"d{n}: non-finite"
        scale = max(np.max(np.abs(r)), 1e-30)
        errs[n] = np.max(np.abs(gpu - r)) / scale
    bad = {n: e for n, e in errs.items() if e > GRAD_TOL}
    assert not bad, f"gradient errors above {GRAD_TOL}: {bad} (all: {errs})"
    if inp.get("seq_lens") is not None:
        for b, n in enumerate(inp["seq_lens"].tolist()):
            for key in ("q", "k", "v", "log_alpha", "beta"):
                assert not torch.any(gg[key][b, n:]), f"d{key} of padding tokens in sequence {b}"


def test_backward_is_deterministic():
    _, _, g1 = _run("bf16", 64, 2, 45, 2, 2, 4, True, False, True, seed=7)
    _, _, g2 = _run("bf16", 64, 2, 45, 2, 2, 4, True, False, True, seed=7)
    for n in G.GRAD_KEYS:
        assert torch.equal(g1[n], g2[n]), f"d{n} differs between two identical calls"


def test_backward_short_sequences_and_an_empty_one():
    """T shorter than a checkpoint block, one sequence of length 0 and one of length 1: the
    gradients of the others match the oracle and the empty one's are exactly zero."""
    B, T, H, D, L = 4, 7, 2, 32, 2
    wl = I.Workload("bwd", "bf16", B, T, H, D, D, L, 4, 16, seed=5, ragged=True)
    inp = I.generate(wl)
    inp["seq_lens"] = torch.tensor([T, 0, 1, 5], dtype=torch.int32)
    rng = np.random.default_rng(5)
    d_out = rng.standard_normal((B, T, H, D)).astype(np.float32)
    d_fs = rng.standard_normal((B, H, D, D)).astype(np.float32)
    ref = G.backward(inp, d_out.astype(np.float64), d_fs.astype(np.float64))
    d = prism.inputs_to_device(inp)
    gg = prism.prism_backward(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["conv_w"],
                              d["Wk"], d["Wp"], d["wbeta"], L, torch.from_numpy(d_out).cuda(),
                              d_final_state=torch.from_numpy(d_fs).cuda(), seq_lens=d["seq_lens"])
    torch.cuda.synchronize()
    for n in G.GRAD_KEYS:
        gpu = gg[n].double().cpu().numpy()
        r = ref[n]
        assert np.all(np.isfinite(gpu)), f"d{n}: non-finite"
        err = np.max(np.abs(gpu - r)) / max(np.max(np.abs(r)), 1e-30)
        assert err <= GRAD_TOL, f"d{n}: {err:.3e}"
    for key in ("q", "k", "v", "log_alpha", "beta"):
        assert not torch.any(gg[key][1]), f"d{key} of the empty sequence"


@pytest.mark.parametrize("D", [32, 128])
def test_backward_every_sequence_empty(D):
    """Every sequence of length 0: no token takes part, so every gradient, those of the
    per-head parameters included, is exactly zero whatever the inputs and d_out hold."""
    B, T, H, L = 3, 40, 2, 2
    wl = I.Workload("bwd", "bf16", B, T, H, D, D, L, 4, 16, seed=6)
    inp = I.generate(wl)
    inp["seq_lens"] = torch.zeros(B, dtype=torch.int32)
    d = prism.inputs_to_device(inp)
    d_out = torch.randn(B, T, H, D, device="cuda")
    d_fs = torch.randn(B, H, D, D, device="cuda")
    gg = prism.prism_backward(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["conv_w"],
                              d["Wk"], d["Wp"], d["wbeta"], L, d_out, d_final_state=d_fs,
                              seq_lens=d["seq_lens"])
    torch.cuda.synchronize()
    for n in G.GRAD_KEYS:
        assert torch.count_nonzero(gg[n]).item() == 0, f"d{n}"


def _random_backward_cases(n, seed):
    import random
    rnd = random.Random(seed)
    out = []
    for _ in range(n):
        dtype = rnd.choice(["bf16", "bf16", "f32"])
        D = rnd.choice([16, 32, 64] if dtype == "f32" else [16, 32, 64, 128])
        out.append((dtype, D, rnd.randint(0, 5), rnd.randint(1, 70), rnd.randint(1, 4), rnd.randint(1, 3),
                    rnd.randint(1, 8), rnd.random() < 0.5, rnd.random() < 0.2, rnd.random() < 0.5))
    return out


@pytest.mark.parametrize("case", _random_backward_cases(12, 11), ids=lambda c: "-".join(map(str, c)))
def test_backward_random_shapes(case):
    """Seeded random shapes over every axis the backward pass supports, against the
    gradient oracle at the same tolerance."""
    dtype, D, L, T, B, H, w, ragged, no_gelu, with_fs = case
    inp, ref, gg = _run(dtype, D, L, T, B, H, w, ragged, no_gelu, with_fs, seed=1500 + D + L + T)
    for n in G.GRAD_KEYS:
        if L == 0 and n in ("Wk", "Wp", "wbeta"):
            continue
        gpu = gg[n].double().cpu().numpy()
        r = ref[n][:, :L] if n in ("Wk", "Wp", "wbeta") else ref[n]
        assert np.all(np.isfinite(gpu)), f"d{n}: non-finite"
        err = np.max(np.abs(gpu - r)) / max(np.max(np.abs(r)), 1e-30)
        assert err <= GRAD_TOL, f"d{n}: {err:.3e}"
