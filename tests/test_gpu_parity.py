"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded inputs, for the five workloads and the edge cases."""
import numpy as np
import pytest
import torch

import oracle
from linear_recurrent_sequence_causal_gb300 import inputs as I
from linear_recurrent_sequence_causal_gb300 import prism
from tests.parity import check, gpu_forward, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("CUDA GPU required for -m gpu tests")
    prism.load()


def test_tiny_f32_workload():
    wl = I.get_workload("tiny_f32")
    inp = I.generate(wl)
    out, fs = gpu_forward(inp, wl.L, wl.chunk)
    ro, rs, _ = oracle.forward(inp)
    check(out, fs, ro, rs, "f32", what="tiny_f32")


@pytest.mark.parametrize("L", [0, 1, 2, 4])
def test_lsweep_bf16_workload(L):
    wl = I.get_workload("lsweep_bf16")
    inp = I.generate(wl, L=L)
    out, fs = gpu_forward(inp, L, wl.chunk)
    ro, rs, _ = oracle.forward(inp, L=L)
    check(out, fs, ro, rs, "bf16", what=f"lsweep L={L}")


def test_lsweep_l0_is_gated_deltanet():
    """At L = 0 the GPU path is the plain gated delta rule: it must match the
    oracle run with the refinement weights removed entirely."""
    wl = I.get_workload("lsweep_bf16")
    inp = I.generate(wl, L=4)
    out, fs = gpu_forward(inp, 0, wl.chunk)
    ro, rs, _ = oracle.forward({**inp, "Wk": inp["Wk"][:, :0], "Wp": inp["Wp"][:, :0],
                                "wbeta": inp["wbeta"][:, :0]}, L=0)
    check(out, fs, ro, rs, "bf16", what="lsweep L=0 vs gated delta rule")


def test_recsys_bf16_workload_ragged_with_nan_padding():
    wl = I.get_workload("recsys_bf16")
    inp = I.generate(wl)
    lens = inp["seq_lens"]
    poisoned = dict(inp)
    for name in ("q", "k", "v", "log_alpha", "beta"):
        x = inp[name].clone()
        for b, n in enumerate(lens.tolist()):
            x[b, n:] = float("nan")
        poisoned[name] = x
    out, fs = gpu_forward(poisoned, wl.L, wl.chunk)
    ro, rs, _ = oracle.forward(inp)
    check(out, fs, ro, rs, "bf16", seq_lens=lens, what="recsys_bf16")
    assert torch.isfinite(fs).all()


def test_lm_bf16_workload_sampled_heads():
    wl = I.get_workload("lm_bf16")
    inp = I.generate(wl)
    out, fs = gpu_forward(inp, wl.L, wl.chunk)
    bh = [(0, 0), (1, 5), (3, 15), (7, 9), (4, 2), (6, 11)]
    ro, rs, _ = oracle.forward(inp, bh_items=bh)
    check(out, fs, ro, rs, "bf16", bh=bh, what="lm_bf16 sampled (b,h)")
    assert torch.isfinite(out).all() and torch.isfinite(fs).all()


def test_longctx_bf16_workload():
    """Full T = 65536 run: outputs of the first 4096 tokens match the oracle on
    the 4096-token prefix (causality); a prefix run's final state matches; two
    heads are checked by the oracle over the whole length."""
    wl = I.get_workload("longctx_bf16")
    inp = I.generate(wl)
    out, fs = gpu_forward(inp, wl.L, wl.chunk)
    assert torch.isfinite(fs).all()
    P = 4096
    pre = {k: (v[:, :P].contiguous() if k in ("q", "k", "v", "log_alpha", "beta") else v)
           for k, v in inp.items()}
    heads = [(0, 0), (0, 13), (0, 31)]
    ro, rs, _ = oracle.forward(pre, bh_items=heads)
    check(out[:, :P], None, ro, rs, "bf16", bh=heads, what="longctx prefix outputs")
    pout, pfs = gpu_forward(pre, wl.L, wl.chunk)
    check(pout, pfs, ro, rs, "bf16", bh=heads, what="longctx prefix run")
    # L = 0 invariant on the prefix
    o0, s0 = gpu_forward(pre, 0, wl.chunk)
    r0, q0, _ = oracle.forward(pre, L=0, bh_items=heads)
    check(o0, s0, r0, q0, "bf16", bh=heads, what="longctx prefix L=0")
    # whole length, two heads
    full_heads = [(0, 7), (0, 22)]
    fo, fsr, _ = oracle.forward(inp, bh_items=full_heads)
    check(out, fs, fo, fsr, "bf16", bh=full_heads, what="longctx full length")


SHAPES = [
    # dtype, B, T, H, D, L, w, chunk, ragged
    ("f32", 2, 37, 3, 16, 2, 4, 16, False),
    ("f32", 1, 100, 2, 32, 3, 3, 32, True),
    ("f32", 2, 70, 1, 64, 1, 4, 32, False),
    ("f32", 1, 130, 1, 64, 2, 2, 64, False),
    ("bf16", 3, 1, 2, 16, 2, 4, 16, False),
    ("bf16", 2, 15, 1, 32, 1, 4, 16, False),
    ("bf16", 2, 77, 2, 32, 3, 4, 32, True),
    ("bf16", 1, 200, 3, 64, 2, 4, 64, True),
    ("bf16", 2, 129, 2, 128, 2, 4, 64, False),
    ("bf16", 1, 95, 2, 128, 5, 8, 32, True),
    ("bf16", 1, 160, 2, 128, 1, 1, 16, False),
    ("bf16", 2, 64, 1, 16, 8, 4, 64, False),
]


@pytest.mark.parametrize("dtype,B,T,H,D,L,w,chunk,ragged", SHAPES)
def test_shapes_and_tails(dtype, B, T, H, D, L, w, chunk, ragged):
    wl = I.Workload("case", dtype, B, T, H, D, D, L, w, chunk, seed=1000 + T, ragged=False)
    inp = I.generate(wl)
    if ragged:
        g = torch.Generator().manual_seed(T)
        lens = torch.randint(0, T + 1, (B,), generator=g, dtype=torch.int32)
        lens[0] = T
        if B > 1:
            lens[-1] = 0      # an empty sequence
        inp["seq_lens"] = lens
    out, fs = gpu_forward(inp, L, chunk)
    ro, rs, _ = oracle.forward(inp)
    if ragged:
        for b, n in enumerate(inp["seq_lens"].tolist()):
            if n == 0:
                rs[b] = 0.0
    check(out, fs, ro, rs, dtype, seq_lens=inp.get("seq_lens"),
          what=f"{dtype} B{B} T{T} H{H} D{D} L{L} w{w} C{chunk}")


@pytest.mark.parametrize("dtype,D,C,L", [("bf16", 32, 32, 3), ("bf16", 64, 64, 2), ("bf16", 128, 64, 4),
                                         ("f32", 32, 32, 2)])
def test_every_sequence_empty(dtype, D, C, L):
    """A batch whose sequences all have length 0: every prepare CTA finds no chunk, the
    outputs and final states are exactly zero whatever the (NaN) inputs hold, and the
    device status word reads 0."""
    B, T, H = 3, 100, 2
    wl = I.Workload("case", dtype, B, T, H, D, D, L, 4, C, seed=77)
    inp = I.generate(wl)
    for name in ("q", "k", "v", "log_alpha", "beta"):
        inp[name] = torch.full_like(inp[name], float("nan"))
    inp["seq_lens"] = torch.zeros(B, dtype=torch.int32)
    d = prism.inputs_to_device(inp)
    dims = prism.make_dims(B, T, H, D, D, 4, L, C, wl.torch_dtype)
    ws = prism.alloc_workspace(dims, "cuda")
    out, fs = prism.forward_inputs(d, L, C, workspace=ws)
    assert prism.device_status(dims, ws) == 0
    assert torch.count_nonzero(out).item() == 0 and torch.count_nonzero(fs).item() == 0


def _random_cases(n, seed):
    """Seeded random shapes over every supported axis (dtype, d, L, w, chunk, T, ragged)."""
    import random
    rnd = random.Random(seed)
    out = []
    for i in range(n):
        dtype = rnd.choice(["bf16", "bf16", "f32"])
        D = rnd.choice([16, 32, 64] if dtype == "f32" else [16, 32, 64, 128])
        out.append((dtype, rnd.randint(1, 4), rnd.randint(1, 300), rnd.randint(1, 3), D,
                    rnd.randint(0, 8), rnd.randint(1, 8), rnd.choice([16, 32, 64]), rnd.random() < 0.5))
    return out


@pytest.mark.parametrize("dtype,B,T,H,D,L,w,chunk,ragged", _random_cases(64, 2026))
def test_random_shapes(dtype, B, T, H, D, L, w, chunk, ragged):
    """Random combinations of the supported axes against the oracle, at the dtype's
    tolerance (ragged batches hold an empty sequence when B > 1)."""
    wl = I.Workload("case", dtype, B, T, H, D, D, L, w, chunk, seed=3000 + T + 7 * D + L, ragged=False)
    inp = I.generate(wl)
    if ragged:
        g = torch.Generator().manual_seed(T + D)
        lens = torch.randint(0, T + 1, (B,), generator=g, dtype=torch.int32)
        if B > 1:
            lens[-1] = 0
        inp["seq_lens"] = lens
    d = prism.inputs_to_device(inp)
    dims = prism.make_dims(B, T, H, D, D, w, L, chunk, wl.torch_dtype)
    ws = prism.alloc_workspace(dims, "cuda")
    out, fs = prism.forward_inputs(d, L, chunk, workspace=ws)
    status = prism.device_status(dims, ws)
    ro, rs, tr = oracle.forward(inp, trace=True)
    if status & 2:
        # the bf16 path flagged a non-finite value: only a refinement chain that reached
        # the fp16 range of the tensor-core operands may do that
        assert dtype == "bf16" and L > 0, "non-finite flag on a path without fp16 operands"
        dl = np.asarray(tr["dl"])
        assert np.nanmax(np.abs(dl)) > 3e4, "non-finite output below the fp16 range"
        return
    assert status == 0
    if ragged:
        for b, n in enumerate(inp["seq_lens"].tolist()):
            if n == 0:
                rs[b] = 0.0
    check(out, fs, ro, rs, dtype, seq_lens=inp.get("seq_lens"),
          what=f"{dtype} B{B} T{T} H{H} D{D} L{L} w{w} C{chunk} ragged={ragged}")


def test_refinement_beyond_fp16_range_is_flagged():
    """A diverging refinement chain (L = 8, |delta^(l)| up to ~2e5) exceeds the fp16 range
    of the tensor-core operands: the bf16 path sets status bit 1 instead of returning
    non-finite outputs silently, and the fp32 path, which has no such limit, matches the
    oracle on the same values."""
    B, T, H, D, L, w, C = 1, 234, 2, 32, 8, 7, 16
    wl = I.Workload("case", "bf16", B, T, H, D, D, L, w, C, seed=3000 + T + 7 * D + L)
    inp = I.generate(wl)
    inp["seq_lens"] = torch.tensor([186], dtype=torch.int32)
    ro, rs, tr = oracle.forward(inp, trace=True)
    assert np.nanmax(np.abs(np.asarray(tr["dl"]))) > 65504
    d = prism.inputs_to_device(inp)
    dims = prism.make_dims(B, T, H, D, D, w, L, C, torch.bfloat16)
    ws = prism.alloc_workspace(dims, "cuda")
    prism.forward_inputs(d, L, C, workspace=ws)
    assert prism.device_status(dims, ws) & 2
    # the same inputs through the fp32 path
    f32 = {k: (v.float() if v is not None and v.dtype == torch.bfloat16 else v) for k, v in inp.items()}
    out, fs = gpu_forward(f32, L, C)
    check(out, fs, ro, rs, "f32", seq_lens=inp["seq_lens"], what="fp32 path, diverging chain")


@pytest.mark.parametrize("chunk", [16, 32, 64])
def test_chunk_size_invariance(chunk):
    wl = I.Workload("case", "bf16", 2, 300, 2, 64, 64, 3, 4, chunk, seed=77)
    inp = I.generate(wl)
    out, fs = gpu_forward(inp, wl.L, chunk)
    ro, rs, _ = oracle.forward(inp)
    check(out, fs, ro, rs, "bf16", what=f"chunk {chunk}")


def test_no_gelu_ablation():
    wl = I.Workload("case", "bf16", 2, 150, 2, 64, 64, 2, 4, 64, seed=5)
    inp = I.generate(wl)
    out, fs = gpu_forward(inp, wl.L, wl.chunk, no_gelu=True)
    ro, rs, _ = oracle.forward(inp, identity_act=True)
    check(out, fs, ro, rs, "bf16", what="no-GELU ablation")


@pytest.mark.parametrize("D,C,L,ragged", [(128, 64, 2, False), (64, 32, 3, True), (32, 16, 1, False),
                                          (16, 64, 0, True), (128, 32, 4, True), (32, 64, 0, False),
                                          (128, 64, 0, False)])
def test_prepare_stage_bf16(D, C, L, ragged):
    """The tensor-core prepare kernel's per-chunk maps (W, Kt, Qt, U, O_intra, N,
    gamma_C) against an fp64 numpy restatement fed with the oracle's factors."""
    from tests.parity import chunk_maps, read_pair, read_region
    wl = I.Workload("case", "bf16", 2, 3 * C + 5, 2, D, D, L, 4, C, seed=40 + D + C, ragged=False)
    inp = I.generate(wl)
    if ragged:
        inp["seq_lens"] = torch.tensor([wl.T, C + 3], dtype=torch.int32)
    d = prism.inputs_to_device(inp)
    dims = prism.make_dims(wl.B, wl.T, wl.H, D, D, wl.w, L, C, torch.bfloat16)
    ws = torch.zeros(prism.workspace_bytes(dims), dtype=torch.uint8, device="cuda")
    prism.prism_prepare(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["conv_w"], d["Wk"],
                        d["Wp"], d["wbeta"], L, C, ws, seq_lens=d.get("seq_lens"))
    torch.cuda.synchronize()
    lay = prism.workspace_layout(dims)
    NC = (wl.T + C - 1) // C
    _, _, tr = oracle.forward(inp, trace=True)
    ref = chunk_maps(inp, tr["kl"], tr["dl"], C)
    shp = (wl.B, wl.H, NC, C, D)
    W, Qth = read_pair(ws, lay, "WQ", shp)
    Qtl, Kt = read_pair(ws, lay, "QK", shp)
    got = {"W": W, "Kt": Kt, "Qt": Qth + Qtl,
           "U": read_region(ws, lay, "U", torch.float32, shp),
           "Oi": read_region(ws, lay, "Oi", torch.float32, shp),
           "gC": read_region(ws, lay, "gC", torch.float32, (wl.B, wl.H, NC))}
    if L:   # stored transposed: rows k, features v
        got["N"] = np.swapaxes(read_region(ws, lay, "N", torch.float32, (wl.B, wl.H, NC, D, D)), -1, -2)
    lens = [wl.T] * wl.B if not ragged else inp["seq_lens"].tolist()
    for name, g in got.items():
        r = ref[name]
        for b in range(wl.B):
            nch = (lens[b] + C - 1) // C
            gb, rb = g[b, :, :nch], r[b, :, :nch]
            err = np.max(np.abs(gb - rb)) / max(np.max(np.abs(rb)), 1e-30)
            assert err <= 5e-3, f"{name} (b={b}): normwise error {err:.3e}"


@pytest.mark.parametrize("D,C,L", [(128, 64, 2), (64, 32, 3), (32, 32, 2), (16, 16, 1)])
def test_weights_with_bits_below_fp16(D, C, L):
    """Weights drawn in fp32 (not bf16-rounded) have lo halves that matter: the weight
    conversion flags them (word 1 of the workspace's status region reads 1, against 0 for
    bf16-rounded weights) and the projections take their third pass with the lo halves.
    The outputs must match the oracle run on the same fp32 weights."""
    wl = I.Workload("case", "bf16", 2, 3 * C + 5, 2, D, D, L, 4, C, seed=91 + D)
    inp = I.generate(wl)
    g = torch.Generator().manual_seed(92 + D)
    inp_x = dict(inp)
    for n in ("Wk", "Wp"):
        inp_x[n] = torch.randn(inp[n].shape, generator=g, dtype=torch.float32) * D ** -0.5
    dims = prism.make_dims(wl.B, wl.T, wl.H, D, D, wl.w, L, C, torch.bfloat16)
    for src, want in ((inp, 0), (inp_x, 1)):
        d = prism.inputs_to_device(src)
        ws = torch.zeros(prism.workspace_bytes(dims), dtype=torch.uint8, device="cuda")
        prism.prism_prepare(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["conv_w"], d["Wk"],
                            d["Wp"], d["wbeta"], L, C, ws)
        torch.cuda.synchronize()
        assert int(ws[4:8].view(torch.int32).item()) == want
    out, fs = gpu_forward(inp_x, L, C)
    ro, rs, _ = oracle.forward(inp_x)
    check(out, fs, ro, rs, "bf16", what=f"fp32 weights d={D}")


def test_prepare_stage_f32():
    """fp32 path: the per-token factors in the workspace against the oracle trace."""
    from tests.parity import read_region
    wl = I.Workload("case", "f32", 2, 90, 2, 32, 32, 3, 4, 32, seed=9)
    inp = I.generate(wl)
    inp["seq_lens"] = torch.tensor([90, 41], dtype=torch.int32)
    d = prism.inputs_to_device(inp)
    dims = prism.make_dims(wl.B, wl.T, wl.H, 32, 32, wl.w, wl.L, wl.chunk, torch.float32)
    ws = torch.zeros(prism.workspace_bytes(dims), dtype=torch.uint8, device="cuda")
    prism.prism_prepare(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["conv_w"], d["Wk"],
                        d["Wp"], d["wbeta"], wl.L, wl.chunk, ws, seq_lens=d["seq_lens"])
    torch.cuda.synchronize()
    lay = prism.workspace_layout(dims)
    _, _, tr = oracle.forward(inp, trace=True)
    shp = (wl.B, wl.T, wl.H, wl.L, 32)
    for name, key in (("Kl", "kl"), ("Dl", "dl")):
        g = read_region(ws, lay, name, torch.float32, shp, piece_major=False)
        for b, n in enumerate([90, 41]):
            ref = tr[key][b, :n]
            err = np.max(np.abs(g[b, :n] - ref)) / np.max(np.abs(ref))
            assert err <= 1e-5, f"{name}: {err:.3e}"
            assert np.all(g[b, n:] == 0.0)


def test_deterministic():
    wl = I.Workload("case", "bf16", 2, 333, 4, 128, 128, 2, 4, 64, seed=3)
    d = prism.inputs_to_device(I.generate(wl))
    o1, s1 = prism.forward_inputs(d, wl.L, wl.chunk)
    o2, s2 = prism.forward_inputs(d, wl.L, wl.chunk)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(s1, s2)


@pytest.mark.parametrize("D,C,L,T,B,H,ragged", [(64, 32, 3, 300, 2, 2, False), (128, 64, 3, 333, 2, 2, False),
                                                 (128, 64, 4, 1000, 2, 2, False), (32, 32, 3, 200, 64, 2, True)])
def test_prepare_reruns_bit_identical(D, C, L, T, B, H, ragged):
    """A race between the tensor core and the epilogue warps (an MMA overwriting TMEM
    columns some warp still reads) shows as reruns that differ: the prepare stage's whole
    workspace, zeroed before each call, must be bit-identical over twelve calls.  Odd L
    puts the last refinement step's scores in the k_hat buffer of even steps."""
    wl = I.Workload("case", "bf16", B, T, H, D, D, L, 4, C, seed=77, ragged=ragged)
    d = prism.inputs_to_device(I.generate(wl))
    dims = prism.make_dims(B, T, H, D, D, 4, L, C, torch.bfloat16)
    runs = []
    for _ in range(12):
        ws = prism.alloc_workspace(dims, "cuda")
        ws.zero_()
        prism.prism_prepare(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["conv_w"], d["Wk"],
                            d["Wp"], d["wbeta"], L, C, ws, seq_lens=d.get("seq_lens"))
        runs.append(ws.cpu())
    assert all(torch.equal(runs[0], r) for r in runs[1:])


def test_recsys_bf16_reruns_bit_identical():
    wl = I.get_workload("recsys_bf16")
    d = prism.inputs_to_device(I.generate(wl))
    o1, s1 = prism.forward_inputs(d, wl.L, wl.chunk)
    for _ in range(8):
        o2, s2 = prism.forward_inputs(d, wl.L, wl.chunk)
        assert torch.equal(o1, o2) and torch.equal(s1, s2)


def test_causality():
    wl = I.Workload("case", "bf16", 1, 256, 2, 64, 64, 2, 4, 64, seed=4)
    inp = I.generate(wl)
    o1, _ = gpu_forward(inp, wl.L, wl.chunk)
    other = {k: (v.clone() if v is not None else None) for k, v in inp.items()}
    for name in ("q", "k", "v"):
        other[name][:, 150:] = -other[name][:, 150:]
    other["beta"][:, 150:] = 0.9
    o2, _ = gpu_forward(other, wl.L, wl.chunk)
    assert torch.equal(o1[:, :150], o2[:, :150])
    assert not torch.equal(o1[:, 150:], o2[:, 150:])


def test_boundary_errors_on_device():
    wl = I.Workload("case", "bf16", 1, 64, 1, 64, 64, 2, 4, 64, seed=6)
    d = prism.inputs_to_device(I.generate(wl))
    # misaligned output pointer
    buf = torch.empty(64 * 64 + 8, dtype=torch.float32, device="cuda")
    bad_out = buf[1:1 + 64 * 64].view(1, 64, 1, 64)
    with pytest.raises(prism.PrismError) as e:
        prism.forward_inputs(d, 2, 64, out=bad_out)
    assert e.value.code == 3
    # workspace too small
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(prism.PrismError) as e:
        prism.forward_inputs(d, 2, 64, workspace=small)
    assert e.value.code == 4
    # unsupported chunk
    with pytest.raises(prism.PrismError) as e:
        prism.forward_inputs(d, 2, 48)
    assert e.value.code == 2


@pytest.mark.parametrize("dtype,D,C", [("bf16", 128, 64), ("bf16", 32, 16), ("f32", 16, 16)])
def test_device_status_after_forward(dtype, D, C):
    """Every bounded wait completed: the workspace's status word, filled with a nonzero
    pattern beforehand, reads 0 through prism_device_status after a forward call."""
    wl = I.Workload("case", dtype, 2, 100, 2, D, D, 2, 4, C, seed=8)
    d = prism.inputs_to_device(I.generate(wl))
    dims = prism.make_dims(2, 100, 2, D, D, 4, 2, C, d["q"].dtype)
    ws = prism.alloc_workspace(dims, "cuda")
    ws.fill_(0xA5)
    prism.forward_inputs(d, wl.L, wl.chunk, workspace=ws)
    assert prism.device_status(dims, ws) == 0
