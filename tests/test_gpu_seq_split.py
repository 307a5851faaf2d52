"""GPU parity of the sequence-split scan: long sequences with few (b, h) pairs are cut
into segments whose affine state maps (S_end = S_start M + c, from the
state-independent update of "Technical Summary: PRISM", §2.2, last paragraph) are
composed across CTAs, then every segment is rescanned from its true entering state.
Checked against the fp64 oracle and against the unsplit scan (PRISM_FLAG_NO_SEQ_SPLIT)."""
import numpy as np
import pytest
import torch

import oracle
from linear_recurrent_sequence_causal_gb300 import inputs as I
from linear_recurrent_sequence_causal_gb300 import prism
from tests.parity import BF16_OUT_TOL, BF16_STATE_TOL, check, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("CUDA GPU required for -m gpu tests")
    prism.load()


def _segments(wl, L):
    return prism.scan_segments(prism.make_dims(wl.B, wl.T, wl.H, wl.dk, wl.dv, wl.w, L, wl.chunk,
                                               wl.torch_dtype))


def _close(out_a, fs_a, out_b, fs_b, what):
    """Split against unsplit: the same arithmetic composed in another order, so equal
    within the bf16-path tolerance (relative to the unsplit result)."""
    oa, ob = to64(out_a), to64(out_b)
    rms = np.sqrt(np.mean(ob ** 2))
    assert np.max(np.abs(oa - ob)) <= BF16_OUT_TOL * rms, what
    sa, sb = to64(fs_a), to64(fs_b)
    assert np.linalg.norm(sa - sb) <= BF16_STATE_TOL * np.linalg.norm(sb), what


def test_long_sequence_few_heads():
    """B = 1, H = 4, T = 65536, d = 128, L = 4, chunk 64 (the long-context shape with
    an eighth of its heads): the scan is cut into 5 segments.  Two heads are checked
    by the oracle over the whole length, all four against the unsplit scan."""
    wl = I.Workload("split_long", "bf16", 1, 65536, 4, 128, 128, 4, 4, 64, seed=41)
    assert _segments(wl, wl.L) == 5
    inp = I.generate(wl)
    d = prism.inputs_to_device(inp)
    out, fs = prism.forward_inputs(d, wl.L, wl.chunk)
    out1, fs1 = prism.forward_inputs(d, wl.L, wl.chunk, flags=prism.PRISM_FLAG_NO_SEQ_SPLIT)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all() and torch.isfinite(fs).all()
    _close(out, fs, out1, fs1, "split vs one chain")
    heads = [(0, 1), (0, 2)]
    ro, rs, _ = oracle.forward(inp, bh_items=heads)
    check(out, fs, ro, rs, "bf16", bh=heads, what="split long sequence, full length")


# B, T, H, chunk, L, lens (None: all T), resumed
CASES = [
    (1, 4096, 2, 64, 2, None, False),
    (1, 5000, 1, 32, 3, None, False),             # T mod C != 0, last segment short
    (3, 3000, 1, 32, 1, [3000, 700, 0], False),   # ragged: a length inside the second segment, an empty one
    (2, 6000, 1, 64, 0, [6000, 4097], False),     # L = 0 (no N maps): gated delta rule
    (1, 4096, 1, 64, 2, None, True),              # entering state and history
]


@pytest.mark.parametrize("B,T,H,C,L,lens,resumed", CASES)
def test_split_shapes(B, T, H, C, L, lens, resumed):
    wl = I.Workload("split", "bf16", B, T, H, 128, 128, L, 4, C, seed=60 + T + B)
    P = _segments(wl, L)
    assert P >= 3, P
    inp = I.generate(wl)
    if lens is not None:
        inp["seq_lens"] = torch.tensor(lens, dtype=torch.int32)
    s0 = vh = None
    if resumed:
        g = torch.Generator().manual_seed(7)
        s0 = 0.1 * torch.randn((B, H, 128, 128), generator=g, dtype=torch.float32)
        vh = torch.randn((B, H, wl.w, 128), generator=g).to(torch.bfloat16)
    d = prism.inputs_to_device(inp)
    kw = dict(seq_lens=d.get("seq_lens"))
    if resumed:
        kw.update(initial_state=s0.cuda(), v_hist=vh.cuda())
    args = (d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["conv_w"], d["Wk"], d["Wp"],
            d["wbeta"], L, C)
    out, fs = prism.prism_forward_from(*args, **kw)
    out1, fs1 = prism.prism_forward_from(*args, flags=prism.PRISM_FLAG_NO_SEQ_SPLIT, **kw)
    torch.cuda.synchronize()
    what = f"B{B} T{T} H{H} C{C} L{L} P{P}"
    _close(out, fs, out1, fs1, what + " split vs one chain")
    ro, rs, _ = oracle.forward(inp, L=L, initial_state=s0, v_hist=vh)
    if lens is not None:
        for b, n in enumerate(lens):
            if n == 0:
                rs[b] = 0.0 if s0 is None else s0[b].double().numpy()
    check(out, fs, ro, rs, "bf16", seq_lens=inp.get("seq_lens"), what=what)


def test_split_is_deterministic():
    wl = I.Workload("split", "bf16", 1, 4096, 2, 128, 128, 2, 4, 64, seed=9)
    d = prism.inputs_to_device(I.generate(wl))
    a = prism.forward_inputs(d, wl.L, wl.chunk)
    b = prism.forward_inputs(d, wl.L, wl.chunk)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
