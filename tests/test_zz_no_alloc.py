"""prism_forward_static: the forward pass for callers that cannot allocate
device memory on their hot path (pre-planned arenas, allocation-free plugin
contexts).  It runs out of the library's fixed device scratch array instead of
a caller workspace.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

from linear_recurrent_sequence_causal_gb300 import inputs as I
from linear_recurrent_sequence_causal_gb300 import prism
from tests.parity import BF16_OUT_TOL, BF16_STATE_TOL, F32_TOL

# Calls in a row on one shared array: bf16 with refinement steps first, so that
# the layouts after it (fp32, whose regions differ, and bf16 at L = 0, which has no
# weight blocks or N region and leaves the weights flag unwritten) start from the
# leftovers of a real call.
CASES = [("bf16", 2, 300, 2, 64, 3, 64), ("bf16", 3, 129, 2, 128, 2, 32),
         ("f32", 1, 64, 1, 16, 2, 16), ("bf16", 2, 200, 2, 32, 0, 32),
         ("bf16", 2, 300, 2, 64, 3, 64)]


@pytest.mark.gpu
def test_static_scratch_matches_workspace_path_in_a_row():
    """Each call must agree with the workspace entry point (same kernels, so the
    results should coincide), and no call may see an earlier call's leftovers in
    the shared array."""
    prism.load()
    for seed, (dt, B, T, H, D, L, C) in enumerate(CASES):
        wl = I.Workload("static", dt, B, T, H, D, D, L, 4, C, seed=500 + seed)
        inp = I.generate(wl)
        inp["seq_lens"] = torch.tensor([T] + [T // 2] * (B - 1), dtype=torch.int32)
        d = prism.inputs_to_device(inp)
        dims = prism.make_dims(B, T, H, D, D, wl.w, L, C, wl.torch_dtype)
        assert prism.workspace_bytes(dims) <= prism.STATIC_SCRATCH_BYTES
        o_ref, s_ref = prism.forward_inputs(d, L, C)
        o_st, s_st = prism.prism_forward_static(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"],
                                                d["conv_w"], d["Wk"], d["Wp"], d["wbeta"], L, C,
                                                seq_lens=d["seq_lens"])
        torch.cuda.synchronize()
        o_ref, o_st = o_ref.double().cpu().numpy(), o_st.double().cpu().numpy()
        s_ref, s_st = s_ref.double().cpu().numpy(), s_st.double().cpu().numpy()
        what = f"case {seed} ({dt}, L={L})"
        if dt == "f32":
            assert np.max(np.abs(o_st - o_ref)) <= F32_TOL * np.max(np.abs(o_ref)), what
            assert np.max(np.abs(s_st - s_ref)) <= F32_TOL * np.max(np.abs(s_ref)), what
        else:
            rms = np.sqrt(np.mean(o_ref ** 2))
            assert np.max(np.abs(o_st - o_ref)) <= BF16_OUT_TOL * rms, what
            assert np.linalg.norm(s_st - s_ref) <= BF16_STATE_TOL * np.linalg.norm(s_ref), what
        for b, n in enumerate(inp["seq_lens"].tolist()):
            assert np.all(o_st[b, n:] == 0.0), what


def test_static_scratch_rejects_oversized_dims():
    """Dims that need more than the static array are refused before any launch."""
    lib = prism.load()
    d = prism.make_dims(8, 4096, 16, 128, 128, 4, 2, 64, prism.PRISM_BF16)
    assert prism.workspace_bytes(d) > prism.STATIC_SCRATCH_BYTES
    rc = lib.prism_forward_static(ctypes.byref(d), *[0x1000] * 12, None)
    assert rc == 7 and b"STATIC_SCRATCH" in lib.prism_strerror(rc)


@pytest.mark.gpu
def test_static_status_word():
    """prism_static_status reads the bounded-wait status word a static call left in the
    library's scratch: 0 after a normal call; nonzero after a call whose diagnostic flag
    makes a wait of each scan CTA run out (nothing in flight; the outputs are still those
    of the normal call); 0 again after the next normal call."""
    prism.load()
    B, T, H, D, L, C = 2, 300, 2, 128, 2, 64
    wl = I.Workload("static", "bf16", B, T, H, D, D, L, 4, C, seed=611)
    d = prism.inputs_to_device(I.generate(wl))
    dims = prism.make_dims(B, T, H, D, D, 4, L, C, torch.bfloat16)
    chk = prism.PRISM_FLAG_CHECK_WAIT_TIMEOUT
    dims_chk = prism.make_dims(B, T, H, D, D, 4, L, C, torch.bfloat16, flags=chk)
    args = (d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["conv_w"], d["Wk"], d["Wp"],
            d["wbeta"], L, C)
    o0, s0 = prism.prism_forward_static(*args)
    assert prism.static_status(dims) == 0
    o1, s1 = prism.prism_forward_static(*args, flags=chk)
    assert prism.static_status(dims_chk) != 0
    assert torch.equal(o0, o1) and torch.equal(s0, s1)
    o2, _ = prism.prism_forward_static(*args)
    assert prism.static_status(dims) == 0
    assert torch.equal(o0, o2)
