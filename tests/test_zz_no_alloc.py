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
from tests.parity import BF16_OUT_TOL, BF16_STATE_TOL


@pytest.mark.gpu
def test_static_scratch_matches_workspace_path_twice():
    """Two calls in a row on different inputs: each must agree with the
    workspace entry point (same kernels, so the results should coincide), and
    the second must not see the first call's leftovers in the shared array."""
    prism.load()
    for seed, (B, T, H, D, L, C) in enumerate([(2, 300, 2, 64, 3, 64), (3, 129, 2, 128, 2, 32)]):
        wl = I.Workload("static", "bf16", B, T, H, D, D, L, 4, C, seed=500 + seed)
        inp = I.generate(wl)
        inp["seq_lens"] = torch.tensor([T] + [T // 2] * (B - 1), dtype=torch.int32)
        d = prism.inputs_to_device(inp)
        dims = prism.make_dims(B, T, H, D, D, wl.w, L, C, torch.bfloat16)
        assert prism.workspace_bytes(dims) <= prism.STATIC_SCRATCH_BYTES
        o_ref, s_ref = prism.forward_inputs(d, L, C)
        o_st, s_st = prism.prism_forward_static(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"],
                                                d["conv_w"], d["Wk"], d["Wp"], d["wbeta"], L, C,
                                                seq_lens=d["seq_lens"])
        torch.cuda.synchronize()
        o_ref, o_st = o_ref.double().cpu().numpy(), o_st.double().cpu().numpy()
        s_ref, s_st = s_ref.double().cpu().numpy(), s_st.double().cpu().numpy()
        rms = np.sqrt(np.mean(o_ref ** 2))
        assert np.max(np.abs(o_st - o_ref)) <= BF16_OUT_TOL * rms
        assert np.linalg.norm(s_st - s_ref) <= BF16_STATE_TOL * np.linalg.norm(s_ref)


def test_static_scratch_rejects_oversized_dims():
    """Dims that need more than the static array are refused before any launch."""
    lib = prism.load()
    d = prism.make_dims(8, 4096, 16, 128, 128, 4, 2, 64, prism.PRISM_BF16)
    assert prism.workspace_bytes(d) > prism.STATIC_SCRATCH_BYTES
    rc = lib.prism_forward_static(ctypes.byref(d), *[0x1000] * 12, None)
    assert rc == 7 and b"STATIC_SCRATCH" in lib.prism_strerror(rc)
