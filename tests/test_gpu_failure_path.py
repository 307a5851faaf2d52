"""The failure path of the bounded waits, exercised without faulting or hanging the GPU.

Every wait of the tensor-core kernels on an mbarrier is bounded; one that gives up sets
the device status word instead of hanging, and prism_device_status reads it back.
PRISM_FLAG_CHECK_WAIT_TIMEOUT makes each scan CTA first wait, with a short poll limit, on
an mbarrier that nothing completes, at a point where none of its copies or MMAs is in
flight: the wait runs out exactly as a real one would, the call returns, the status reads
nonzero, and the outputs are those of the same call without the flag."""
import pytest
import torch

from linear_recurrent_sequence_causal_gb300 import inputs as I
from linear_recurrent_sequence_causal_gb300 import prism

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("CUDA GPU required for -m gpu tests")
    prism.load()


@pytest.mark.parametrize("B,T,H,C", [(2, 300, 2, 64), (1, 4096, 1, 64), (2, 100, 1, 32)])
def test_wait_that_runs_out_sets_the_status_word(B, T, H, C):
    wl = I.Workload("case", "bf16", B, T, H, 128, 128, 2, 4, C, seed=17 + T)
    d = prism.inputs_to_device(I.generate(wl))
    check = prism.PRISM_FLAG_CHECK_WAIT_TIMEOUT
    dims = prism.make_dims(B, T, H, 128, 128, 4, 2, C, torch.bfloat16)
    dims_chk = prism.make_dims(B, T, H, 128, 128, 4, 2, C, torch.bfloat16, flags=check)
    assert prism.workspace_bytes(dims_chk) == prism.workspace_bytes(dims)
    ws = prism.alloc_workspace(dims, "cuda")
    out0, fs0 = prism.forward_inputs(d, wl.L, C, workspace=ws)
    assert prism.device_status(dims, ws) == 0
    out1, fs1 = prism.forward_inputs(d, wl.L, C, workspace=ws, flags=check)
    assert prism.device_status(dims_chk, ws) != 0          # the wait gave up, and the call returned
    assert torch.equal(out0, out1) and torch.equal(fs0, fs1)
    # the word is cleared at the start of every call: the next normal call reads 0 again
    out2, _ = prism.forward_inputs(d, wl.L, C, workspace=ws)
    assert prism.device_status(dims, ws) == 0
    assert torch.equal(out0, out2)
    if T == 4096:                                           # the split scan runs the check in each pass
        assert prism.scan_segments(dims) > 1
