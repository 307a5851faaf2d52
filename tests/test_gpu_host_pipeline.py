"""GPU: the host-to-host forward (prism_forward_host through prism.HostPipeline: copies
overlapped with the kernels) gives the results of one prism_forward call on the same
inputs, and the oracle's."""
import pytest
import torch

import oracle
from linear_recurrent_sequence_causal_gb300 import inputs as I
from linear_recurrent_sequence_causal_gb300 import prism
from tests.parity import check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("CUDA GPU required for -m gpu tests")
    prism.load()


@pytest.mark.parametrize("B,T,H,D,L,chunk,ragged,pieces", [
    (6, 300, 2, 64, 2, 64, True, 4),      # groups of sequences
    (1, 1000, 3, 128, 4, 64, False, 5),   # token segments resumed from the previous state
    (1, 77, 2, 32, 1, 32, False, 3),
    (3, 90, 2, 32, 2, 32, True, 1),       # one piece: a single stream
    (6, 77, 1, 32, 2, 16, True, 3),       # T*H odd: groups rounded to 4 sequences
])
def test_host_pipeline_equals_one_call(B, T, H, D, L, chunk, ragged, pieces):
    wl = I.Workload("hp", "bf16", B, T, H, D, D, L, 4, chunk, seed=11 + B + D, ragged=ragged)
    host = I.generate(wl)
    pinned = {k: (v.pin_memory() if v is not None else None) for k, v in host.items()}
    shapes = {k: tuple(v.shape) for k, v in host.items() if v is not None}
    pipe = prism.HostPipeline(shapes, torch.bfloat16, L, chunk, pieces=pieces, min_piece_bytes=0)
    assert (len(pipe.pieces) > 1) == (pieces > 1)
    h_out = torch.empty((B, T, H, D), dtype=torch.float32).pin_memory()
    h_fs = torch.empty((B, H, D, D), dtype=torch.float32).pin_memory()
    pipe.run(pinned, h_out, h_fs)
    torch.cuda.synchronize()
    d = prism.inputs_to_device(host)
    ref_out, ref_fs = prism.forward_inputs(d, L, chunk)
    torch.cuda.synchronize()
    assert torch.equal(h_out, ref_out.cpu()), "outputs differ from one prism_forward call"
    assert torch.equal(h_fs, ref_fs.cpu()), "final state differs from one prism_forward call"
    if T <= 300 or B == 1:
        ro, rs, _ = oracle.forward(host)
        check(h_out, h_fs, ro, rs, "bf16", seq_lens=host.get("seq_lens"), what="host pipeline")


@pytest.mark.parametrize("length", [0, 1, 130, 500])
def test_host_pipeline_one_sequence_with_a_length(length):
    """B = 1 with seq_lens: the segments stop at the length (the one holding it runs up to
    it, later ones only zero their rows); pageable host buffers.  Equal to one call within
    fp32 rounding, the oracle's result within the bf16 tolerance over the valid tokens,
    zeros past the length."""
    B, T, H, D, L, chunk = 1, 500, 2, 64, 2, 64
    wl = I.Workload("hp1", "bf16", B, T, H, D, D, L, 4, chunk, seed=29)
    host = I.generate(wl)
    host["seq_lens"] = torch.tensor([length], dtype=torch.int32)
    shapes = {k: tuple(v.shape) for k, v in host.items() if v is not None}
    pipe = prism.HostPipeline(shapes, torch.bfloat16, L, chunk, pieces=4, min_piece_bytes=0)
    assert len(pipe.pieces) == 4
    h_out = torch.full((B, T, H, D), float("nan"), dtype=torch.float32)
    h_fs = torch.full((B, H, D, D), float("nan"), dtype=torch.float32)
    pipe.run(host, h_out, h_fs)
    torch.cuda.synchronize()
    assert torch.all(h_out[:, length:] == 0)
    d = prism.inputs_to_device(host)
    ref_out, ref_fs = prism.forward_inputs(d, L, chunk)
    torch.cuda.synchronize()
    ref_out, ref_fs = ref_out.cpu(), ref_fs.cpu()
    scale = max(ref_out.abs().max().item(), 1e-30)
    assert torch.allclose(h_out, ref_out, rtol=0, atol=1e-5 * scale)
    assert torch.allclose(h_fs, ref_fs, rtol=0, atol=1e-5 * max(ref_fs.abs().max().item(), 1e-30))
    if length == 0:
        assert torch.all(h_fs == 0)
    else:
        # against the oracle over the valid tokens: RMS(o) of the padded tensor would count
        # the zero rows (one valid token in 500 shrinks it 22-fold)
        ro, rs, _ = oracle.forward(host)
        check(h_out[:, :length], h_fs, ro[:, :length], rs, "bf16", what="host pipeline, one sequence")
