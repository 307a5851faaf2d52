"""The bf16 prepare kernel's activation (GELU with erf from Hastings' rational
approximation, Abramowitz and Stegun 7.1.26) against the exact GELU of "Technical Summary:
PRISM", §2.2 in fp64 and against CUDA's own erf-based GELU (torch's exact GELU on the GPU)."""
import math

import numpy as np
import pytest
import torch

from linear_recurrent_sequence_causal_gb300 import prism

scipy_special = pytest.importorskip("scipy.special")


@pytest.mark.gpu
def test_prepare_activation_within_the_approximation_bound():
    prism.load()
    xs = torch.cat([torch.linspace(-12.0, 12.0, 1_000_001),
                    torch.tensor([0.0, -0.0, 1e-30, -1e-30, 1e-7, -1e-7, 30.0, -30.0, 1e4, -1e4])])
    x = xs.float().cuda()
    y = prism.debug_activation(x)
    torch.cuda.synchronize()
    xd = x.double().cpu().numpy()
    yd = y.double().cpu().numpy()
    exact = xd * 0.5 * scipy_special.erfc(-xd / math.sqrt(2.0))
    scale = np.maximum(np.abs(xd), 1.0)
    # erf within 1.5e-7 (the formula's bound), times |x|/2, plus fp32 rounding of the
    # reciprocal, exponential and products
    assert np.max(np.abs(yd - exact) / scale) <= 5e-7
    cuda_gelu = torch.nn.functional.gelu(x).double().cpu().numpy()
    assert np.max(np.abs(yd - cuda_gelu) / scale) <= 1e-6
    # odd part and limits: GELU(x) - GELU(-x) = x; large |x| gives x and 0
    n = 1_000_001
    assert np.max(np.abs((yd[:n] - yd[:n][::-1]) - xd[:n]) / scale[:n]) <= 1e-6
    assert yd[n + 6] == 30.0 and yd[n + 8] == 1e4
    assert abs(yd[n + 7]) < 1e-30 and yd[n + 9] == 0.0


@pytest.mark.gpu
def test_prepare_activation_nan_and_empty():
    prism.load()
    x = torch.tensor([float("nan"), 1.0], device="cuda")
    y = prism.debug_activation(x)
    assert torch.isnan(y[0]).item() and abs(y[1].item() - 0.8413447460685429) < 1e-6
    assert prism.debug_activation(torch.empty(0, device="cuda")).numel() == 0
