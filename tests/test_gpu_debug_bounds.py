"""The bounds-checked debug build of the library (compiled with -DPRISM_DEBUG_BOUNDS: every
plain load and store of the tensor-core forward kernels and of the decode kernel, their
shared-memory tile writes and the source ranges of their bulk copies are checked against
the extent of the array they address; a violation is skipped and recorded in a word that
prism_debug_bounds reads).  compute-sanitizer is not available here, so this is the direct
evidence that the kernels stay inside their arrays: forward cases over every head dim,
chunk size, ragged and resumed sequences and the sequence split, and decode steps, each
matching the oracle, with the word still 0 at the end."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_debug_build_stays_in_bounds():
    if not torch.cuda.is_available():
        pytest.fail("CUDA GPU required for -m gpu tests")
    from linear_recurrent_sequence_causal_gb300 import build
    lib = build.build_debug()
    env = dict(os.environ, PRISM_LIBRARY=lib)
    r = subprocess.run([sys.executable, "-m", "tests.debug_bounds_cases"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "bounds word after" in r.stdout and r.stdout.strip().endswith(": 0"), r.stdout
