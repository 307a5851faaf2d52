"""The oracle against its stored regression fixtures (tests/golden/*.json, CPU only).

The fixtures were written by ``tests/golden/make_golden.py`` from the oracle itself (the
pages print no worked example), so they pin nothing about the method: they make any
change to the oracle's arithmetic visible.  Such a change has to name the passage of the
pages that justifies it, and the fixtures are then re-written by that script.
"""
import glob
import json
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import grad

GOLDEN = sorted(glob.glob(os.path.join(os.path.dirname(__file__), "golden", "*.json")))
# Same source, other compiler or libm (erf, exp): a few ulps per operation at most.
FWD_TOL = 1e-12
GRAD_TOL = 1e-10


def _err(a, b):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape
    return np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300)


def _load(path):
    rec = json.load(open(path))
    inp = {k: (torch.tensor(v, dtype=torch.int32) if k == "seq_lens"
               else torch.tensor(v, dtype=torch.float64))
           for k, v in rec["inputs"].items()}
    inp.setdefault("seq_lens", None)
    return rec, inp


def test_fixtures_present_and_cited():
    names = {os.path.basename(p) for p in GOLDEN}
    assert {"prism_tiny.json", "prism_tiny_no_gelu.json", "prism_tiny_resumed.json"} <= names
    for p in GOLDEN:
        assert "Technical Summary: PRISM" in json.load(open(p))["source"]


@pytest.mark.parametrize("path", GOLDEN, ids=os.path.basename)
def test_forward_matches_fixture(path):
    rec, inp = _load(path)
    extra = {k: np.asarray(v) for k, v in rec["resume"].items()}
    out, fs, _ = oracle.forward(inp, identity_act=rec["identity_act"], **extra)
    assert _err(out, rec["out"]) <= FWD_TOL
    assert _err(fs, rec["final_state"]) <= FWD_TOL


@pytest.mark.parametrize("path", [p for p in GOLDEN if "grads" in json.load(open(p))],
                         ids=os.path.basename)
def test_gradients_match_fixture(path):
    rec, inp = _load(path)
    g = grad.backward(inp, np.asarray(rec["d_out"]), np.asarray(rec["d_final_state"]),
                      identity_act=rec["identity_act"])
    for k in grad.GRAD_KEYS:
        assert _err(g[k], rec["grads"][k]) <= GRAD_TOL, k
