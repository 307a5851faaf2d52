"""Writes the regression fixtures in this folder from the oracle alone.

The pages print no worked example, so nothing here is the authors' number: each
fixture holds small seeded inputs and what ``oracle.forward`` (the fp64 C oracle) and
``oracle.grad.backward`` (its differentiable restatement) return for them, printed in the
shortest decimal form that reads back to the same double.  ``tests/test_golden.py`` re-runs the oracle on the stored inputs
and compares; a later change to the oracle's arithmetic shows up there and has to be
justified by the passage of the pages it follows.

Run from the repository root:  python -m tests.golden.make_golden
"""
from __future__ import annotations

import json
import os

import numpy as np
import torch

import oracle
from oracle import grad
from linear_recurrent_sequence_causal_gb300.inputs import random_small

HERE = os.path.dirname(os.path.abspath(__file__))

# name, (B, T, H, d_k, d_v, L, w), seed, ragged lengths, identity activation, resumed
CASES = [
    ("prism_tiny", (2, 7, 2, 3, 4, 2, 3), 101, [7, 4], False, False),
    ("prism_tiny_no_gelu", (1, 6, 1, 4, 4, 3, 2), 102, None, True, False),
    ("prism_tiny_resumed", (1, 5, 2, 3, 3, 1, 2), 103, None, False, True),
]


def _listed(a):
    return np.asarray(a, dtype=np.float64).tolist()


def make(name, shape, seed, lens, identity_act, resumed):
    B, T, H, dk, dv, L, w = shape
    inp = random_small(B, T, H, dk, dv, L, w, seed=seed)
    if lens is not None:
        inp["seq_lens"] = torch.tensor(lens, dtype=torch.int32)
    extra = {}
    if resumed:
        g = np.random.default_rng(seed)
        extra["initial_state"] = g.standard_normal((B, H, dv, dk)) * 0.5
        extra["v_hist"] = g.standard_normal((B, H, w, dv))
    out, fs, _ = oracle.forward(inp, identity_act=identity_act, **extra)
    rec = {
        "source": ("written by tests/golden/make_golden.py from the fp64 oracle (oracle.forward"
                   + ("" if resumed else ", oracle.grad.backward") + "); the method is the PRISM "
                   "mixer of 'Technical Summary: PRISM (Parallel Residual Iterative Sequence "
                   "Model)', sections 2.1 and 2.2, which prints no worked example"),
        "shape": dict(zip(("B", "T", "H", "dk", "dv", "L", "w"), shape)),
        "identity_act": identity_act,
        "inputs": {k: (v.tolist() if k == "seq_lens" else _listed(v.numpy()))
                   for k, v in inp.items() if v is not None},
        "resume": {k: _listed(v) for k, v in extra.items()},
        "out": _listed(out),
        "final_state": _listed(fs),
    }
    if not resumed:
        g = np.random.default_rng(seed + 1)
        d_out = g.standard_normal((B, T, H, dv))
        d_fs = g.standard_normal((B, H, dv, dk))
        gr = grad.backward(inp, d_out, d_fs, identity_act=identity_act)
        rec["d_out"] = _listed(d_out)
        rec["d_final_state"] = _listed(d_fs)
        rec["grads"] = {k: _listed(v) for k, v in gr.items()}
    return rec


def main():
    for name, shape, seed, lens, ida, resumed in CASES:
        rec = make(name, shape, seed, lens, ida, resumed)
        path = os.path.join(HERE, name + ".json")
        with open(path, "w") as f:
            json.dump(rec, f, separators=(",", ":"), default=float)
            f.write("\n")
        print(path, os.path.getsize(path), "bytes")


if __name__ == "__main__":
    main()
