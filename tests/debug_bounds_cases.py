"""Cases run by tests/test_gpu_debug_bounds.py in a child process whose PRISM_LIBRARY is the
bounds-checked debug build of the library: each case is checked against the fp64 oracle,
and after all of them the debug word must read 0 (no access outside its array)."""
import sys

import numpy as np
import torch

import oracle
from linear_recurrent_sequence_causal_gb300 import inputs as I
from linear_recurrent_sequence_causal_gb300 import prism
from tests.parity import check

# dtype, B, T, H, D, L, w, chunk, ragged, resumed
FORWARD = [
    ("bf16", 2, 300, 2, 128, 2, 4, 64, True, False),
    ("bf16", 1, 95, 2, 128, 5, 8, 32, True, True),
    ("bf16", 3, 77, 2, 64, 4, 4, 64, True, False),
    ("bf16", 2, 150, 1, 64, 3, 3, 32, False, True),
    ("bf16", 4, 200, 2, 32, 3, 4, 32, True, False),
    ("bf16", 2, 64, 1, 16, 2, 4, 16, False, False),
    ("bf16", 2, 40, 2, 16, 0, 2, 64, True, False),
    ("bf16", 1, 4096, 2, 128, 2, 4, 64, False, False),     # sequence split (P > 1)
]
# dtype, D, L, B, H
DECODE = [("bf16", 128, 2, 3, 2), ("bf16", 64, 8, 48, 8), ("f32", 32, 3, 2, 3), ("bf16", 16, 0, 2, 3)]


def forward_case(dtype, B, T, H, D, L, w, chunk, ragged, resumed):
    wl = I.Workload("dbg", dtype, B, T, H, D, D, L, w, chunk, seed=300 + T + D)
    inp = I.generate(wl)
    if ragged:
        g = torch.Generator().manual_seed(T)
        lens = torch.randint(0, T + 1, (B,), generator=g, dtype=torch.int32)
        lens[0] = T
        inp["seq_lens"] = lens
    s0 = vh = None
    if resumed:
        g = torch.Generator().manual_seed(11)
        s0 = 0.1 * torch.randn((B, H, D, D), generator=g, dtype=torch.float32)
        vh = torch.randn((B, H, w, D), generator=g).to(wl.torch_dtype)
    d = prism.inputs_to_device(inp)
    kw = dict(seq_lens=d.get("seq_lens"))
    if resumed:
        kw.update(initial_state=s0.cuda(), v_hist=vh.cuda())
    out, fs = prism.prism_forward_from(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["conv_w"],
                                       d["Wk"], d["Wp"], d["wbeta"], L, chunk, **kw)
    torch.cuda.synchronize()
    ro, rs, _ = oracle.forward(inp, L=L, initial_state=s0, v_hist=vh)
    if ragged:
        for b, n in enumerate(inp["seq_lens"].tolist()):
            if n == 0:
                rs[b] = 0.0 if s0 is None else s0[b].double().numpy()
    check(out, fs, ro, rs, dtype, seq_lens=inp.get("seq_lens"), what=f"debug build forward D{D} C{chunk} L{L}")


def decode_case(dtype, D, L, B, H):
    T0, n, chunk = 21, 3, 16
    wl = I.Workload("dbg", dtype, B, T0 + n, H, D, D, L, 4, chunk, seed=500 + D + L + B)
    inp = I.generate(wl)
    ro, rs, _ = oracle.forward(inp)
    d = prism.inputs_to_device(inp)
    keys = ("q", "k", "v", "log_alpha", "beta")
    pre = dict(d)
    for k in keys:
        pre[k] = d[k][:, :T0].contiguous()
    pre["seq_lens"] = None
    out0, state = prism.forward_inputs(pre, L, chunk)
    hist = prism.v_history(d["v"], wl.w, T0)
    outs = [out0]
    for t in range(T0, T0 + n):
        tok = {k: d[k][:, t].clone() for k in keys}
        o = prism.prism_decode_step(tok["q"], tok["k"], tok["v"], tok["log_alpha"], tok["beta"], d["conv_w"],
                                    d["Wk"], d["Wp"], d["wbeta"], L, state, hist)
        outs.append(o[:, None])
    torch.cuda.synchronize()
    check(torch.cat(outs, dim=1), state, ro, rs, dtype, what=f"debug build decode D{D} L{L}")


def main():
    prism.load()
    word = prism.debug_bounds(clear=True)
    if word is None:
        print("the loaded library is not the debug build")
        return 2
    for c in FORWARD:
        forward_case(*c)
    for c in DECODE:
        decode_case(*c)
    word = prism.debug_bounds(clear=True)
    print(f"bounds word after {len(FORWARD)} forward and {len(DECODE)} decode cases: {word}")
    return 0 if word == 0 else 1


if __name__ == "__main__":
    sys.exit(main())
