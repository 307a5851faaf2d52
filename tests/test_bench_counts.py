"""The algorithmic bytes and flops that bench.py divides by kernel time (the roofline's
numerators) against independent counts (CPU only).

* Flops: prepare + scan together equal the chunk-form count per token-head,
  F_scan = C d (10 + 8L) + d^2 (6 + 2L) + C^2/3, plus the anchor and refinement count
  F_anchor = 2 w d + L (4 d^2 + 2 d), over all token-heads.
* Bytes: the chunk maps the prepare kernel writes and the scan kernel reads are the
  workspace regions the library lays out for them (prism_workspace_layout), so the scan's
  byte count minus its output and final state equals the sizes of those regions.
"""
import pytest

import bench
from linear_recurrent_sequence_causal_gb300 import build, inputs as I, prism


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    prism.load()


def _f_scan(C, d, L):
    return C * d * (10 + 8 * L) + d * d * (6 + 2 * L) + C * C / 3.0


def _f_anchor(w, d, L):
    return 2 * w * d + L * (4 * d * d + 2 * d)


@pytest.mark.parametrize("name", sorted(I.WORKLOADS))
@pytest.mark.parametrize("L", [0, 1, 4])
def test_flops_are_the_chunk_form_count(name, L):
    wl = I.WORKLOADS[name]
    alg = bench.algorithmic(wl, L)
    th = wl.B * wl.T * wl.H
    total = alg["prepare"][1] + alg["scan"][1]
    expect = th * (_f_scan(wl.chunk, wl.dk, L) + _f_anchor(wl.w, wl.dk, L))
    assert total == pytest.approx(expect, rel=1e-12)


def test_longctx_figures():
    """The long-context figures quoted beside the measurements: 8.09 GB and 1.55 TFLOP for
    the prepare kernel, 7.52 GB for the scan."""
    alg = bench.algorithmic(I.WORKLOADS["longctx_bf16"], 4)
    assert alg["prepare"][0] == pytest.approx(8.0869e9, rel=1e-4)
    assert alg["prepare"][1] == pytest.approx(1.5533e12, rel=1e-4)
    assert alg["scan"][0] == pytest.approx(7.5184e9, rel=1e-4)


@pytest.mark.parametrize("name", ["lsweep_bf16", "lm_bf16", "longctx_bf16"])
@pytest.mark.parametrize("L", [0, 2])
def test_scan_bytes_are_the_workspace_maps(name, L):
    wl = I.WORKLOADS[name]
    assert wl.T % wl.chunk == 0
    d = prism.make_dims(wl.B, wl.T, wl.H, wl.dk, wl.dv, wl.w, L, wl.chunk, prism.PRISM_BF16)
    lay = prism.workspace_layout(d)
    total = prism.workspace_bytes(d)
    order = sorted((off, n) for n, off in lay.items() if off is not None)
    size = {n: (order[i + 1][0] if i + 1 < len(order) else total) - off
            for i, (off, n) in enumerate(order)}
    maps = sum(size[n] for n in ("WQ", "QK", "U", "Oi", "N", "gC") if n in size)
    th = wl.B * wl.T * wl.H
    scan_bytes = bench.algorithmic(wl, L)["scan"][0]
    written = th * 4 * wl.dv + wl.B * wl.H * wl.dv * wl.dk * 4      # out and final state
    # regions are padded to 256 bytes each
    assert abs((scan_bytes - written) - maps) <= 6 * 256


@pytest.mark.parametrize("name", sorted(I.WORKLOADS))
@pytest.mark.parametrize("L", [0, 2, 4])
def test_method_counts(name, L):
    """The roofline numerators of the method's own work: the two kernels' flops add up to
    F_scan + F_anchor, the same as the whole path's; the path moves (2 d_k + 2 d_v) e + 8
    bytes per token-head (1032 at d = 128 in bf16) plus the weights and the final state."""
    wl = I.WORKLOADS[name]
    m = bench.method_counts(wl, L)
    th = wl.B * wl.T * wl.H
    d, e = wl.dk, (4 if wl.dtype == "f32" else 2)
    expect = th * (_f_scan(wl.chunk, d, L) + _f_anchor(wl.w, d, L))
    assert m["prepare"][1] + m["scan"][1] == pytest.approx(expect, rel=1e-12)
    assert m["path"][1] == pytest.approx(expect, rel=1e-12)
    assert m["scan"][1] == pytest.approx(th * 6 * d * d, rel=1e-12)
    weights = wl.H * (L * (2 * d * d + d) + wl.w * d) * 4
    state = wl.B * wl.H * d * d * 4
    per = (m["path"][0] - weights - state) / th
    assert per == pytest.approx(4 * d * e + 8, rel=1e-12)
    if d == 128 and e == 2:
        assert per == 1032


def test_longctx_method_figures():
    """Long context: 740,693 flops per token-head for the prepare kernel (1.553 TFLOP per
    launch) and 838,997 for the path (1.760 TFLOP): tensor-bound at the measured peaks."""
    wl = I.WORKLOADS["longctx_bf16"]
    m = bench.method_counts(wl, 4)
    th = wl.B * wl.T * wl.H
    assert m["prepare"][1] / th == pytest.approx(740693.33, rel=1e-6)
    assert m["path"][1] / th == pytest.approx(838997.33, rel=1e-6)
    r = bench.roofline_of(*m["prepare"], 7.126, 6775.3, 1915.6)
    assert r["bound"] == "tensor" and r["frac"] == pytest.approx(1.5533e12 / 7.126e-3 / 1915.6e12, rel=1e-3)
