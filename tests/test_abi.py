"""The C-ABI library builds, loads and exports every symbol include/prism.h
declares; host-side argument checks answer without touching a GPU (CPU only)."""
import ctypes
import os
import re

import pytest

from linear_recurrent_sequence_causal_gb300 import build, prism

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return prism.load()


def declared_symbols():
    names = []
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            names += re.findall(r"PRISM_API\s+[\w\s\*]+?\b(prism_\w+)\s*\(", src)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert "prism_forward" in names and len(names) >= 5
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
    assert set(names) >= set(prism.EXPORTS)


def test_workspace_and_strerror(lib):
    B, T, H, D, L, C = 8, 4096, 16, 128, 2, 64
    d = prism.make_dims(B, T, H, D, D, 4, L, C, prism.PRISM_BF16)
    NC = T // C
    per = B * H * NC * C * D
    expect = (256 + H * L * 4 * 128 * D * 2 + 4 * per * 2 + 2 * per * 4 + B * H * NC * D * D * 4
              + B * H * NC * 4)
    assert prism.workspace_bytes(d) == expect
    lay = prism.workspace_layout(d)
    assert lay["status"] == 0 and lay["Kl"] is None and lay["gC"] + B * H * NC * 4 == expect
    offs = sorted(v for v in lay.values() if v is not None)
    assert all(o % 256 == 0 for o in offs)
    d0 = prism.make_dims(B, T, H, D, D, 4, 0, C, prism.PRISM_BF16)
    assert prism.workspace_layout(d0)["N"] is None and prism.workspace_layout(d0)["wblocks"] is None
    assert prism.workspace_bytes(prism.make_dims(1, 8, 1, 128, 128, 4, 2, 64, prism.PRISM_F32)) == 0
    f = prism.make_dims(1, 8, 1, 32, 32, 4, 2, 16, prism.PRISM_F32)
    assert prism.workspace_bytes(f) == 256 + 2 * (1 * 8 * 1 * 2 * 32 * 4)   # Kl, Dl fp32
    for code in range(7):
        assert lib.prism_strerror(code)
    assert b"unknown" in lib.prism_strerror(99)


def _fwd(lib, dims, ptrs, ws=0):
    return lib.prism_forward(ctypes.byref(dims), *ptrs, ws, None)


@pytest.mark.parametrize("field,value,code", [
    ("B", 0, 1), ("T", -1, 1), ("d_k", 48, 2), ("chunk", 48, 2), ("L", 9, 2),
    ("conv_width", 9, 2), ("conv_width", 0, 1), ("dtype", 7, 1), ("flags", 16, 1)])
def test_bad_dims(lib, field, value, code):
    d = prism.make_dims(2, 64, 2, 64, 64, 4, 2, 64, prism.PRISM_BF16)
    if field == "d_k":
        d.d_k = d.d_v = value
    else:
        setattr(d, field, value)
    fake = [0x1000] * 13
    assert _fwd(lib, d, fake, 1 << 40) == code


def test_null_and_misaligned_pointers(lib):
    d = prism.make_dims(2, 64, 2, 64, 64, 4, 2, 64, prism.PRISM_BF16)
    good = [0x1000] * 13
    assert _fwd(lib, d, [None] + good[1:], 1 << 40) == 1          # q NULL
    bad = list(good); bad[2] = 0x1008                                 # v misaligned
    assert _fwd(lib, d, bad, 1 << 40) == 3
    assert _fwd(lib, d, good, 16) == 4                                # workspace too small
    nows = list(good); nows[12] = None
    assert _fwd(lib, d, nows, 1 << 40) == 4                           # workspace NULL
    big = 1 << 40
    ws = 0x100000
    # prepare: conv_w NULL with L > 0
    assert lib.prism_prepare(ctypes.byref(d), *[0x1000] * 5, None, *[0x1000] * 4, ws, big, None) == 1
    # prepare: workspace not 256-byte aligned
    assert lib.prism_prepare(ctypes.byref(d), *[0x1000] * 10, 0x1010, big, None) == 3
    # scan: out NULL
    assert lib.prism_scan(ctypes.byref(d), *[0x1000] * 6, ws, big, None, None, None) == 1


def test_decode_step_argument_errors(lib):
    """prism_decode_step rejects bad dims and pointers before any launch."""
    d = prism.Dims(B=2, T=1, H=2, d_k=32, d_v=32, conv_width=4, L=2, chunk=16, dtype=1, flags=0)
    ok = [0x1000] * 12
    d.T = 2
    assert lib.prism_decode_step(ctypes.byref(d), *ok, None) == 1          # T must be 1
    d.T = 1
    d.d_k = 48
    assert lib.prism_decode_step(ctypes.byref(d), *ok, None) == 2          # d_k != d_v
    d.d_k = d.d_v = 96
    assert lib.prism_decode_step(ctypes.byref(d), *ok, None) == 2          # unsupported head dim
    d.d_k = d.d_v = 32
    bad = list(ok); bad[9] = None                                          # no state
    assert lib.prism_decode_step(ctypes.byref(d), *bad, None) == 1
    bad = list(ok); bad[10] = 0x1008                                       # misaligned history
    assert lib.prism_decode_step(ctypes.byref(d), *bad, None) == 3



def test_backward_argument_errors(lib):
    """prism_backward and its workspace query reject bad dims and pointers before any
    launch."""
    d = prism.make_dims(2, 64, 2, 32, 32, 4, 2, 64, prism.PRISM_BF16)
    nbytes = lib.prism_backward_workspace_bytes(ctypes.byref(d))
    assert nbytes > 0 and nbytes % 256 == 0
    d2 = prism.make_dims(2, 128, 2, 32, 32, 4, 2, 64, prism.PRISM_BF16)
    assert lib.prism_backward_workspace_bytes(ctypes.byref(d2)) > nbytes     # grows with T
    ok = [0x1000] * 21
    ws = 0x100000

    def call(dims, ptrs, wsb=1 << 40, w=ws):
        return lib.prism_backward(ctypes.byref(dims), *ptrs, w, wsb, None)

    bad = prism.make_dims(2, 64, 2, 32, 64, 4, 2, 64, prism.PRISM_BF16)       # d_k != d_v
    assert lib.prism_backward_workspace_bytes(ctypes.byref(bad)) == 0
    assert call(bad, ok) == 2
    big_l = prism.make_dims(2, 64, 2, 32, 32, 4, 9, 64, prism.PRISM_BF16)     # L > 8
    assert call(big_l, ok) == 2
    for i in (0, 9, 11, 15):                       # q, d_out, dq, dbeta NULL
        p = list(ok)
        p[i] = None
        assert call(d, p) == 1, f"pointer {i} NULL accepted"
    p = list(ok)
    p[10] = None                                   # d_final_state may be NULL
    assert call(d, p, wsb=16) == 4                 # ... then the small workspace is reported
    p = list(ok)
    p[12] = 0x1004                                 # dk misaligned
    assert call(d, p) == 3
    assert call(d, ok, wsb=nbytes - 1) == 4        # workspace too small


def test_static_status_argument_errors(lib):
    """prism_static_status rejects bad dims, a NULL result pointer and dims whose
    workspace exceeds the static scratch before touching the device."""
    word = ctypes.c_int(-1)
    d = prism.make_dims(2, 64, 2, 32, 32, 4, 2, 32, prism.PRISM_BF16)
    bad = prism.make_dims(2, 64, 2, 32, 32, 4, 2, 48, prism.PRISM_BF16)       # chunk 48
    assert lib.prism_static_status(ctypes.byref(bad), ctypes.byref(word), None) == 2
    assert lib.prism_static_status(ctypes.byref(d), None, None) == 1
    big = prism.make_dims(64, 65536, 32, 128, 128, 4, 4, 64, prism.PRISM_BF16)
    assert prism.workspace_bytes(big) > prism.STATIC_SCRATCH_BYTES
    assert lib.prism_static_status(ctypes.byref(big), ctypes.byref(word), None) == 7
    assert word.value == -1


def test_device_status_argument_errors(lib):
    """prism_device_status rejects bad dims, a NULL result pointer and a missing, misaligned
    or short workspace before touching the device."""
    d = prism.make_dims(2, 64, 2, 32, 32, 4, 2, 32, prism.PRISM_BF16)
    need = prism.workspace_bytes(d)
    word = ctypes.c_int(-1)

    def call(dims, ws, nbytes, out=ctypes.byref(word)):
        return lib.prism_device_status(ctypes.byref(dims), ws, nbytes, out, None)

    bad = prism.make_dims(2, 64, 2, 32, 32, 4, 2, 48, prism.PRISM_BF16)       # chunk 48
    assert call(bad, 0x100000, need) == 2
    assert call(d, 0x100000, need, None) == 1
    assert call(d, 0x100010, need) == 3
    assert call(d, None, need) == 4
    assert call(d, 0x100000, need - 1) == 4
    assert word.value == -1


def test_scan_segments_rule(lib):
    """The sequence split is a function of the dims alone: taken only for the tcgen05
    scan (bf16, d = 128, chunk 32 or 64) when the first pass of B*H*4*(2P-1) CTAs fits
    the 152 SMs with P >= 3 and at least 8 chunks per segment; the workspace then
    holds three [B,H,P,d,d] fp32 arrays."""
    bf = prism.PRISM_BF16
    seg = lambda *a, **k: prism.scan_segments(prism.make_dims(*a, **k))
    assert seg(1, 65536, 32, 128, 128, 4, 4, 64, bf) == 1          # 128 scan CTAs: no room
    assert seg(8, 4096, 16, 128, 128, 4, 2, 64, bf) == 1
    assert seg(1, 65536, 4, 128, 128, 4, 4, 64, bf) == 5           # 16 x 9 = 144 <= 152
    assert seg(1, 65536, 1, 128, 128, 4, 4, 64, bf) == 16          # capped
    assert seg(1, 4096, 2, 128, 128, 4, 2, 64, bf) == 8            # 64 chunks / 8
    assert seg(1, 1000, 1, 128, 128, 4, 2, 64, bf) == 1            # 16 chunks: too short
    assert seg(1, 65536, 4, 128, 128, 4, 4, 64, bf, flags=prism.PRISM_FLAG_NO_SEQ_SPLIT) == 1
    assert seg(1, 65536, 4, 64, 64, 4, 4, 64, bf) == 1             # d < 128: other scan kernel
    assert seg(1, 65536, 4, 128, 128, 4, 4, 16, bf) == 1           # chunk 16: other scan kernel
    assert seg(1, 4096, 1, 32, 32, 4, 2, 16, prism.PRISM_F32) == 1
    assert seg(1, 64, 1, 100, 100, 4, 2, 16, bf) == 0              # invalid dims
    for B, T, H in ((1, 65536, 4), (2, 3000, 1), (1, 4096, 2), (8, 4096, 16)):
        for C in (32, 64):
            d = prism.make_dims(B, T, H, 128, 128, 4, 2, C, bf)
            P = prism.scan_segments(d)
            NC = -(-T // C)
            assert P == 1 or (P >= 3 and B * H * 4 * (2 * P - 1) <= 152 and NC >= 8 * P and P <= 16)
            lay = prism.workspace_layout(d)
            if P == 1:
                assert lay["seg"] is None
            else:
                assert lay["seg"] % 256 == 0
                assert prism.workspace_bytes(d) >= lay["seg"] + 3 * B * H * P * 128 * 128 * 4
                nosplit = prism.make_dims(B, T, H, 128, 128, 4, 2, C, bf,
                                          flags=prism.PRISM_FLAG_NO_SEQ_SPLIT)
                assert prism.workspace_layout(nosplit)["seg"] is None
                assert prism.workspace_bytes(nosplit) == lay["seg"]


def test_debug_bounds_word_only_in_the_debug_build(lib):
    """The normal build answers that it is not the bounds-checked one (no GPU touched)."""
    if os.environ.get("PRISM_LIBRARY"):
        pytest.skip("another build of the library is loaded")
    word = ctypes.c_int(-1)
    assert lib.prism_debug_bounds(ctypes.byref(word), 0) == 2      # PRISM_ERR_UNSUPPORTED
    assert word.value == 0
    assert lib.prism_debug_bounds(None, 0) == 1                    # PRISM_ERR_INVALID_ARG
    assert prism.debug_bounds() is None
