"""How the host-to-host forward (prism_forward_host) cuts the work, and its argument checks
(CPU: the library's host code, no GPU): the pieces tile the sequences or the tokens
exactly, groups of sequences start 16-byte aligned in the gate arrays, token segments are
chunk-aligned and long enough to hold the next one's history, and small transfers stay in
one piece."""
import ctypes

import pytest

from linear_recurrent_sequence_causal_gb300 import build, prism


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    return prism.load()


def _covers(pieces, n):
    assert pieces[0][0] == 0 and pieces[-1][1] == n
    for (a0, a1), (b0, _) in zip(pieces, pieces[1:]):
        assert a1 == b0 and a1 > a0


def _dims(B, T, H=2, D=64, chunk=64, w=4, L=2, dtype=prism.PRISM_BF16):
    return prism.make_dims(B, T, H, D, D, w, L, chunk, dtype)


@pytest.mark.parametrize("B,T,H", [(8, 4096, 2), (512, 200, 2), (6, 300, 2), (3, 90, 1), (6, 77, 1),
                                   (10, 33, 2)])
def test_sequence_groups(B, T, H):
    p = prism.plan_pieces(_dims(B, T, H), 8, 0)
    _covers(p, B)
    assert len(p) <= 8
    for a0, _ in p:
        assert (a0 * T * H * 4) % 16 == 0, "a piece's log_alpha / beta would start misaligned"


@pytest.mark.parametrize("T,chunk,w", [(65536, 64, 4), (1000, 64, 4), (77, 32, 8), (64, 16, 4)])
def test_token_segments(T, chunk, w):
    p = prism.plan_pieces(_dims(1, T, chunk=chunk, w=w), 8, 0)
    _covers(p, T)
    for a0, a1 in p[:-1]:
        assert (a1 - a0) % chunk == 0 and a1 - a0 >= max(chunk, w)


def test_small_transfers_stay_whole():
    # 512 x 200 tokens x 2 heads x 32: 62.5 MiB of q, k, v and out
    assert prism.plan_pieces(_dims(512, 200, 2, 32, 32), 8, 32 << 20) == [(0, 512)]
    assert len(prism.plan_pieces(_dims(1, 65536, 32, 128), 8, 32 << 20)) == 8
    assert len(prism.plan_pieces(_dims(4, 1024, 2, 64), 8, 0)) == 4


def test_arena_and_argument_errors(_lib):
    lib = _lib
    d = _dims(6, 300)
    n_ok = lib.prism_host_arena_bytes(ctypes.byref(d), 4, 0)
    assert n_ok > 0 and n_ok % 256 == 0
    # the arena holds the inputs and outputs at full size plus a piece's workspace
    assert n_ok > 6 * 300 * 2 * 64 * (3 * 2 + 4)
    assert lib.prism_host_arena_bytes(ctypes.byref(d), 0, 0) == 0
    assert lib.prism_host_arena_bytes(ctypes.byref(d), prism.PRISM_HOST_MAX_PIECES + 1, 0) == 0
    n = ctypes.c_int(0)
    bounds = (ctypes.c_int * 20)()
    assert lib.prism_host_plan(ctypes.byref(d), 0, 0, ctypes.byref(n), bounds) == 1
    tm = _dims(1, 300)
    tm.flags = prism.PRISM_FLAG_VHIST_TOKEN_MAJOR
    assert lib.prism_host_plan(ctypes.byref(tm), 4, 0, ctypes.byref(n), bounds) == 1
    bad = _dims(6, 300, chunk=48)
    assert lib.prism_host_plan(ctypes.byref(bad), 4, 0, ctypes.byref(n), bounds) == 2
    assert lib.prism_host_plan(ctypes.byref(d), 4, 0, None, bounds) == 1

    host = [0x1000] * 12                     # never dereferenced: the checks come first

    def call(ptrs, arena, nbytes):
        return lib.prism_forward_host(ctypes.byref(d), *ptrs, 4, 0, arena, nbytes, None)

    p = list(host)
    p[0] = None                              # q
    assert call(p, 0x100000, n_ok) == 1
    p = list(host)
    p[6] = None                              # Wk with L = 2
    assert call(p, 0x100000, n_ok) == 1
    assert call(host, 0x100000, n_ok - 1) == 4
    assert call(host, None, n_ok) == 4
    assert call(host, 0x100080, n_ok) == 3


def test_plan_properties_over_random_dims():
    """For random supported dims: the pieces tile the work, stay within max_pieces, groups
    of sequences start 16-byte aligned in the gate arrays, token segments are chunk-aligned
    and hold at least max(chunk, w) tokens (but the last), and the arena is at least the
    full-size inputs and outputs."""
    hyp = pytest.importorskip("hypothesis")
    st = pytest.importorskip("hypothesis.strategies")

    @hyp.settings(max_examples=300, deadline=None)
    @hyp.given(B=st.integers(1, 64), T=st.integers(1, 5000), H=st.integers(1, 8),
               D=st.sampled_from([16, 32, 64, 128]), chunk=st.sampled_from([16, 32, 64]),
               w=st.integers(1, 8), L=st.integers(0, 8), pieces=st.integers(1, 16),
               floor=st.sampled_from([0, 1 << 16, 32 << 20]), f32=st.booleans())
    def check(B, T, H, D, chunk, w, L, pieces, floor, f32):
        if f32 and D > 64:
            D = 64
        d = prism.make_dims(B, T, H, D, D, w, L, chunk, prism.PRISM_F32 if f32 else prism.PRISM_BF16)
        p = prism.plan_pieces(d, pieces, floor)
        n = B if B > 1 else T
        _covers(p, n)
        assert 1 <= len(p) <= pieces
        if B > 1:
            for a0, _ in p:
                assert (a0 * T * H * 4) % 16 == 0
        else:
            for a0, a1 in p[:-1]:
                assert (a1 - a0) % chunk == 0 and a1 - a0 >= max(chunk, w)
        esz = 4 if f32 else 2
        arena = prism.host_arena_bytes(d, pieces, floor)
        assert arena % 256 == 0
        assert arena >= B * T * H * D * (3 * esz + 4) + B * T * H * 8

    check()
