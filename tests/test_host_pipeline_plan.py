"""How the host pipeline cuts the work (CPU): the pieces tile the sequences or the tokens
exactly, token segments are chunk-aligned and long enough to hold the next one's history,
and small transfers stay in one piece."""
import pytest

from linear_recurrent_sequence_causal_gb300.prism import plan_pieces


def _covers(pieces, n):
    assert pieces[0][0] == 0 and pieces[-1][1] == n
    for (a0, a1), (b0, _) in zip(pieces, pieces[1:]):
        assert a1 == b0 and a1 > a0


@pytest.mark.parametrize("B,T", [(8, 4096), (512, 200), (6, 300), (3, 90)])
def test_sequence_groups(B, T):
    p = plan_pieces(B, T, 64, 4, 1 << 40)
    _covers(p, B)
    assert len(p) <= 8


@pytest.mark.parametrize("T,chunk,w", [(65536, 64, 4), (1000, 64, 4), (77, 32, 8), (64, 16, 4)])
def test_token_segments(T, chunk, w):
    p = plan_pieces(1, T, chunk, w, 1 << 40)
    _covers(p, T)
    for a0, a1 in p[:-1]:
        assert (a1 - a0) % chunk == 0 and a1 - a0 >= max(chunk, w)


def test_small_transfers_stay_whole():
    assert plan_pieces(512, 200, 32, 4, 62 << 20) == [(0, 512)]
    assert len(plan_pieces(1, 65536, 64, 4, 2560 << 20)) == 8
    assert len(plan_pieces(4, 1024, 64, 4, 10 << 20, min_piece_bytes=0)) == 4
