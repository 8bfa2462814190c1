"""Pins for the oracle's decoder window attention (CPU only).

The window partition against a token-by-token labelling (each token's window
from its row and column alone) and against the pages' worked numbers for a
full window (tests/golden/decoder_window_visible_set.txt: about 512 queries
against 1,541 keys, 517 at stream start); one window covering the frame
reduces the layer to the session oracle's chunk attention; causality; the
cache keeps the last four frames.
"""
import math
import os

import numpy as np
import pytest

import synthetic as syn
from oracle import OracleSession, f64_to_bf16_bits
from oracle.decoder import DecoderLayerOracle, window_partition

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                vals[k] = int(v)
    return vals


def _label(gh, gw, window, shifted):
    """Window id of every token from its own row and column: the band index
    along each axis is floor((x + window/2) / window) when shifted, else
    floor(x / window)."""
    off = window // 2 if shifted else 0
    rb = (np.arange(gh) + (window - off if shifted else 0)) // window
    cb = (np.arange(gw) + (window - off if shifted else 0)) // window
    nc = cb.max() + 1
    return rb[:, None] * nc + cb[None, :]


@pytest.mark.parametrize("gh,gw,window", [(45, 80, 16), (40, 40, 16), (16, 16, 16), (10, 7, 4), (48, 84, 16)])
@pytest.mark.parametrize("shifted", [False, True])
def test_partition_covers_every_token_once_and_matches_the_labelling(gh, gw, window, shifted):
    wins = window_partition(gh, gw, window, shifted)
    cover = np.zeros((gh, gw), int)
    lab = _label(gh, gw, window, shifted)
    for i, (r0, c0, nr, nc) in enumerate(wins):
        assert 1 <= nr <= window and 1 <= nc <= window
        cover[r0:r0 + nr, c0:c0 + nc] += 1
        assert np.all(lab[r0:r0 + nr, c0:c0 + nc] == lab[r0, c0])
    assert np.all(cover == 1)
    assert len(set(lab.ravel().tolist())) == len(wins)


def test_full_window_visible_set_matches_the_page():
    g = _golden("decoder_window_visible_set.txt")
    H, d = 1, 8
    lay = DecoderLayerOracle(32, 32, g["grid_h"], False, H, d, cache_frames=g["window_frames"])
    gk = np.zeros((g["n_sink"], H, d), np.uint16)
    x = np.zeros((g["chunk_frames"], 32, 32, H, d), np.uint16)
    r0, c0, nr, nc = lay.windows[0]
    assert nr * nc * g["chunk_frames"] == g["queries"]
    keys = lambda: g["n_sink"] + sum(nr * nc for _ in lay.cache) + g["chunk_frames"] * nr * nc
    assert keys() == g["keys_empty_cache"]
    for _ in range(3):
        lay.commit(x, x)
    assert keys() == g["keys_full_cache"]
    assert len(lay.cache) == g["window_frames"]


def test_one_window_over_the_frame_is_the_session_attention():
    gh, gw, H, d = 4, 6, 2, 16
    sh = syn.Shape("one window", H, d, gh, gw, 2, 4, 5, 1)
    gkb, gvb = syn.session_sinks(sh, 3)
    lay = DecoderLayerOracle(gh, gw, 8, False, H, d, cache_frames=4, t_clock0=3)
    ses = OracleSession(H, d, gh, gw, 2, 4, 5, 1, gkb, gvb, t_clock0=3)
    assert lay.windows == [(0, 0, gh, gw)]
    rng = np.random.default_rng(0)
    for c in range(4):
        q, k, v, ck, cv = (syn.normal_bf16_bits((2, gh, gw, H, d), rng) for _ in range(5))
        o = lay.step(q, k, v, gkb[0], gvb[0])
        qo, ko = ses.rope3d_qk(q.reshape(-1, H, d), k.reshape(-1, H, d))
        ref, _ = ses.chunk_attention(0, qo, ko, v.reshape(-1, H, d))
        assert np.allclose(o.reshape(-1, H, d), ref, rtol=1e-12, atol=1e-12)
        lay.commit(ck, cv)
        ses.cache_commit(ck.reshape(-1, H, d), cv.reshape(-1, H, d))


def test_a_later_chunk_changes_no_earlier_output():
    gh, gw, H, d = 10, 12, 1, 8
    rng = np.random.default_rng(1)
    chunks = [[syn.normal_bf16_bits((2, gh, gw, H, d), rng) for _ in range(5)] for _ in range(3)]
    gk, gv = syn.normal_bf16_bits((5, H, d), rng), syn.normal_bf16_bits((5, H, d), rng)
    outs = []
    for alt in (False, True):
        lay = DecoderLayerOracle(gh, gw, 4, True, H, d)
        res = []
        for c, (q, k, v, ck, cv) in enumerate(chunks):
            if alt and c == 2:
                q, k, v = (syn.normal_bf16_bits((2, gh, gw, H, d), rng) for _ in range(3))
            res.append(lay.step(q, k, v, gk, gv))
            lay.commit(ck, cv)
        outs.append(res)
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])
    assert not np.allclose(outs[0][2], outs[1][2])


def _tiled(pattern, reps_h, reps_w):
    """A frame stack [F][gh][gw][H][d] made by repeating one window's tokens
    [F][wh][ww][H][d] reps_h x reps_w times across the frame."""
    return np.tile(pattern, (1, reps_h, reps_w, 1, 1))


def test_windows_with_identical_contents_give_identical_outputs():
    """Spatial positions are relative to the window ([H3-page] 3.2 Iteration 2,
    "Space"): four 4x4 windows of an 8x8 frame that hold the same tokens, the
    same cached frames and see the same global tokens compute the same
    attention, bit for bit. With the frame's absolute (h, w) the windows at
    column 4 or row 4 would rotate their tokens differently."""
    H, d, w = 2, 12, 4
    rng = np.random.default_rng(7)
    lay = DecoderLayerOracle(8, 8, w, False, H, d, cache_frames=4, t_clock0=11)
    assert lay.windows == [(0, 0, 4, 4), (0, 4, 4, 4), (4, 0, 4, 4), (4, 4, 4, 4)]
    gk, gv = syn.normal_bf16_bits((5, H, d), rng), syn.normal_bf16_bits((5, H, d), rng)
    for c in range(3):
        q, k, v, ck, cv = (_tiled(syn.normal_bf16_bits((2, w, w, H, d), rng), 2, 2) for _ in range(5))
        o = lay.step(q, k, v, gk, gv)
        ref = o[:, 0:4, 0:4]
        for r0, c0 in ((0, 4), (4, 0), (4, 4)):
            assert np.array_equal(o[:, r0:r0 + 4, c0:c0 + 4], ref), (c, r0, c0)
        # the windows' outputs are not trivially equal: different windows of a
        # frame with distinct contents differ
        lay.commit(ck, cv)


def test_shifted_interior_window_rotates_from_its_own_corner():
    """The first token of a window that starts at (r0, c0) != (0, 0) sits at
    spatial position (0, 0) of its window, so its h and w sub-vectors are not
    rotated at all (a rotation by angle 0 is the identity), while its t
    sub-vector turns by the frame time. Token (r0, c0 + 1) turns its w
    sub-vector by exactly one position step and leaves h alone."""
    H, d = 1, 6                       # d = 6: one pair per axis, frequency 1 (angle = position)
    lay = DecoderLayerOracle(8, 8, 4, True, H, d, cache_frames=2, t_clock0=5)
    # cuts at 0, 2, 6, 8 on each axis: window 4 is the interior one at (2, 2)
    assert lay.windows[4] == (2, 2, 4, 4)
    x = np.random.default_rng(3).standard_normal((1, 8, 8, H, d))
    y = lay._rotate(x, 0)
    first = y[0, 2, 2, 0]
    assert np.array_equal(first[2:6], x[0, 2, 2, 0, 2:6])           # h and w pairs untouched
    t_ang = 5.0                                                      # t_clock0 + frame 0
    x0, x1 = x[0, 2, 2, 0, 0], x[0, 2, 2, 0, 1]
    assert np.allclose(first[0:2], [x0 * math.cos(t_ang) - x1 * math.sin(t_ang),
                                    x0 * math.sin(t_ang) + x1 * math.cos(t_ang)], rtol=0, atol=1e-15)
    nxt = y[0, 2, 3, 0]
    assert np.array_equal(nxt[2:4], x[0, 2, 3, 0, 2:4])             # same row of the window: h = 0
    a0, a1 = x[0, 2, 3, 0, 4], x[0, 2, 3, 0, 5]
    assert np.allclose(nxt[4:6], [a0 * math.cos(1.0) - a1 * math.sin(1.0),
                                  a0 * math.sin(1.0) + a1 * math.cos(1.0)], rtol=0, atol=1e-15)
