"""Pins for the oracle's decoder window attention (CPU only).

The window partition against a token-by-token labelling (each token's window
from its row and column alone) and against the pages' worked numbers for a
full window (tests/golden/decoder_window_visible_set.txt: about 512 queries
against 1,541 keys, 517 at stream start); one window covering the frame
reduces the layer to the session oracle's chunk attention; causality; the
cache keeps the last four frames.
"""
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
