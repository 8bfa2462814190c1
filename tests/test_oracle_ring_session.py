"""Pins for the oracle's ring cache and session (CPU only).

Ring: the slot of frame g is g mod W, checked against a closed form for the
slot table and against a deque brute force of "the last W frames".
Session: the visible-set size of the H3 project page's worked example
(tests/golden/decoder_window_visible_set.txt), causality (frames already
evicted and future chunks change nothing), and clock-shift invariance of
the scores (the Iteration 4 fix: a score is a function of the gap in time,
not of absolute time).
Chunks of varying length and a recent-history window (the unit rhythm):
recent(h) against a plain list of every committed frame (including commits
longer than the ring), positions of a chunk of any length from the frame
counter, and attention with a history window against the same visible set
assembled by hand.
"""
import collections
import math
import os

import numpy as np
import pytest

import synthetic as syn
from oracle import (OracleSession, RingCache, attention, bf16_bits_to_f64, f64_to_bf16_bits, rope3d,
                    token_positions)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                vals[k] = int(v)
    return vals


@pytest.mark.parametrize("W,F", [(4, 2), (6, 2), (5, 2), (3, 1), (8, 2)])
def test_slot_table_closed_form_and_deque(W, F):
    T, H, d = 3, 1, 2
    ring = RingCache(W, T, H, d)
    window = collections.deque(maxlen=W)
    for chunk in range(23):
        frames = np.arange(ring.n, ring.n + F, dtype=np.float64)
        k = np.repeat(frames, T)[:, None, None] * np.ones((1, H, d))
        ring.commit(k, -k, F)
        window.extend(range(ring.n - F, ring.n))
        n = ring.n
        for s in range(W):
            cands = [g for g in range(n) if g % W == s]
            assert ring.slot_frame[s] == (max(cands) if cands else -1)
            if cands:   # the slot holds exactly that frame's tokens
                assert np.all(ring.k[s * T:(s + 1) * T] == max(cands))
        assert sorted(g for g in ring.slot_frame if g >= 0) == sorted(window)
        assert ring.slot_of(n) == n % W


def test_visible_set_size_matches_pages_worked_example():
    g = _load_golden("decoder_window_visible_set.txt")
    sess = OracleSession(1, 8, g["grid_h"], g["grid_w"], g["chunk_frames"],
                         g["window_frames"], g["n_sink"], 1)
    Lq = sess.F * sess.T
    assert Lq == g["queries"]
    kz = np.zeros((Lq, 1, 8), np.uint16)
    k, _ = sess.visible_kv(0, kz, kz)
    assert k.shape[0] == g["keys_empty_cache"]
    for _ in range(3):
        sess.cache_commit(kz, kz)
    k, _ = sess.visible_kv(0, kz, kz)
    assert k.shape[0] == g["keys_full_cache"]


def _session(shape, **kw):
    sk, sv = syn.session_sinks(shape, 1)
    return OracleSession(shape.n_heads, shape.head_dim, shape.grid_h, shape.grid_w,
                         shape.chunk_frames, shape.window_frames, shape.n_sink,
                         shape.n_steps, sk, sv, **kw)


def test_evicted_frames_do_not_matter():
    shape = syn.TINY
    a, b = _session(shape), _session(shape)
    for c in range(4):
        x = syn.chunk_inputs(shape, 1, chunk=c)
        a.cache_commit(x.clean_k, x.clean_v)
        y = syn.chunk_inputs(shape, 1, chunk=c + 100) if c == 0 else x   # chunk 0 differs
        b.cache_commit(y.clean_k, y.clean_v)
    # W = 4 frames, F = 2: after 4 chunks frames 0 and 1 (chunk 0) are evicted
    assert a.ring.n == 8 and sorted(a.ring.slot_frame) == [4, 5, 6, 7]
    x = syn.chunk_inputs(shape, 1, chunk=9)
    qa, ka = a.rope3d_qk(x.q[0], x.k[0])
    qb, kb = b.rope3d_qk(x.q[0], x.k[0])
    oa, la = a.chunk_attention(0, qa, ka, x.v[0])
    ob, lb = b.chunk_attention(0, qb, kb, x.v[0])
    assert np.array_equal(oa, ob) and np.array_equal(la, lb)


def test_uncommitted_future_chunk_does_not_leak():
    shape = syn.TINY
    a = _session(shape)
    x = syn.chunk_inputs(shape, 1, chunk=0)
    q, k = a.rope3d_qk(x.q[1], x.k[1])
    before, _ = a.chunk_attention(1, q, k, x.v[1])
    future = syn.chunk_inputs(shape, 1, chunk=1)
    _ = a.rope3d_qk(future.q[0], future.k[0])    # rotating another chunk's Q/K is stateless
    after, _ = a.chunk_attention(1, q, k, x.v[1])
    assert np.array_equal(before, after)


def test_step_selects_its_own_sink_bank():
    shape = syn.TINY
    a = _session(shape)
    x = syn.chunk_inputs(shape, 1)
    q, k = a.rope3d_qk(x.q[0], x.k[0])
    o0, _ = a.chunk_attention(0, q, k, x.v[0])
    o1, _ = a.chunk_attention(1, q, k, x.v[0])
    assert not np.allclose(o0, o1)
    kv = a.visible_kv(1, k, x.v[0])[0]
    assert np.array_equal(kv[:shape.n_sink], a.sink_k[1])


def test_clock_shift_invariance_without_sinks():
    # With no unrotated sink keys in the visible set, every score depends only
    # on time differences, so shifting the stream clock changes nothing
    # (exactly, before bf16 rounding).
    g = np.random.default_rng(0)
    T, F, W, H, d = 6, 2, 4, 2, 64
    hist = g.standard_normal((W * T, H, d))
    chunk_k = g.standard_normal((F * T, H, d))
    chunk_v = g.standard_normal((F * T, H, d))
    q = g.standard_normal((F * T, H, d))
    hist_v = g.standard_normal((W * T, H, d))
    outs = []
    for clock in (0, 100, 1000):
        th, hh, wh = token_positions(W * T, 2, 3, clock)          # frames clock .. clock+3
        tc, hc, wc = token_positions(F * T, 2, 3, clock + W)      # the chunk follows them
        k = np.concatenate([rope3d(hist, th, hh, wh, 1e4), rope3d(chunk_k, tc, hc, wc, 1e4)])
        v = np.concatenate([hist_v, chunk_v])
        o, _ = attention(rope3d(q, tc, hc, wc, 1e4), k, v, 1 / 8)
        outs.append(o)
    assert np.allclose(outs[0], outs[1], rtol=0, atol=1e-11)
    assert np.allclose(outs[0], outs[2], rtol=0, atol=1e-11)


def test_commit_rotates_keys_at_absolute_frames():
    shape = syn.TINY
    a = _session(shape, t_clock0=50)
    x0 = syn.chunk_inputs(shape, 1, chunk=0)
    x1 = syn.chunk_inputs(shape, 1, chunk=1)
    a.cache_commit(x0.clean_k, x0.clean_v)
    a.cache_commit(x1.clean_k, x1.clean_v)
    T = shape.tokens_per_frame
    # frame 3 (second frame of chunk 1) is in slot 3 with time position 50 + 3
    t, h, w = token_positions(T, shape.grid_h, shape.grid_w, 53)
    want = rope3d(bf16_bits_to_f64(x1.clean_k)[T:2 * T], t, h, w, 1e4)
    got = a.ring.k[3 * T:4 * T]
    assert np.allclose(got, want, rtol=2.0 ** -8, atol=1e-30)
    assert np.array_equal(a.ring.v[3 * T:4 * T], bf16_bits_to_f64(x1.clean_v)[T:2 * T])


# ---- chunks of varying length and a recent-history window (the unit rhythm)

def test_recent_history_against_a_list_of_committed_frames():
    # commits of 9, 3, 2, 3, 2, ... frames (the page's first window, then the
    # alternating chunks) into a ring of W frames; recent(h) must return the
    # last h frames in stream order, taken from a plain list of every frame
    T, H, d = 2, 1, 1
    for W in (3, 4, 5):
        ring = RingCache(W, T, H, d)
        stream = []
        for F in [9, 3, 2, 3, 2, 3, 2, 3]:
            frames = np.arange(ring.n, ring.n + F, dtype=np.float64)
            k = np.repeat(frames, T)[:, None, None]
            ring.commit(k, -k, F)
            stream.extend(range(ring.n - F, ring.n))
            kept = stream[-W:]
            assert sorted(g for g in ring.slot_frame if g >= 0) == kept   # later frames of one commit evict earlier ones
            for h in range(0, min(ring.n, W) + 1):
                rk, rv, fr = ring.recent(h)
                assert fr == stream[len(stream) - h:]
                assert np.array_equal(rk[:, 0, 0], np.repeat(np.array(fr, np.float64), T))
                assert np.array_equal(rv, -rk)
            with pytest.raises(ValueError):
                ring.recent(min(ring.n, W) + 1)


def test_chunk_of_other_length_takes_positions_from_the_frame_counter():
    shape = syn.TINY
    a = _session(shape, t_clock0=7)
    T = shape.tokens_per_frame
    g = np.random.default_rng(3)
    for F in (3, 1, 2):
        n0 = a.n_committed
        x = g.standard_normal((F * T, shape.n_heads, shape.head_dim))
        bits = f64_to_bf16_bits(x)
        q, _ = a.rope3d_qk(bits, bits, frames=F)
        t, h, w = token_positions(F * T, shape.grid_h, shape.grid_w, 7 + n0)
        assert t[0] == 7 + n0 and t[-1] == 7 + n0 + F - 1
        assert np.array_equal(q, f64_to_bf16_bits(rope3d(bf16_bits_to_f64(bits), t, h, w, 1e4)))
        a.cache_commit(bits, bits, frames=F)
        assert a.n_committed == n0 + F


def test_history_window_selects_exactly_the_last_frames():
    # with hist = h the visible set is bank[step] + frames n-h .. n-1 + chunk,
    # and the output equals attention over that set assembled by hand
    shape = syn.TINY
    a = _session(shape)
    T = shape.tokens_per_frame
    g = np.random.default_rng(5)
    kept = {}
    for F in (3, 2, 3):
        k = f64_to_bf16_bits(g.standard_normal((F * T, shape.n_heads, shape.head_dim)))
        v = f64_to_bf16_bits(g.standard_normal((F * T, shape.n_heads, shape.head_dim)))
        n0 = a.n_committed
        a.cache_commit(k, v, frames=F)
        for f in range(F):
            kept[n0 + f] = (a.ring.k[((n0 + f) % a.W) * T:((n0 + f) % a.W + 1) * T].copy(),
                            bf16_bits_to_f64(v)[f * T:(f + 1) * T])
    n = a.n_committed                     # 8 frames committed into W = 4 slots
    F = 2
    q = f64_to_bf16_bits(g.standard_normal((F * T, shape.n_heads, shape.head_dim)))
    ck = f64_to_bf16_bits(g.standard_normal((F * T, shape.n_heads, shape.head_dim)))
    cv = f64_to_bf16_bits(g.standard_normal((F * T, shape.n_heads, shape.head_dim)))
    for h in (0, 2, 3, 4):
        kk, _ = a.visible_kv(0, ck, cv, hist=h)
        assert kk.shape[0] == shape.n_sink + h * T + F * T
        hk = np.concatenate([kept[gg][0] for gg in range(n - h, n)] or [np.empty((0, shape.n_heads, shape.head_dim))])
        hv = np.concatenate([kept[gg][1] for gg in range(n - h, n)] or [np.empty((0, shape.n_heads, shape.head_dim))])
        K = np.concatenate([a.sink_k[0], hk, bf16_bits_to_f64(ck)])
        V = np.concatenate([a.sink_v[0], hv, bf16_bits_to_f64(cv)])
        want, _ = attention(bf16_bits_to_f64(q), K, V, a.scale)
        got, _ = a.chunk_attention(0, q, ck, cv, hist=h)
        assert np.allclose(got, want, rtol=1e-12, atol=1e-12)
    full, _ = a.chunk_attention(0, q, ck, cv)
    last_w, _ = a.chunk_attention(0, q, ck, cv, hist=a.W)
    assert np.allclose(full, last_w, rtol=1e-12, atol=1e-12)   # the whole ring = the last W frames
