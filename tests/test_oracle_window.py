"""Pins for the oracle's page-faithful window (CPU only).

The window of the pages has a fixed prefix and a moving part with an
asymmetric mask: prefix rows attend only to the prefix, moving rows attend to
everything ([teardown] "A window that slides, and a prefix that doesn't";
[H3 page] section 3.1.2 "Prefix cache"). The oracle computes it as two
attentions over two key sets; here it is checked against one dense attention
over the whole window with that mask written out element by element, against
the consequences the pages draw from the mask (the prefix outputs are a
function of the prefix alone, so they do not change when the moving rows do),
and the moving rows against the ring path when the recomputed history equals
what the ring holds. Recomputed history rows keep their own frame times.
"""
import math

import numpy as np
import pytest

import synthetic as syn
from oracle import (OracleSession, bf16_bits_to_f64, f64_to_bf16_bits, rope3d, token_positions)


def _masked_dense(q, k, v, scale, allowed):
    """softmax over the allowed keys only, one (row, head) at a time, from the
    definition: exp of the scores minus their max over allowed keys."""
    Lq, H, d = q.shape
    o = np.zeros((Lq, H, v.shape[2]))
    lse = np.zeros((H, Lq))
    for h in range(H):
        for i in range(Lq):
            js = [j for j in range(k.shape[0]) if allowed[i, j]]
            s = np.array([scale * math.fsum(q[i, h] * k[j, h]) for j in js])
            m = s.max()
            e = np.exp(s - m)
            z = math.fsum(e)
            o[i, h] = (e[:, None] * v[js, h]).sum(0) / z
            lse[h, i] = m + math.log(z)
    return o, lse


def _session(S=7, W=4):
    sh = syn.Shape("window tiny", 2, 8, 2, 3, 2, W, S, 2)
    sk, sv = syn.session_sinks(sh, 9)
    return sh, OracleSession(sh.n_heads, sh.head_dim, sh.grid_h, sh.grid_w, sh.chunk_frames, W, S, 2, sk, sv)


@pytest.mark.parametrize("with_prefix", [True, False])
def test_window_equals_dense_attention_with_the_asymmetric_mask(with_prefix):
    sh, a = _session()
    g = np.random.default_rng(1)
    T, S = sh.tokens_per_frame, sh.n_sink
    M = 5 * T                                             # 2 frames of history + 3 of chunk
    P = S if with_prefix else 0
    q = f64_to_bf16_bits(g.standard_normal((P + M, sh.n_heads, sh.head_dim)))
    km = f64_to_bf16_bits(g.standard_normal((M, sh.n_heads, sh.head_dim)))
    vm = f64_to_bf16_bits(g.standard_normal((M, sh.n_heads, sh.head_dim)))
    for step in (0, 1):
        got, lse = a.window_attention(step, q, km, vm, with_prefix)
        K = np.concatenate([a.sink_k[step], bf16_bits_to_f64(km)])
        V = np.concatenate([a.sink_v[step], bf16_bits_to_f64(vm)])
        allowed = np.ones((P + M, S + M), bool)
        allowed[:P, S:] = False                           # prefix rows: prefix keys only
        want, wl = _masked_dense(bf16_bits_to_f64(q), K, V, a.scale, allowed)
        assert np.allclose(got, want, rtol=1e-12, atol=1e-12)
        assert np.allclose(lse, wl, rtol=1e-12, atol=1e-12)


def test_prefix_outputs_do_not_see_the_moving_rows():
    sh, a = _session()
    g = np.random.default_rng(2)
    T, S = sh.tokens_per_frame, sh.n_sink
    M = 3 * T
    q = f64_to_bf16_bits(g.standard_normal((S + M, sh.n_heads, sh.head_dim)))
    k1, v1, k2, v2 = (f64_to_bf16_bits(g.standard_normal((M, sh.n_heads, sh.head_dim))) for _ in range(4))
    o1, _ = a.window_attention(0, q, k1, v1, True)
    o2, _ = a.window_attention(0, q, k2, v2, True)
    assert np.array_equal(o1[:S], o2[:S])                 # the prefix is a function of the session only
    assert not np.allclose(o1[S:], o2[S:])


def test_moving_rows_match_the_ring_path_when_history_is_the_ring():
    # when the recomputed history K/V are exactly what the ring holds, the
    # chunk rows of the window see the same key set as the ring path
    sh, a = _session(W=4)
    g = np.random.default_rng(3)
    T = sh.tokens_per_frame
    for F in (2, 2):
        raw = f64_to_bf16_bits(g.standard_normal((F * T, sh.n_heads, sh.head_dim)))
        a.cache_commit(raw, raw)
    h, F = 3, 2
    rk, rv, _ = a.ring.recent(h)
    q = f64_to_bf16_bits(g.standard_normal((F * T, sh.n_heads, sh.head_dim)))
    ck = f64_to_bf16_bits(g.standard_normal((F * T, sh.n_heads, sh.head_dim)))
    cv = f64_to_bf16_bits(g.standard_normal((F * T, sh.n_heads, sh.head_dim)))
    ring_o, _ = a.chunk_attention(1, q, ck, cv, hist=h)
    qm = np.concatenate([f64_to_bf16_bits(g.standard_normal((h * T, sh.n_heads, sh.head_dim))), q])
    km = np.concatenate([f64_to_bf16_bits(rk), ck])
    vm = np.concatenate([f64_to_bf16_bits(rv), cv])
    win_o, _ = a.window_attention(1, qm, km, vm, False)
    assert np.allclose(win_o[h * T:], ring_o, rtol=1e-12, atol=1e-12)


def test_recomputed_history_rows_keep_their_frame_times():
    sh, a = _session()
    g = np.random.default_rng(4)
    T = sh.tokens_per_frame
    x = f64_to_bf16_bits(g.standard_normal((5 * T, sh.n_heads, sh.head_dim)))
    for first in (0, 3, 11):
        q, k = a.rope3d_at(first, 5, x, x)
        t, hh, ww = token_positions(5 * T, sh.grid_h, sh.grid_w, first)
        assert t[0] == first and t[-1] == first + 4
        assert np.array_equal(q, f64_to_bf16_bits(rope3d(bf16_bits_to_f64(x), t, hh, ww, 1e4)))
        assert np.array_equal(q, k)
    # the chunk part equals rope3d_qk at the session's frame counter
    a.cache_commit(x[:2 * T], x[:2 * T])
    q_all, _ = a.rope3d_at(a.n_committed - 3, 5, x, x)
    q_chunk, _ = a.rope3d_qk(x[3 * T:], x[3 * T:])
    assert np.array_equal(q_all[3 * T:], q_chunk)
