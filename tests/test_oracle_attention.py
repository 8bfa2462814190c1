"""Pins for the oracle's attention (CPU only).

Brute force with exact summation on tiny inputs, a library routine
(torch's scaled_dot_product_attention in float64), and the closed forms and
invariants of softmax attention: probabilities sum to one, permuting keys
with their values changes nothing, equal keys give the mean of V, one key
gives its value, a common shift of every key shifts every logit of a row
equally, outputs are affine in V, and a dominant key wins.
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention, attention_rows


def _qkv(Lq=7, Lk=11, H=3, d=8, seed=0, scale_q=1.0):
    g = np.random.default_rng(seed)
    return (g.standard_normal((Lq, H, d)) * scale_q, g.standard_normal((Lk, H, d)),
            g.standard_normal((Lk, H, d)))


def test_brute_force_exact_sums():
    q, k, v = _qkv(Lq=3, Lk=5, H=2, d=4, seed=1)
    scale = 0.37
    o, lse = attention(q, k, v, scale)
    for h in range(2):
        for i in range(3):
            s = [scale * math.fsum(q[i, h, c] * k[j, h, c] for c in range(4)) for j in range(5)]
            m = max(s)
            e = [math.exp(x - m) for x in s]
            z = math.fsum(e)
            for c in range(4):
                want = math.fsum(e[j] * v[j, h, c] for j in range(5)) / z
                assert abs(o[i, h, c] - want) <= 1e-12
            assert abs(lse[h, i] - (m + math.log(z))) <= 1e-12


def test_matches_torch_sdpa_float64():
    q, k, v = _qkv(Lq=33, Lk=70, H=4, d=16, seed=2, scale_q=3.0)
    scale = 1.0 / math.sqrt(16)
    o, lse = attention(q, k, v, scale, q_block=8)
    tq, tk, tv = (torch.from_numpy(a).permute(1, 0, 2) for a in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=scale)
    assert np.allclose(o, ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)
    s = torch.einsum("hid,hjd->hij", tq, tk) * scale
    assert np.allclose(lse, torch.logsumexp(s, dim=-1).numpy(), rtol=0, atol=1e-12)


def test_probabilities_sum_to_one_and_are_nonnegative():
    # With V the identity (one value column per key), O is the probability matrix.
    q, k, _ = _qkv(Lq=9, Lk=13, H=2, d=8, seed=3, scale_q=4.0)
    v = np.broadcast_to(np.eye(13)[:, None, :], (13, 2, 13)).copy()
    p, _ = attention(q, k, v, 0.5)
    assert np.all(p >= 0)
    assert np.allclose(p.sum(axis=-1), 1.0, rtol=0, atol=1e-14)


def test_key_permutation_invariance():
    q, k, v = _qkv(seed=4)
    perm = np.random.default_rng(9).permutation(k.shape[0])
    a, la = attention(q, k, v, 0.3)
    b, lb = attention(q, k[perm], v[perm], 0.3)
    assert np.allclose(a, b, rtol=0, atol=1e-14)
    assert np.allclose(la, lb, rtol=0, atol=1e-13)


def test_equal_keys_give_mean_of_values():
    q, _, v = _qkv(Lk=17, seed=5)
    k = np.broadcast_to(np.random.default_rng(6).standard_normal((1, 3, 8)), (17, 3, 8))
    o, lse = attention(q, k, v, 0.9)
    assert np.allclose(o, np.broadcast_to(v.mean(axis=0), o.shape), rtol=0, atol=1e-14)
    s = 0.9 * np.einsum("ihd,hd->hi", q, k[0])
    assert np.allclose(lse, s + math.log(17), rtol=0, atol=1e-13)


def test_single_key_returns_its_value():
    q, k, v = _qkv(Lk=1, seed=6)
    o, _ = attention(q, k, v, 1.0)
    assert np.array_equal(o, np.broadcast_to(v[0], o.shape))


def test_common_key_shift_is_invisible():
    q, k, v = _qkv(seed=7)
    c = np.random.default_rng(8).standard_normal((1, 3, 8)) * 5
    a, _ = attention(q, k, v, 0.4)
    b, _ = attention(q, k + c, v, 0.4)
    assert np.allclose(a, b, rtol=0, atol=1e-12)


def test_affine_in_values():
    q, k, v = _qkv(seed=9)
    A = np.random.default_rng(10).standard_normal((8, 8))
    bvec = np.random.default_rng(11).standard_normal(8)
    a, _ = attention(q, k, v, 0.4)
    b, _ = attention(q, k, v @ A + bvec, 0.4)
    assert np.allclose(b, a @ A + bvec, rtol=0, atol=1e-12)


def test_dominant_key_wins():
    q, k, v = _qkv(Lq=4, Lk=50, H=1, d=16, seed=12)
    k[23] = q[2] * 40.0
    o, _ = attention(q, k, v, 1.0)
    assert np.allclose(o[2], v[23], rtol=0, atol=1e-10)


def test_query_blocking_does_not_change_result():
    q, k, v = _qkv(Lq=50, seed=13)
    a, la = attention(q, k, v, 0.2, q_block=1024)
    b, lb = attention(q, k, v, 0.2, q_block=7)
    # BLAS may sum in a different order for another block shape
    assert np.allclose(a, b, rtol=0, atol=1e-14) and np.allclose(la, lb, rtol=0, atol=1e-14)


def test_sampled_rows_agree_with_full():
    q, k, v = _qkv(Lq=20, H=5, seed=14)
    o, lse = attention(q, k, v, 0.3)
    rows, heads = [0, 7, 19], [4, 1]
    os_, ls = attention_rows(q, k, v, 0.3, rows, heads)
    assert np.allclose(os_, o[rows][:, heads], rtol=0, atol=1e-15)
    assert np.allclose(ls, lse[heads][:, rows], rtol=0, atol=1e-15)
