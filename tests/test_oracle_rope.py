"""Pins for the oracle's 3D rotary positions (CPU only).

The oracle rotates adjacent pairs inside each of the t, h and w sub-vectors.
These tests tie it to facts that do not depend on its code: the identity at
position 0, norm preservation, the group law of rotations, the relative-
position property that makes scores depend only on position differences
(the Iteration 4 fix of the H3 project page, section 3.2), the complex-number
form of a rotation, and a 2-D rotation matrix written out by hand.
"""
import math

import numpy as np
import pytest

from oracle import axis_split, inverse_frequencies, rope3d, token_positions


def _x(L=5, H=3, d=12, seed=0):
    return np.random.default_rng(seed).standard_normal((L, H, d))


def test_axis_split_reading():
    assert axis_split(128) == (44, 42, 42)
    assert axis_split(64) == (24, 20, 20)
    assert axis_split(6) == (2, 2, 2)
    assert axis_split(12) == (4, 4, 4)
    with pytest.raises(ValueError):
        axis_split(7)


def test_inverse_frequencies_closed_form():
    f = inverse_frequencies(4, 10000.0)
    assert f[0] == 1.0
    assert math.isclose(f[1], 0.01, rel_tol=1e-15)       # 10000 ** (-2/4)
    f44 = inverse_frequencies(44, 10000.0)
    assert len(f44) == 22
    assert math.isclose(f44[11], 10000.0 ** (-0.5), rel_tol=1e-14)


def test_identity_at_origin():
    x = _x()
    z = np.zeros(x.shape[0], int)
    assert np.array_equal(rope3d(x, z, z, z, 10000.0), x)


def test_pair_norms_preserved():
    x = _x(d=128)
    t, h, w = token_positions(5, 2, 3, t_first=17)
    y = rope3d(x, t, h, w, 10000.0)
    nx = x[..., 0::2] ** 2 + x[..., 1::2] ** 2
    ny = y[..., 0::2] ** 2 + y[..., 1::2] ** 2
    assert np.allclose(nx, ny, rtol=1e-13, atol=1e-13)


def test_composition_is_addition_of_positions():
    x = _x(d=64)
    p1 = (np.array([3, 1, 0, 9, 2]), np.array([0, 4, 2, 1, 1]), np.array([5, 0, 7, 3, 1]))
    p2 = (np.array([1, 2, 3, 4, 5]), np.array([6, 0, 1, 2, 3]), np.array([0, 9, 2, 4, 8]))
    a = rope3d(rope3d(x, *p1, 10000.0), *p2, 10000.0)
    b = rope3d(x, *(u + v for u, v in zip(p1, p2)), 10000.0)
    assert np.allclose(a, b, rtol=0, atol=1e-12)


def test_scores_depend_only_on_position_difference():
    g = np.random.default_rng(3)
    q = g.standard_normal((1, 2, 128))
    k = g.standard_normal((1, 2, 128))
    base = 10000.0
    for dt, dh, dw in [(100, 0, 0), (1000, 3, 7), (0, 11, 2)]:
        pq = (np.array([4]), np.array([2]), np.array([9]))
        pk = (np.array([1]), np.array([5]), np.array([3]))
        s0 = np.einsum("lhd,lhd->h", rope3d(q, *pq, base), rope3d(k, *pk, base))
        sh = (np.array([4 + dt]), np.array([2 + dh]), np.array([9 + dw]))
        kh = (np.array([1 + dt]), np.array([5 + dh]), np.array([3 + dw]))
        s1 = np.einsum("lhd,lhd->h", rope3d(q, *sh, base), rope3d(k, *kh, base))
        assert np.allclose(s0, s1, rtol=0, atol=1e-10)


def test_matches_complex_multiplication():
    # Each pair (x0, x1) as x0 + i x1 is multiplied by exp(i * p * base^(-2j/d_a)).
    x = _x(L=4, H=2, d=128, seed=5)
    t, h, w = token_positions(4, 2, 2, t_first=1000)
    y = rope3d(x, t, h, w, 500.0)
    want = np.empty_like(x)
    off = 0
    for pos, d_a in zip((t, h, w), (44, 42, 42)):
        z = x[:, :, off:off + d_a:2] + 1j * x[:, :, off + 1:off + d_a:2]
        j = np.arange(d_a // 2)
        rot = np.exp(1j * pos[:, None] * (500.0 ** (-2.0 * j / d_a)))[:, None, :]
        zr = z * rot
        want[:, :, off:off + d_a:2] = zr.real
        want[:, :, off + 1:off + d_a:2] = zr.imag
        off += d_a
    assert np.allclose(y, want, rtol=0, atol=1e-11)


def test_two_dim_axis_is_a_plain_rotation_matrix():
    # d = 6: each axis holds one pair with frequency 1, so the t pair turns by
    # exactly t radians, the h pair by h, the w pair by w.
    x = np.array([[[1.0, 2.0, -0.5, 0.25, 3.0, -1.0]]])
    t, h, w = np.array([2]), np.array([0]), np.array([1])
    y = rope3d(x, t, h, w, 10000.0)[0, 0]
    def rot(a, v):
        return np.array([[math.cos(a), -math.sin(a)], [math.sin(a), math.cos(a)]]) @ v
    assert np.allclose(y[0:2], rot(2.0, x[0, 0, 0:2]), atol=1e-15)
    assert np.allclose(y[2:4], x[0, 0, 2:4], atol=0)
    assert np.allclose(y[4:6], rot(1.0, x[0, 0, 4:6]), atol=1e-15)


def test_token_positions_frame_row_column():
    # a 2x3 grid, two frames starting at absolute time 7
    t, h, w = token_positions(12, 2, 3, t_first=7)
    assert t.tolist() == [7] * 6 + [8] * 6
    assert h.tolist() == [0, 0, 0, 1, 1, 1] * 2
    assert w.tolist() == [0, 1, 2] * 4


# --- positions far from the origin: the stream time grows without bound ---

def test_two_pi_and_frequencies_closed_forms():
    from decimal import Decimal, localcontext
    from oracle.rope import omega, two_pi
    assert float(two_pi() / 2) == math.pi
    assert abs(float(two_pi()) - 2 * math.pi) == 0.0
    # 10000 ** (-2*11/44) = 10000 ** -0.5 = 1/100 exactly; 10000 ** (-2/4) likewise
    assert abs(omega(11, 44, 10000.0) - Decimal("0.01")) < Decimal(10) ** -55
    assert abs(omega(1, 4, 10000.0) - Decimal("0.01")) < Decimal(10) ** -55
    # frequencies of one axis form a geometric sequence: w_i * w_j = w_0 * w_(i+j)
    with localcontext() as ctx:
        ctx.prec = 80
        assert abs(omega(3, 42, 10000.0) * omega(5, 42, 10000.0) - omega(8, 42, 10000.0)) < Decimal(10) ** -55
    assert omega(0, 42, 10000.0) == 1


@pytest.mark.parametrize("t", [2 ** 24 + 3, 2 ** 30, 2 ** 33, 2 ** 40, -(2 ** 40) + 7, 123456789012])
def test_huge_time_turns_a_frequency_one_pair_by_exactly_t_radians(t):
    # d = 6: the t axis holds a single pair with frequency base**0 = 1, so its
    # angle is t radians; math.cos/sin of the float64 t (exact below 2**53)
    # reduce the argument exactly.
    x = np.array([[[0.75, -1.25, 0.0, 0.0, 0.0, 0.0]]])
    y = rope3d(x, np.array([t]), np.array([0]), np.array([0]), 10000.0)[0, 0]
    c, s = math.cos(float(t)), math.sin(float(t))
    assert np.allclose(y[0:2], [0.75 * c + 1.25 * s, 0.75 * s - 1.25 * c], rtol=0, atol=4e-16)


def test_composition_holds_at_large_positions():
    # R(p1) R(p2) = R(p1 + p2) for every pair of a d = 128 head. A float64
    # product p * omega would break this by ~|p| * 2**-53 rad (6e-5 at 2**39).
    x = _x(L=3, H=2, d=128, seed=9)
    p1 = (np.array([2 ** 39 + 5, 2 ** 33, 2 ** 24 + 1]), np.array([0, 7, 3]), np.array([1, 0, 9]))
    p2 = (np.array([2 ** 38 - 3, 12345, 2 ** 31]), np.array([4, 0, 1]), np.array([2, 6, 0]))
    a = rope3d(rope3d(x, *p1, 10000.0), *p2, 10000.0)
    b = rope3d(x, *(u + v for u, v in zip(p1, p2)), 10000.0)
    assert np.allclose(a, b, rtol=0, atol=1e-13)


def test_scores_depend_only_on_position_difference_at_large_offsets():
    g = np.random.default_rng(4)
    q = g.standard_normal((1, 2, 128))
    k = g.standard_normal((1, 2, 128))
    pq = (np.array([4]), np.array([2]), np.array([9]))
    pk = (np.array([1]), np.array([5]), np.array([3]))
    s0 = np.einsum("lhd,lhd->h", rope3d(q, *pq, 10000.0), rope3d(k, *pk, 10000.0))
    for dt in (2 ** 24 + 3, 2 ** 35 + 17, 2 ** 40):
        sh = (pq[0] + dt, pq[1], pq[2])
        kh = (pk[0] + dt, pk[1], pk[2])
        s1 = np.einsum("lhd,lhd->h", rope3d(q, *sh, 10000.0), rope3d(k, *kh, 10000.0))
        assert np.allclose(s0, s1, rtol=0, atol=1e-12)
