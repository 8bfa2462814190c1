"""3D (t, h, w) rotary positions, float64 (test infrastructure only).

[H3-page] section 3.2, Iteration 3 item 2: each new latent frame receives its
rotary position once and is written into its ring slot in place. Iteration 4:
cached keys keep the positions they were computed with, so frame tokens take
the absolute latent-frame index of the stream; scores then depend only on
time differences.

The pages name the three axes but not the split of the head dimension nor the
frequency law. Reading used here (plainest standard 3D-RoPE):
  * d = d_t + d_h + d_w with d_h = d_w = 2*floor(d/6), d_t = d - 2*d_h
    (d = 128 -> 44 | 42 | 42; d = 64 -> 24 | 20 | 20);
  * inside axis a, adjacent pairs (x[2i], x[2i+1]), i < d_a/2, rotate by
    theta = p_a * base**(-2i/d_a), p_a the token's position on that axis:
        (x0, x1) -> (x0 cos theta - x1 sin theta, x0 sin theta + x1 cos theta);
  * token n of a chunk lies in frame f = n // T at row h = (n % T) // grid_w,
    column w = n % grid_w; its time position is t_clock0 + n_committed + f.

The angle is the definition written out exactly: p * base**(-2i/d_a) is
formed and reduced modulo 2*pi in 60-digit decimal arithmetic, and only the
reduced angle becomes a float64. A float64 product p * omega would carry an
absolute error of about |p| * 2**-53 rad, 1e-4 rad at p = 2**40; the stream
time grows without bound, so the oracle does not take that shortcut.
"""
import functools
from decimal import ROUND_HALF_EVEN, Decimal, localcontext

import numpy as np

_DIGITS = 60


def axis_split(d: int):
    """(d_t, d_h, d_w) for head dim d."""
    if d % 2:
        raise ValueError("head dim must be even")
    dh = 2 * (d // 6)
    return d - 2 * dh, dh, dh


def inverse_frequencies(d_a: int, base: float) -> np.ndarray:
    """base**(-2i/d_a) for the d_a/2 pairs of one axis (float64)."""
    i = np.arange(d_a // 2, dtype=np.float64)
    return np.power(np.float64(base), -2.0 * i / d_a)


@functools.lru_cache(maxsize=None)
def two_pi() -> Decimal:
    """2*pi to _DIGITS + 10 significant digits from Machin's formula,
    pi = 16 atan(1/5) - 4 atan(1/239), atan(1/x) = sum_k (-1)^k / ((2k+1) x^(2k+1))."""
    with localcontext() as ctx:
        ctx.prec = _DIGITS + 10
        eps = Decimal(10) ** -(_DIGITS + 12)

        def atan_inv(x):
            x2 = Decimal(x) * Decimal(x)
            power = 1 / Decimal(x)          # x^-(2k+1)
            total, k = Decimal(0), 0
            while power > eps:
                term = power / (2 * k + 1)
                total = total - term if k % 2 else total + term
                power /= x2
                k += 1
            return total

        return 2 * (16 * atan_inv(5) - 4 * atan_inv(239))


@functools.lru_cache(maxsize=None)
def omega(i: int, d_a: int, base: float) -> Decimal:
    """base**(-2i/d_a) to _DIGITS significant digits."""
    with localcontext() as ctx:
        ctx.prec = _DIGITS
        return Decimal(float(base)) ** (Decimal(-2 * i) / Decimal(d_a))


@functools.lru_cache(maxsize=1 << 20)
def reduced_angle(p: int, i: int, d_a: int, base: float) -> float:
    """p * base**(-2i/d_a) minus the nearest multiple of 2*pi, in [-pi, pi],
    rounded to float64 only at the end."""
    with localcontext() as ctx:
        ctx.prec = _DIGITS + 10
        theta = Decimal(int(p)) * omega(i, d_a, base)
        k = (theta / two_pi()).to_integral_value(rounding=ROUND_HALF_EVEN)
        return float(theta - k * two_pi())


def rotation_angles(pos, d_a: int, base: float) -> np.ndarray:
    """[L][d_a/2] reduced angles of every position and pair of one axis."""
    pos = np.asarray(pos, dtype=np.int64)
    uniq, inv = np.unique(pos, return_inverse=True)
    table = np.array([[reduced_angle(int(p), i, d_a, float(base)) for i in range(d_a // 2)] for p in uniq],
                     dtype=np.float64).reshape(len(uniq), d_a // 2)
    return table[inv.reshape(-1)]


def token_positions(n_tokens: int, grid_h: int, grid_w: int, t_first: int):
    """(t, h, w) integer positions of the tokens of consecutive frames
    starting at absolute time ``t_first``."""
    T = grid_h * grid_w
    n = np.arange(n_tokens, dtype=np.int64)
    return t_first + n // T, (n % T) // grid_w, n % grid_w


def rope3d(x: np.ndarray, t, h, w, base: float) -> np.ndarray:
    """Rotate x [L][H][d] (float64) by the 3D positions of its L tokens."""
    x = np.asarray(x, dtype=np.float64)
    L, H, d = x.shape
    d_t, d_h, d_w = axis_split(d)
    out = np.empty_like(x)
    start = 0
    for pos, d_a in ((t, d_t), (h, d_h), (w, d_w)):
        if d_a == 0:
            continue
        theta = rotation_angles(np.broadcast_to(np.asarray(pos), (L,)), d_a, base)
        c = np.cos(theta)[:, None, :]        # [L][1][d_a/2], same for every head
        s = np.sin(theta)[:, None, :]
        x0 = x[:, :, start:start + d_a:2]
        x1 = x[:, :, start + 1:start + d_a:2]
        out[:, :, start:start + d_a:2] = x0 * c - x1 * s
        out[:, :, start + 1:start + d_a:2] = x0 * s + x1 * c
        start += d_a
    return out
