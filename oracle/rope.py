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
"""
import numpy as np


def axis_split(d: int):
    """(d_t, d_h, d_w) for head dim d."""
    if d % 2:
        raise ValueError("head dim must be even")
    dh = 2 * (d // 6)
    return d - 2 * dh, dh, dh


def inverse_frequencies(d_a: int, base: float) -> np.ndarray:
    """base**(-2i/d_a) for the d_a/2 pairs of one axis."""
    i = np.arange(d_a // 2, dtype=np.float64)
    return np.power(np.float64(base), -2.0 * i / d_a)


def token_positions(n_tokens: int, grid_h: int, grid_w: int, t_first: int):
    """(t, h, w) integer positions of the tokens of consecutive frames
    starting at absolute time ``t_first``."""
    T = grid_h * grid_w
    n = np.arange(n_tokens)
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
        theta = np.asarray(pos, dtype=np.float64)[:, None] * inverse_frequencies(d_a, base)[None, :]
        c = np.cos(theta)[:, None, :]        # [L][1][d_a/2], same for every head
        s = np.sin(theta)[:, None, :]
        x0 = x[:, :, start:start + d_a:2]
        x1 = x[:, :, start + 1:start + d_a:2]
        out[:, :, start:start + d_a:2] = x0 * c - x1 * s
        out[:, :, start + 1:start + d_a:2] = x0 * s + x1 * c
        start += d_a
    return out
