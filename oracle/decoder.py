"""Window attention of the pages' streaming decoder, one layer, float64
(test infrastructure only).

[H3-page] "Interactive Coding Worlds with Real-time Streaming Diffusion
Render", section 3.2 Iteration 2 ("Time", "Space"), Iteration 3 items 2 and 4,
Iteration 4:
  * a latent frame of grid_h x grid_w tokens is cut into windows of
    window x window tokens; every other layer shifts the cuts by half a window,
    so the windows at the frame's edges are smaller; spatial positions are
    relative to the window;
  * a chunk is two latent frames; each window's chunk tokens attend to the
    window's tokens of the chunk itself and of the cached previous frames (four
    in the pages), never to a later frame; cache slots still empty at stream
    start are left out;
  * the global tokens (four register tokens and one class token) attend with
    the frame: here every window's queries also see their keys and values,
    which the caller supplies final (no rotary position is applied to them);
  * cached keys keep the rotary position of the absolute latent frame they were
    stored with.
The layer is computed from whole frames: cut into windows, gather each
window's tokens, apply the definition, scatter the rows back.
"""
import math

import numpy as np

from .attention import attention
from .bf16 import bf16_bits_to_f64, f64_to_bf16_bits
from .rope import rope3d


def window_cuts(n: int, window: int, shifted: bool):
    """Cut positions of one axis: 0, then every window tokens starting at
    window (plain) or at window / 2 (shifted), then n."""
    first = window // 2 if shifted else window
    cuts = [0] + list(range(first, n, window)) + [n]
    return sorted(set(cuts))


def window_partition(grid_h: int, grid_w: int, window: int, shifted: bool):
    """Windows (row0, col0, rows, cols), row by row."""
    rc, cc = window_cuts(grid_h, window, shifted), window_cuts(grid_w, window, shifted)
    return [(r0, c0, r1 - r0, c1 - c0) for r0, r1 in zip(rc, rc[1:]) for c0, c1 in zip(cc, cc[1:])]


def _window_positions(frames, rows, cols, t0):
    """(t, h, w) of a window's tokens, frame by frame, row-major inside the window."""
    f, r, c = np.meshgrid(np.arange(frames), np.arange(rows), np.arange(cols), indexing="ij")
    return (t0 + f).ravel(), r.ravel(), c.ravel()


class DecoderLayerOracle:
    """One decoder layer's window attention over a stream of chunks."""

    def __init__(self, grid_h, grid_w, window, shifted, n_heads, head_dim, cache_frames=4,
                 t_clock0=0, rope_base=1e4, scale=None):
        self.gh, self.gw, self.window, self.shifted = grid_h, grid_w, window, shifted
        self.H, self.d = n_heads, head_dim
        self.C = cache_frames
        self.t0 = t_clock0
        self.base = rope_base
        self.scale = scale if scale else 1.0 / math.sqrt(head_dim)
        self.windows = window_partition(grid_h, grid_w, window, shifted)
        self.n = 0                      # frames committed
        self.cache = []                 # (frame g, rotated K [gh][gw][H][d], V [gh][gw][H][d]), oldest first

    def _rotate(self, x, first_frame):
        """x: [F][gh][gw][H][d] float64; each window's tokens rotated with
        window-relative (h, w) and absolute time first_frame + f."""
        F = x.shape[0]
        out = np.empty_like(x)
        for (r0, c0, nr, nc) in self.windows:
            blk = x[:, r0:r0 + nr, c0:c0 + nc].reshape(F * nr * nc, self.H, self.d)
            t, h, w = _window_positions(F, nr, nc, self.t0 + first_frame)
            out[:, r0:r0 + nr, c0:c0 + nc] = rope3d(blk, t, h, w, self.base).reshape(F, nr, nc, self.H, self.d)
        return out

    def step(self, q_bits, k_bits, v_bits, gk_bits, gv_bits):
        """q, k, v: [F][gh][gw][H][d] bf16 bits of the chunk (not rotated);
        gk, gv: [G][H][d] global-token keys and values. Returns o [F][gh][gw][H][d]
        (float64): every window's chunk rows over global tokens U the window's
        cached frames U its chunk frames."""
        F = q_bits.shape[0]
        q = bf16_bits_to_f64(f64_to_bf16_bits(self._rotate(bf16_bits_to_f64(q_bits), self.n)))
        k = bf16_bits_to_f64(f64_to_bf16_bits(self._rotate(bf16_bits_to_f64(k_bits), self.n)))
        v = bf16_bits_to_f64(v_bits)
        gk, gv = bf16_bits_to_f64(gk_bits), bf16_bits_to_f64(gv_bits)
        o = np.empty_like(q)
        for (r0, c0, nr, nc) in self.windows:
            sl = (slice(None), slice(r0, r0 + nr), slice(c0, c0 + nc))
            qw = q[sl].reshape(-1, self.H, self.d)
            kc = [ck[r0:r0 + nr, c0:c0 + nc].reshape(-1, self.H, self.d) for _, ck, _ in self.cache]
            vc = [cv[r0:r0 + nr, c0:c0 + nc].reshape(-1, self.H, self.d) for _, _, cv in self.cache]
            K = np.concatenate([gk] + kc + [k[sl].reshape(-1, self.H, self.d)])
            V = np.concatenate([gv] + vc + [v[sl].reshape(-1, self.H, self.d)])
            ow, _ = attention(qw, K, V, self.scale)
            o[sl] = ow.reshape(F, nr, nc, self.H, self.d)
        return o

    def commit(self, k_bits, v_bits):
        """Store the chunk's frames in the cache: K rotated per window at its
        absolute frames, K and V rounded to bf16; keep the last C frames."""
        F = k_bits.shape[0]
        k = bf16_bits_to_f64(f64_to_bf16_bits(self._rotate(bf16_bits_to_f64(k_bits), self.n)))
        v = bf16_bits_to_f64(v_bits)
        for f in range(F):
            self.cache.append((self.n + f, k[f], v[f]))
        self.cache = self.cache[-self.C:] if self.C > 0 else []
        self.n += F
