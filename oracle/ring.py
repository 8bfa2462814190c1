"""Rolling history ring of W latent frames (test infrastructure only).

[H3-page] "Interactive Coding Worlds with Real-time Streaming Diffusion
Render", section 3.2 Iteration 3 item 2: the cache is a ring allocated up
front, and a new latent frame overwrites one fixed slot of it rather than
being appended. Section 3.3 "Persistent KV layout": the changing part of the
cache is modified where it lives.

Frame g (absolute index in the stream) goes to slot g mod W; writing it
evicts whatever frame the slot held (the frame g - W). ``slot_frame[s]`` is
the absolute frame in slot s, -1 while the slot is still empty.
"""
import numpy as np


class RingCache:
    def __init__(self, window_frames: int, tokens_per_frame: int, n_heads: int, head_dim: int):
        self.W = window_frames
        self.T = tokens_per_frame
        self.k = np.full((window_frames * tokens_per_frame, n_heads, head_dim), np.nan)
        self.v = np.full_like(self.k, np.nan)
        self.slot_frame = np.full((window_frames,), -1, np.int64)
        self.n = 0                                   # frames committed so far

    def slot_of(self, g: int) -> int:
        return g % self.W

    def write_frame(self, g: int, k_frame: np.ndarray, v_frame: np.ndarray):
        """Store frame g ([T][H][d] each, already in its stored precision)."""
        s = self.slot_of(g)
        self.k[s * self.T:(s + 1) * self.T] = k_frame
        self.v[s * self.T:(s + 1) * self.T] = v_frame
        self.slot_frame[s] = g

    def commit(self, k: np.ndarray, v: np.ndarray, frames: int):
        """Append ``frames`` consecutive frames (k, v: [frames*T][H][d]) in
        stream order. When ``frames`` exceeds W the chunk's own later frames
        evict its earlier ones, and only its last W frames stay."""
        for f in range(frames):
            g = self.n + f
            self.write_frame(g, k[f * self.T:(f + 1) * self.T], v[f * self.T:(f + 1) * self.T])
        self.n += frames

    def visible(self):
        """K and V of the occupied slots, in slot order (any order is equally
        valid: softmax attention is a function of the key set)."""
        occupied = [s for s in range(self.W) if self.slot_frame[s] >= 0]
        if not occupied:
            shape = (0,) + self.k.shape[1:]
            return np.empty(shape), np.empty(shape), occupied
        idx = np.concatenate([np.arange(s * self.T, (s + 1) * self.T) for s in occupied])
        return self.k[idx], self.v[idx], occupied

    def recent(self, h: int):
        """K and V of the last h committed frames (frames n-h .. n-1), in
        stream order: the recent history of the next chunk."""
        if h < 0 or h > min(self.n, self.W):
            raise ValueError("history longer than what the ring holds")
        frames = list(range(self.n - h, self.n))
        for g in frames:
            if self.slot_frame[self.slot_of(g)] != g:
                raise ValueError(f"frame {g} is no longer in the ring")
        if not frames:
            shape = (0,) + self.k.shape[1:]
            return np.empty(shape), np.empty(shape), frames
        idx = np.concatenate([np.arange(self.slot_of(g) * self.T, (self.slot_of(g) + 1) * self.T) for g in frames])
        return self.k[idx], self.v[idx], frames
