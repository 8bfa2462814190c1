"""The streaming decoder's window attention on this library (host-side orchestration).

[H3 page] "Interactive Coding Worlds with Real-time Streaming Diffusion Render",
section 3.2 Iterations 2-4: each latent frame's tokens are cut into windows of
16x16 tokens (shifted by half a window on alternate layers); a window's chunk
tokens attend to the global tokens, the window's cached frames and its own
chunk frames, with positions relative to the window; the cache of each window
is a preallocated ring written in place.

Here every window is one session of the C library (grid = the window's size,
F = chunk frames, W = cached frames), all sessions of a layer share one bank
buffer holding the global tokens' keys and values (rewritten by the caller per
chunk), and a layer's attention is the batched call over its windows, at most
SR_MAX_BATCH windows per launch. Inputs come packed window by window, frame by
frame, row-major inside the window (the variable-length layout: no padding);
``packing_index`` gives the token permutation from whole frames to that layout.
Nothing here computes: the rotary positions, the attention and the cache writes
run in libsr.so.
"""
from __future__ import annotations

import torch

from . import Session, chunk_attention_batch
from ._native import SR_MAX_BATCH, sr_plan_window, sr_window_count


class DecoderWindowLayer:
    def __init__(self, grid_h: int, grid_w: int, n_heads: int, head_dim: int, n_global: int, *,
                 window: int = 16, shifted: bool = False, chunk_frames: int = 2, cache_frames: int = 4,
                 t_clock0: int = 0, device="cuda"):
        self.gh, self.gw, self.H, self.d = grid_h, grid_w, n_heads, head_dim
        self.F, self.C = chunk_frames, cache_frames
        self.device = torch.device(device)
        n = sr_window_count(grid_h, grid_w, window, shifted)
        self.windows = [sr_plan_window(grid_h, grid_w, window, shifted, i) for i in range(n)]
        # the global tokens' K/V: one bank (one step) shared by every window
        self.bank_k = torch.zeros((1, n_global, n_heads, head_dim), dtype=torch.bfloat16, device=self.device)
        self.bank_v = torch.zeros_like(self.bank_k)
        self.sessions = [Session(n_heads, head_dim, w.rows, w.cols, chunk_frames, cache_frames, n_global, 1,
                                 bank=(self.bank_k, self.bank_v), t_clock0=t_clock0, device=self.device)
                         for w in self.windows]
        self.offsets = [0]
        for s in self.sessions:
            self.offsets.append(self.offsets[-1] + s.lq)
        # groups of windows per launch, each a contiguous row range of the packed layout
        self.groups = [range(i, min(i + SR_MAX_BATCH, n)) for i in range(0, n, SR_MAX_BATCH)]

    @property
    def rows(self) -> int:
        return self.offsets[-1]

    def packing_index(self) -> torch.Tensor:
        """Token index into frames flattened as [F][grid_h][grid_w] for every
        packed row (window by window, frame by frame, row-major in the window)."""
        idx = []
        for w in self.windows:
            f = torch.arange(self.F).view(-1, 1, 1)
            r = torch.arange(w.row0, w.row0 + w.rows).view(1, -1, 1)
            c = torch.arange(w.col0, w.col0 + w.cols).view(1, 1, -1)
            idx.append(((f * self.gh + r) * self.gw + c).reshape(-1))
        return torch.cat(idx)

    def _slices(self, t: torch.Tensor, i: int) -> torch.Tensor:
        return t[self.offsets[i]:self.offsets[i + 1]]

    def set_global(self, k: torch.Tensor, v: torch.Tensor) -> None:
        """The chunk's global-token keys and values, [G][H][d] (final, no rotation)."""
        self.bank_k[0].copy_(k)
        self.bank_v[0].copy_(v)

    def rope(self, q: torch.Tensor, k: torch.Tensor) -> None:
        """Rotary positions (relative to each window, absolute frame time) on packed q, k."""
        for i, s in enumerate(self.sessions):
            s.rope3d_qk(self._slices(q, i), self._slices(k, i))

    def attention(self, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out: torch.Tensor | None = None):
        """Every window's chunk rows over global tokens U its cached frames U its chunk."""
        if out is None:
            out = torch.empty_like(q)
        for g in self.groups:
            a, b = self.offsets[g.start], self.offsets[g.stop]
            chunk_attention_batch([self.sessions[i] for i in g], 0, q[a:b], k[a:b], v[a:b], out=out[a:b])
        return out

    def commit(self, k: torch.Tensor, v: torch.Tensor) -> None:
        """Write the chunk's frames into every window's cache ring (K rotated at its frames)."""
        for i, s in enumerate(self.sessions):
            s.cache_commit(self._slices(k, i), self._slices(v, i))

    def error_status(self) -> int:
        return max(abs(s.error_status()) for s in self.sessions)

    def close(self) -> None:
        for s in self.sessions:
            s.close()
