"""The streaming decoder's window attention on this library (host-side orchestration).

[H3 page] "Interactive Coding Worlds with Real-time Streaming Diffusion Render",
section 3.2 Iterations 2-6: each latent frame's tokens are cut into windows of
16x16 tokens (shifted by half a window on alternate layers); a window's chunk
tokens attend to the global tokens, the window's cached frames and its own
chunk frames, with positions relative to the window; the cache of each window
is a preallocated ring written in place; the window gather is fused with the
rotary embedding, and the rotary embedding with the cache write.

Here every window is one session of the C library (grid = the window's size,
F = chunk frames, W = cached frames), and all sessions of a layer share one
bank buffer holding the global tokens' keys and values (rewritten by the
caller per chunk). A layer takes three kinds of launch, each covering every
window (up to SR_MAX_LAYER_WINDOWS, resp. SR_MAX_BATCH for the attention):

* ``gather_rope``: frame-major Q, K, V [F][grid_h][grid_w][H][d] -> the
  window-packed layout (window by window, frame by frame, row-major inside
  the window; no padding), Q and K rotated at window-relative positions;
* ``attention``: the batched attention of every window over its visible set;
* ``commit``: every window's frames of the clean K (rotated) and V into the
  window's ring.

``packing_index`` gives the token permutation from whole frames to the packed
layout (to scatter packed outputs back). Nothing here computes: the gather,
the rotary positions, the attention and the cache writes run in libsr.so.
"""
from __future__ import annotations

import torch

from . import Session, _ptr, _stream, chunk_attention_batch
from ._native import (SR_MAX_BATCH, SR_MAX_LAYER_WINDOWS, sr_layer_commit, sr_layer_rope_gather, sr_plan_window,
                      sr_window_count)


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
        # groups of windows per attention launch, each a contiguous row range of the packed layout
        self.groups = [range(i, min(i + SR_MAX_BATCH, n)) for i in range(0, n, SR_MAX_BATCH)]
        # groups of windows per gather / commit launch
        self.layer_groups = [range(i, min(i + SR_MAX_LAYER_WINDOWS, n)) for i in range(0, n, SR_MAX_LAYER_WINDOWS)]

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

    def _frames(self, name: str, t: torch.Tensor) -> None:
        ok = (t.dtype == torch.bfloat16 and t.device == self.device and t.is_contiguous()
              and t.numel() == self.F * self.gh * self.gw * self.H * self.d)
        if not ok:
            raise ValueError(f"{name}: expected a contiguous bf16 [F][grid_h][grid_w][H][d] tensor on {self.device}")

    def _packed(self, name: str, t: torch.Tensor) -> None:
        if t.dtype != torch.bfloat16 or t.device != self.device or not t.is_contiguous() or \
                tuple(t.shape) != (self.rows, self.H, self.d):
            raise ValueError(f"{name}: expected a contiguous bf16 [{self.rows}][{self.H}][{self.d}] tensor")

    def set_global(self, k: torch.Tensor, v: torch.Tensor) -> None:
        """The chunk's global-token keys and values, [G][H][d] (final, no rotation)."""
        self.bank_k[0].copy_(k)
        self.bank_v[0].copy_(v)

    def gather_rope(self, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor | None = None,
                    out: tuple | None = None):
        """Frame-major q, k (and v) -> packed (q, k, v): q and k rotated at
        window-relative (h, w) and absolute frame time, v copied (None: not
        gathered, returned as None). One launch per SR_MAX_LAYER_WINDOWS windows."""
        for name, t in (("q", q), ("k", k)) + ((("v", v),) if v is not None else ()):
            self._frames(name, t)
        if out is None:
            out = tuple(torch.empty((self.rows, self.H, self.d), dtype=torch.bfloat16, device=self.device)
                        if t is not None else None for t in (q, k, v))
        for name, t in zip(("q_out", "k_out", "v_out"), out):
            if t is not None:
                self._packed(name, t)
        qo, ko, vo = out
        for g in self.layer_groups:
            row = self.offsets[g.start]
            at = lambda t: 0 if t is None else t[row:].data_ptr()
            sr_layer_rope_gather([self.sessions[i].handle for i in g], [self.windows[i] for i in g], self.gh, self.gw,
                                 q.data_ptr(), k.data_ptr(), _ptr(v), at(qo), at(ko), at(vo), _stream(self.device))
        return qo, ko, vo

    def attention(self, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out: torch.Tensor | None = None):
        """Every window's chunk rows (packed) over global tokens U its cached frames U its chunk."""
        if out is None:
            out = torch.empty_like(q)
        for g in self.groups:
            a, b = self.offsets[g.start], self.offsets[g.stop]
            chunk_attention_batch([self.sessions[i] for i in g], 0, q[a:b], k[a:b], v[a:b], out=out[a:b])
        return out

    def commit(self, k: torch.Tensor, v: torch.Tensor) -> None:
        """Write the chunk's frames (frame-major clean K and V) into every window's
        cache ring, K rotated at its frames. One launch per SR_MAX_LAYER_WINDOWS windows."""
        self._frames("k", k)
        self._frames("v", v)
        for g in self.layer_groups:
            sr_layer_commit([self.sessions[i].handle for i in g], [self.windows[i] for i in g], self.gh, self.gw,
                            k.data_ptr(), v.data_ptr(), _stream(self.device))

    def error_status(self) -> int:
        return max(abs(s.error_status()) for s in self.sessions)

    def close(self) -> None:
        for s in self.sessions:
            s.close()
