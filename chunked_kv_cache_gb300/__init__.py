"""GB300-native streaming chunk attention with a 3D-RoPE ring-buffer KV cache.

The compute lives in libsr.so (hand-written CUDA for sm_103a, C ABI in
include/sr.h). This package is the thin Python side: the ctypes binding with
the C names (``_native``) and ``Session``, which allocates a session's
persistent device buffers with torch and marshals tensors into those calls.
torch provides device memory and streams only; nothing here computes.
"""
from __future__ import annotations

import torch

from . import _native
from ._native import (SrConfig, SrBuffers, SrError, sr_session_init, sr_session_restore, sr_session_frames,
                      sr_rope3d_qk, sr_chunk_attention, sr_cache_commit, sr_session_free,
                      sr_chunk_attention_batch, sr_device_error_status, sr_debug_wait_timeout,
                      sr_workspace_bytes, sr_plan_chunk, sr_rope3d_qk_frames, sr_chunk_attention_frames,
                      sr_cache_commit_frames, SrChunkPlan, sr_window_attention, sr_rope3d_qk_at,
                      sr_rope3d_qk_dev, sr_chunk_attention_dev, sr_cache_commit_dev, SR_MAX_BATCH)

__all__ = [
    "Session", "chunk_attention_batch", "SrConfig", "SrBuffers", "SrError",
    "sr_session_init", "sr_session_restore", "sr_session_frames", "sr_rope3d_qk", "sr_chunk_attention",
    "sr_cache_commit", "sr_session_free", "sr_chunk_attention_batch", "sr_device_error_status",
    "sr_debug_wait_timeout", "sr_workspace_bytes", "sr_plan_chunk", "sr_rope3d_qk_frames",
    "sr_chunk_attention_frames", "sr_cache_commit_frames", "SrChunkPlan", "plan_chunk",
    "sr_window_attention", "sr_rope3d_qk_at", "sr_rope3d_qk_dev", "sr_chunk_attention_dev",
    "sr_cache_commit_dev",
]

_BF16 = torch.bfloat16


def _ptr(t: torch.Tensor | None) -> int:
    return 0 if t is None or t.numel() == 0 else t.data_ptr()


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _check_tensor(name: str, t: torch.Tensor, shape, device, dtype=_BF16) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_contiguous() or t.device != device:
        raise ValueError(f"{name}: expected contiguous {dtype} {tuple(shape)} on {device}, "
                         f"got {t.dtype} {tuple(t.shape)} on {t.device} (contiguous={t.is_contiguous()})")


class Session:
    """One streaming session and its caller-owned device buffers.

    Buffers: per-step sink banks [n_steps][S][H][d], ring K/V [W*T][H][d],
    slot table [W] int32 and an error word, all bf16 unless stated, all
    allocated here with torch and handed to the library by pointer.
    """

    def __init__(self, n_heads: int, head_dim: int, grid_h: int, grid_w: int, chunk_frames: int,
                 window_frames: int, n_sink: int, n_steps: int = 2, *, sink_k: torch.Tensor | None = None,
                 sink_v: torch.Tensor | None = None, t_clock0: int = 0, rope_base: float = 10000.0,
                 softmax_scale: float = 0.0, wait_timeout_ns: int = 0, tail_split: int = 0,
                 workspace: bool = True, device_state: bool = False, bank=None, device="cuda"):
        self.device = torch.device(device)
        if self.device.type == "cuda" and self.device.index is None:
            self.device = torch.device("cuda", torch.cuda.current_device())
        self.H, self.d = n_heads, head_dim
        self.T = grid_h * grid_w
        self.F, self.W, self.S, self.n_steps = chunk_frames, window_frames, n_sink, n_steps
        self.lq = chunk_frames * self.T
        dev = self.device
        if bank is not None:
            # an external bank, possibly shared by several sessions (the decoder's
            # windows share the global tokens); used in place, not copied
            if sink_k is not None or sink_v is not None:
                raise ValueError("give bank or sink_k/sink_v, not both")
            self.sink_k, self.sink_v = bank
            for name, t in (("bank k", self.sink_k), ("bank v", self.sink_v)):
                _check_tensor(name, t, (n_steps, n_sink, n_heads, head_dim), dev)
        else:
            self.sink_k = torch.empty((n_steps, n_sink, n_heads, head_dim), dtype=_BF16, device=dev)
            self.sink_v = torch.empty_like(self.sink_k)
        self.ring_k = torch.empty((window_frames * self.T, n_heads, head_dim), dtype=_BF16, device=dev)
        self.ring_v = torch.empty_like(self.ring_k)
        self.slot_frame = torch.empty((max(window_frames, 1),), dtype=torch.int32, device=dev)
        self.err_word = torch.zeros((1,), dtype=torch.int32, device=dev)
        if (sink_k is None) != (sink_v is None):
            raise ValueError("give both sink_k and sink_v, or neither")
        if sink_k is not None:
            _check_tensor("sink_k", sink_k, self.sink_k.shape, dev)
            _check_tensor("sink_v", sink_v, self.sink_v.shape, dev)
        self.cfg = SrConfig(n_heads, head_dim, grid_h, grid_w, chunk_frames, window_frames, n_sink, n_steps,
                            t_clock0, rope_base, softmax_scale, wait_timeout_ns, tail_split)
        # scratch for key-split last blocks (256-byte aligned: torch's allocator aligns to 512)
        self.workspace = None
        if workspace:
            nbytes = sr_workspace_bytes(self.cfg)
            self.workspace = torch.empty((nbytes,), dtype=torch.uint8, device=dev)
        # device-resident frame counter for the *_dev calls (CUDA-graph capture)
        self.frame_counter = torch.zeros((1,), dtype=torch.int64, device=dev) if device_state else None
        self.bufs = SrBuffers(_ptr(self.sink_k), _ptr(self.sink_v), _ptr(self.ring_k), _ptr(self.ring_v),
                              self.slot_frame.data_ptr(), self.err_word.data_ptr(), _ptr(self.workspace),
                              _ptr(self.frame_counter))
        self.handle = None
        with torch.cuda.device(dev):
            self.handle = sr_session_init(self.cfg, self.bufs, _ptr(sink_k), _ptr(sink_v), _stream(dev))

    # ---------------------------------------------------------------- state
    @property
    def frames(self) -> int:
        return sr_session_frames(self.handle)

    def restore(self, n_committed: int) -> None:
        sr_session_restore(self.handle, n_committed)

    def error_status(self) -> int:
        """Synchronises the stream and maps the device error word to a status."""
        return sr_device_error_status(int(self.err_word.item()))

    def _chunk(self, name: str, t: torch.Tensor, frames: int | None = None) -> None:
        rows = self.lq if frames is None else frames * self.T
        _check_tensor(name, t, (rows, self.H, self.d), self.device)

    # ---------------------------------------------------------------- calls
    # frames=None: the configured chunk length and the plain C calls; an int:
    # a chunk of that many frames through the *_frames calls (the unit rhythm).
    def rope3d_qk(self, q: torch.Tensor | None, k: torch.Tensor | None, frames: int | None = None) -> None:
        for name, t in (("q", q), ("k", k)):
            if t is not None:
                self._chunk(name, t, frames)
        if frames is None:
            sr_rope3d_qk(self.handle, _ptr(q), _ptr(k), _stream(self.device))
        else:
            sr_rope3d_qk_frames(self.handle, frames, _ptr(q), _ptr(k), _stream(self.device))

    def chunk_attention(self, step: int, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                        out: torch.Tensor | None = None, lse: torch.Tensor | bool | None = None,
                        frames: int | None = None, hist: int | None = None):
        """hist: visible recent history in frames (None: every occupied slot)."""
        for name, t in (("q", q), ("k", k), ("v", v)):
            self._chunk(name, t, frames)
        if out is None:
            out = torch.empty_like(q)
        self._chunk("out", out, frames)
        rows = q.shape[0]
        if lse is True:
            lse = torch.empty((self.H, rows), dtype=torch.float32, device=self.device)
        if isinstance(lse, torch.Tensor):
            _check_tensor("lse", lse, (self.H, rows), self.device, torch.float32)
        else:
            lse = None
        if frames is None and hist is None:
            sr_chunk_attention(self.handle, step, q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                               _ptr(lse), _stream(self.device))
        else:
            sr_chunk_attention_frames(self.handle, step, self.F if frames is None else frames,
                                      -1 if hist is None else hist, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                      out.data_ptr(), _ptr(lse), _stream(self.device))
        return (out, lse) if lse is not None else out

    def cache_commit(self, k: torch.Tensor, v: torch.Tensor, frames: int | None = None) -> None:
        self._chunk("k", k, frames)
        self._chunk("v", v, frames)
        if frames is None:
            sr_cache_commit(self.handle, k.data_ptr(), v.data_ptr(), _stream(self.device))
        else:
            sr_cache_commit_frames(self.handle, frames, k.data_ptr(), v.data_ptr(), _stream(self.device))

    # ------------------------------------------------ device-resident chunk state
    # The *_dev calls read the committed-frame count from self.frame_counter when
    # the kernels run (Session(device_state=True)); a captured sequence of them
    # serves every chunk of its length.
    def rope3d_qk_dev(self, q: torch.Tensor | None, k: torch.Tensor | None, frames: int) -> None:
        for name, t in (("q", q), ("k", k)):
            if t is not None:
                self._chunk(name, t, frames)
        sr_rope3d_qk_dev(self.handle, frames, _ptr(q), _ptr(k), _stream(self.device))

    def chunk_attention_dev(self, step: int, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, frames: int,
                            hist: int = -1, out: torch.Tensor | None = None, lse: torch.Tensor | None = None):
        for name, t in (("q", q), ("k", k), ("v", v)):
            self._chunk(name, t, frames)
        if out is None:
            out = torch.empty_like(q)
        self._chunk("out", out, frames)
        if lse is not None:
            _check_tensor("lse", lse, (self.H, q.shape[0]), self.device, torch.float32)
        sr_chunk_attention_dev(self.handle, step, frames, hist, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                               out.data_ptr(), _ptr(lse), _stream(self.device))
        return out

    def cache_commit_dev(self, k: torch.Tensor, v: torch.Tensor, frames: int) -> None:
        self._chunk("k", k, frames)
        self._chunk("v", v, frames)
        sr_cache_commit_dev(self.handle, frames, k.data_ptr(), v.data_ptr(), _stream(self.device))

    # ------------------------------------------------ the page-faithful window
    def rope3d_at(self, first_frame: int, frames: int, q: torch.Tensor | None, k: torch.Tensor | None) -> None:
        """RoPE on rows of `frames` frames starting at the stream's frame `first_frame`."""
        for name, t in (("q", q), ("k", k)):
            if t is not None:
                self._chunk(name, t, frames)
        sr_rope3d_qk_at(self.handle, first_frame, frames, _ptr(q), _ptr(k), _stream(self.device))

    def window_attention(self, step: int, q: torch.Tensor, k_moving: torch.Tensor, v_moving: torch.Tensor,
                         moving_frames: int, with_prefix: bool = False, out: torch.Tensor | None = None,
                         lse: torch.Tensor | bool | None = None):
        """Prefix rows (first n_sink rows of q when with_prefix) see the bank only;
        moving rows see the bank and k_moving / v_moving."""
        M = moving_frames * self.T
        P = self.S if with_prefix else 0
        _check_tensor("q", q, (P + M, self.H, self.d), self.device)
        _check_tensor("k_moving", k_moving, (M, self.H, self.d), self.device)
        _check_tensor("v_moving", v_moving, (M, self.H, self.d), self.device)
        if out is None:
            out = torch.empty_like(q)
        _check_tensor("out", out, (P + M, self.H, self.d), self.device)
        if lse is True:
            lse = torch.empty((self.H, P + M), dtype=torch.float32, device=self.device)
        if isinstance(lse, torch.Tensor):
            _check_tensor("lse", lse, (self.H, P + M), self.device, torch.float32)
        else:
            lse = None
        sr_window_attention(self.handle, step, moving_frames, with_prefix, q.data_ptr(), k_moving.data_ptr(),
                            v_moving.data_ptr(), out.data_ptr(), _ptr(lse), _stream(self.device))
        return (out, lse) if lse is not None else out

    def close(self) -> None:
        if self.handle is not None:
            sr_session_free(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def plan_chunk(chunk_index: int, bootstrap_units: int = 7, chunk_units: int = 2, window_units: int = 2,
               sink_units: int = 2, merge_single_frame_units: bool = True) -> dict:
    """The unit rhythm's plan for one chunk (host arithmetic in libsr.so):
    first_frame, n_frames, hist_frames, sink_frames."""
    p = sr_plan_chunk(chunk_index, bootstrap_units, chunk_units, window_units, sink_units,
                      merge_single_frame_units)
    return {"first_frame": p.first_frame, "n_frames": p.n_frames, "hist_frames": p.hist_frames,
            "sink_frames": p.sink_frames}


def chunk_attention_batch(sessions, step: int, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                          out: torch.Tensor | None = None, lse: torch.Tensor | bool | None = None):
    """One launch over several sessions' chunks packed along L (session i owns
    rows [off[i], off[i+1]) with off the running sum of each session's F*T)."""
    s0 = sessions[0]
    offs = [0]
    for s in sessions:
        offs.append(offs[-1] + s.lq)
    shape = (offs[-1], s0.H, s0.d)
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check_tensor(name, t, shape, s0.device)
    if out is None:
        out = torch.empty_like(q)
    _check_tensor("out", out, shape, s0.device)
    if lse is True:
        lse = torch.empty((s0.H, offs[-1]), dtype=torch.float32, device=s0.device)
    if isinstance(lse, torch.Tensor):
        _check_tensor("lse", lse, (s0.H, offs[-1]), s0.device, torch.float32)
    else:
        lse = None
    sr_chunk_attention_batch([s.handle for s in sessions], step, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                             offs, out.data_ptr(), _ptr(lse), _stream(s0.device))
    return (out, lse) if lse is not None else out
