"""One streaming session, step by step, float64 (test infrastructure only).

The calls follow the streaming loop of [H3-page] "Interactive Coding Worlds
with Real-time Streaming Diffusion Render":
  * session set-up: one static-context (sink) K/V bank per denoising step,
    made at the start of the session and read by every chunk after (section 3.3
    "Static-context KV caching"; [teardown] "A window that slides, and a
    prefix that doesn't": text rows carry the timestep, so the steps cannot
    share a bank);
  * per chunk, two denoising steps (section 3.1.3 "Two-step generation"),
    each: rotary positions on the chunk's Q and K, then attention of the
    chunk's queries over  bank[step]  U  occupied ring frames  U  the chunk
    itself (section 3.1.2);
  * after the last step, the clean chunk's K (rotated at its absolute frame
    positions) and V are written into the ring, evicting the oldest frames
    (section 3.2 Iteration 3 item 2, Iteration 4).

Rounding points: bf16 (ties to even) exactly where the API stores bf16 --
the rotated Q/K handed back by ``rope3d_qk`` and the ring's K/V. Attention
output and LSE stay float64.

Sink banks are opaque, already-final K/V: no rotary position is applied to
them (the pages do not say which positions the conditioning rows carry).
"""
import math
import numpy as np

from .bf16 import bf16_bits_to_f64, f64_to_bf16_bits
from .rope import token_positions, rope3d
from .attention import attention
from .ring import RingCache


class OracleSession:
    def __init__(self, n_heads, head_dim, grid_h, grid_w, chunk_frames, window_frames,
                 n_sink, n_steps, sink_k_bits=None, sink_v_bits=None, t_clock0=0,
                 rope_base=10000.0, softmax_scale=None):
        self.H, self.d = n_heads, head_dim
        self.grid_h, self.grid_w = grid_h, grid_w
        self.T = grid_h * grid_w
        self.F, self.W, self.S, self.n_steps = chunk_frames, window_frames, n_sink, n_steps
        self.t_clock0 = t_clock0
        self.base = rope_base
        self.scale = softmax_scale if softmax_scale else 1.0 / math.sqrt(head_dim)
        shape = (n_steps, n_sink, n_heads, head_dim)
        self.sink_k = np.zeros(shape) if sink_k_bits is None else bf16_bits_to_f64(sink_k_bits).reshape(shape)
        self.sink_v = np.zeros(shape) if sink_v_bits is None else bf16_bits_to_f64(sink_v_bits).reshape(shape)
        self.ring = RingCache(window_frames, self.T, n_heads, head_dim)

    @property
    def n_committed(self) -> int:
        return self.ring.n

    def load_ring(self, ring_k_bits, ring_v_bits, slot_frame, n_committed):
        """Start mid-stream from a given ring state."""
        self.ring.k[:] = bf16_bits_to_f64(ring_k_bits)
        self.ring.v[:] = bf16_bits_to_f64(ring_v_bits)
        self.ring.slot_frame[:] = slot_frame
        self.ring.n = n_committed

    def chunk_positions(self, frames=None):
        frames = self.F if frames is None else frames
        return token_positions(frames * self.T, self.grid_h, self.grid_w,
                               self.t_clock0 + self.ring.n)

    def rope3d_qk(self, q_bits, k_bits, frames=None):
        """Rotate the chunk's Q and K at frames n .. n+F-1 (F = ``frames``,
        default the configured chunk length); bf16 bits out."""
        t, h, w = self.chunk_positions(frames)
        q = rope3d(bf16_bits_to_f64(q_bits), t, h, w, self.base)
        k = rope3d(bf16_bits_to_f64(k_bits), t, h, w, self.base)
        return f64_to_bf16_bits(q), f64_to_bf16_bits(k)

    def rope3d_at(self, first_frame, frames, q_bits, k_bits):
        """Rotate the rows of ``frames`` consecutive frames whose first frame is
        the stream's frame ``first_frame`` (time t_clock0 + first_frame + f):
        used for recomputed history rows, which keep their own frame times."""
        t, h, w = token_positions(frames * self.T, self.grid_h, self.grid_w, self.t_clock0 + first_frame)
        q = rope3d(bf16_bits_to_f64(q_bits), t, h, w, self.base)
        k = rope3d(bf16_bits_to_f64(k_bits), t, h, w, self.base)
        return f64_to_bf16_bits(q), f64_to_bf16_bits(k)

    def window_attention(self, step, q_bits, k_moving_bits, v_moving_bits, with_prefix):
        """The pages' window with a fixed prefix and a moving part ([teardown]
        "A window that slides, and a prefix that doesn't"; [H3-page] 3.1.2
        "Prefix cache"): the prefix rows attend only to the prefix, the moving
        rows (recomputed recent history, then the chunk) attend to the whole
        window. The prefix's keys and values are the bank of the step.
        q: [S + M][H][d] with the S prefix rows first when ``with_prefix``,
        else [M][H][d]; k_moving, v_moving: [M][H][d]. Returns (o, lse) for
        the rows of q, in order."""
        if not 0 <= step < self.n_steps:
            raise ValueError("step out of range")
        S = self.S if with_prefix else 0
        q = bf16_bits_to_f64(q_bits)
        km, vm = bf16_bits_to_f64(k_moving_bits), bf16_bits_to_f64(v_moving_bits)
        kp, vp = self.sink_k[step], self.sink_v[step]
        o_m, l_m = attention(q[S:], np.concatenate([kp, km]), np.concatenate([vp, vm]), self.scale)
        if not with_prefix:
            return o_m, l_m
        o_p, l_p = attention(q[:S], kp, vp, self.scale)
        return np.concatenate([o_p, o_m]), np.concatenate([l_p, l_m], axis=1)

    def visible_kv(self, step, k_bits, v_bits, hist=None):
        """bank[step], then the ring's frames (every occupied slot, or only
        the last ``hist`` committed frames), then the chunk."""
        rk, rv, _ = self.ring.visible() if hist is None else self.ring.recent(hist)
        k = np.concatenate([self.sink_k[step], rk, bf16_bits_to_f64(k_bits)], axis=0)
        v = np.concatenate([self.sink_v[step], rv, bf16_bits_to_f64(v_bits)], axis=0)
        return k, v

    def chunk_attention(self, step, q_bits, k_bits, v_bits, rows=None, heads=None, hist=None):
        """Attention of the (already rotated) chunk queries for denoising
        step ``step``, over the ring's occupied frames or, with ``hist``, its
        last ``hist`` committed frames. Optionally only for a sample of rows
        and heads."""
        if not 0 <= step < self.n_steps:
            raise ValueError("step out of range")
        k, v = self.visible_kv(step, k_bits, v_bits, hist)
        q = bf16_bits_to_f64(q_bits)
        if rows is not None:
            q = q[np.asarray(rows)]
        if heads is not None:
            heads = np.asarray(heads)
            q, k, v = q[:, heads], k[:, heads], v[:, heads]
        return attention(q, k, v, self.scale)

    def cache_commit(self, k_raw_bits, v_bits, frames=None):
        """Rotate the clean chunk's K at its frame positions, round K and V
        to bf16 and write frames n .. n+F-1 into slots (n+f) mod W (F =
        ``frames``, default the configured chunk length)."""
        frames = self.F if frames is None else frames
        t, h, w = self.chunk_positions(frames)
        k = rope3d(bf16_bits_to_f64(k_raw_bits), t, h, w, self.base)
        k = bf16_bits_to_f64(f64_to_bf16_bits(k))
        v = bf16_bits_to_f64(v_bits)
        if self.W == 0:
            self.ring.n += frames
            return
        self.ring.commit(k, v, frames)

    def ring_bits(self):
        return f64_to_bf16_bits(self.ring.k), f64_to_bf16_bits(self.ring.v)
