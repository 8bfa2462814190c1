"""Seeded synthetic inputs for the streaming chunk-attention path.

This module is shared by the tests, the bench and the smoke check. It holds
the workload shapes and the random draws, and none of the method's arithmetic:
no RoPE, no attention, no slot math. Both the float64 oracle and the CUDA
library receive the same bf16 bit patterns produced here.

Every tensor is a seeded standard normal draw, rounded once to bf16 (round to
nearest even) so that both sides see identical bits. Seeds follow
``SeedSequence([base_seed, config, session, chunk, step, tensor_id])``.

Layouts are token-major ``[L][H][d]`` (row stride ``H*d``), the packed
variable-length layout that FlashAttention-style kernels read.
"""
from __future__ import annotations

import dataclasses
import numpy as np
import torch

# tensor ids of the seed tuple
T_Q, T_K, T_V, T_SINK_K, T_SINK_V, T_CLEAN_K, T_CLEAN_V, T_RING_K, T_RING_V = range(9)


@dataclasses.dataclass(frozen=True)
class Shape:
    """One workload shape.

    T = grid_h*grid_w tokens per latent frame; a chunk is F frames (Lq = F*T
    queries); the ring holds W frames; each denoising step has its own bank of
    S sink tokens.
    """
    name: str
    n_heads: int
    head_dim: int
    grid_h: int
    grid_w: int
    chunk_frames: int
    window_frames: int
    n_sink: int
    n_steps: int = 2
    rope_base: float = 10000.0

    @property
    def tokens_per_frame(self) -> int:
        return self.grid_h * self.grid_w

    @property
    def lq(self) -> int:
        return self.chunk_frames * self.tokens_per_frame

    def lk(self, valid_frames: int) -> int:
        return self.n_sink + valid_frames * self.tokens_per_frame + self.lq

    def attention_flops(self, valid_frames: int) -> float:
        """QK^T plus PV at two flops per multiply-add."""
        return 4.0 * self.n_heads * self.lq * self.lk(valid_frames) * self.head_dim


# Workload shapes. The 832x480 and 720p shapes use a /16 latent stride
# (30x52 and 45x80 tokens per frame), two latent frames per chunk, sinks of
# one reference frame plus 512 prompt tokens.
TINY = Shape("tiny 4x64, 6x10 grid, S=64, W=4", 4, 64, 6, 10, 2, 4, 64)
SHAPE_832x480 = Shape("832x480 chunk, 24x128, 30x52 grid, S=2072, W=6", 24, 128, 30, 52, 2, 6, 1560 + 512)
SHAPE_720P = Shape("720p chunk, 40x128, 45x80 grid, S=4112, W=8", 40, 128, 45, 80, 2, 8, 3600 + 512)

SHAPES = {1: TINY, 2: SHAPE_832x480, 3: SHAPE_720P}

# Multi-session batch: eight 832x480 sessions with ring fills of 0..6 frames
# plus one full ring.
BATCH_FILLS = (0, 1, 2, 3, 4, 5, 6, 6)
LONG_SESSION_CHUNKS = 240


def rng(config: int, session: int = 0, chunk: int = 0, step: int = 0,
        tensor_id: int = 0, base_seed: int = 0) -> np.random.Generator:
    return np.random.default_rng(
        np.random.SeedSequence([base_seed, config, session, chunk, step, tensor_id]))


def normal_bf16_bits(shape, gen: np.random.Generator, scale: float = 1.0) -> np.ndarray:
    """Standard normal draw (times ``scale``) rounded to bf16; returns uint16 bits."""
    x = gen.standard_normal(size=shape, dtype=np.float32)
    if scale != 1.0:
        x = x * np.float32(scale)
    t = torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bits_to_torch(bits: np.ndarray) -> torch.Tensor:
    """uint16 bf16 bits -> CPU torch.bfloat16 tensor with the same bits."""
    return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16)


def torch_to_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16).copy()


@dataclasses.dataclass
class ChunkInputs:
    """Raw (un-roped) per-step Q/K/V plus the clean K/V committed after the last step."""
    q: list          # per step, uint16 [Lq][H][d]
    k: list
    v: list
    clean_k: np.ndarray
    clean_v: np.ndarray


def session_sinks(shape: Shape, config: int, session: int = 0, base_seed: int = 0):
    """Sink banks [n_steps][S][H][d] (uint16 bits), one independent draw per step."""
    dims = (shape.n_steps, shape.n_sink, shape.n_heads, shape.head_dim)
    sk = np.empty(dims, np.uint16)
    sv = np.empty(dims, np.uint16)
    for s in range(shape.n_steps):
        sk[s] = normal_bf16_bits(dims[1:], rng(config, session, 0, s, T_SINK_K, base_seed))
        sv[s] = normal_bf16_bits(dims[1:], rng(config, session, 0, s, T_SINK_V, base_seed))
    return sk, sv


def chunk_inputs(shape: Shape, config: int, session: int = 0, chunk: int = 0,
                 base_seed: int = 0, q_scale: float = 1.0, frames: int | None = None) -> ChunkInputs:
    """Inputs of one chunk of ``frames`` latent frames (default: the shape's chunk length)."""
    rows = shape.lq if frames is None else frames * shape.tokens_per_frame
    dims = (rows, shape.n_heads, shape.head_dim)
    q, k, v = [], [], []
    for s in range(shape.n_steps):
        q.append(normal_bf16_bits(dims, rng(config, session, chunk, s, T_Q, base_seed), q_scale))
        k.append(normal_bf16_bits(dims, rng(config, session, chunk, s, T_K, base_seed)))
        v.append(normal_bf16_bits(dims, rng(config, session, chunk, s, T_V, base_seed)))
    ck = normal_bf16_bits(dims, rng(config, session, chunk, 0, T_CLEAN_K, base_seed))
    cv = normal_bf16_bits(dims, rng(config, session, chunk, 0, T_CLEAN_V, base_seed))
    return ChunkInputs(q, k, v, ck, cv)


def ring_prefill(shape: Shape, config: int, frames: int, session: int = 0, base_seed: int = 0):
    """Already-committed ring contents for a session that starts mid-stream.

    Frames 0..frames-1 sit in slots 0..frames-1 (their K already carries its
    rotary position: it is simply a draw here). Returns (ring_k, ring_v,
    slot_frame) with ring tensors of shape [W*T][H][d]; slots past ``frames``
    hold the bf16 bit pattern of NaN so that any read of them shows.
    """
    T = shape.tokens_per_frame
    W = shape.window_frames
    assert 0 <= frames <= W
    dims = (W * T, shape.n_heads, shape.head_dim)
    rk = np.full(dims, 0x7FC0, np.uint16)
    rv = np.full(dims, 0x7FC0, np.uint16)
    if frames:
        sub = (frames * T, shape.n_heads, shape.head_dim)
        rk[:frames * T] = normal_bf16_bits(sub, rng(config, session, 0, 0, T_RING_K, base_seed))
        rv[:frames * T] = normal_bf16_bits(sub, rng(config, session, 0, 0, T_RING_V, base_seed))
    slot_frame = np.full((W,), -1, np.int32)
    slot_frame[:frames] = np.arange(frames, dtype=np.int32)
    return rk, rv, slot_frame


def plant_keys(q_bits: np.ndarray, k_bits: np.ndarray, every: int = 97, gain: float = 3.0):
    """Peaky variant: copy a scaled query into the key at the same token for
    every ``every``-th token, so that those queries have one dominant key.
    Works on bits through torch bf16 arithmetic (input preparation only)."""
    q = bits_to_torch(q_bits).float()
    k = bits_to_torch(k_bits).float().clone()
    idx = torch.arange(0, q.shape[0], every)
    k[idx] = q[idx] * gain
    return torch_to_bits(k.to(torch.bfloat16))


def device_normal_bf16(shape, device, config: int, session: int = 0, chunk: int = 0, step: int = 0,
                       tensor_id: int = 0, base_seed: int = 0):
    """Seeded standard normal bf16 tensor drawn on the device (torch's CUDA
    generator), for long runs where host-side draws would dominate. The same
    seed tuple always gives the same bits; callers copy slices to the host
    when the oracle needs them."""
    seed = int(np.random.SeedSequence([base_seed, config, session, chunk, step, tensor_id, 7919])
               .generate_state(1, dtype=np.uint64)[0] & ((1 << 63) - 1))
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def chunk_inputs_device(shape: Shape, config: int, device, session: int = 0, chunk: int = 0,
                        base_seed: int = 0, with_steps: bool = True):
    """Device-side counterpart of ``chunk_inputs`` (different bits, same recipe).
    Returns dict with lists q, k, v (per step, empty if not with_steps) and
    clean_k, clean_v as torch bf16 tensors on ``device``."""
    dims = (shape.lq, shape.n_heads, shape.head_dim)
    out = {"q": [], "k": [], "v": []}
    if with_steps:
        for s in range(shape.n_steps):
            out["q"].append(device_normal_bf16(dims, device, config, session, chunk, s, T_Q, base_seed))
            out["k"].append(device_normal_bf16(dims, device, config, session, chunk, s, T_K, base_seed))
            out["v"].append(device_normal_bf16(dims, device, config, session, chunk, s, T_V, base_seed))
    out["clean_k"] = device_normal_bf16(dims, device, config, session, chunk, 0, T_CLEAN_K, base_seed)
    out["clean_v"] = device_normal_bf16(dims, device, config, session, chunk, 0, T_CLEAN_V, base_seed)
    return out
