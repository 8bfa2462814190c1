"""Float64 CPU oracle for the streaming chunk-attention path.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use it. It shares no code with the CUDA library (no kernels,
headers, tables or constant generators); both receive the same seeded bf16
inputs from the separate ``synthetic`` module.

What it computes, and where the pages define it. The pages are
  [H3-page]  "Interactive Coding Worlds with Real-time Streaming Diffusion
             Render" (NVlabs Sol-Engine, StreamRender-H3 project page), and
  [teardown] "StreamRender-H3: the engine paints flat colours, a 33B video
             model paints the rest".

* ``attention``  softmax(scale * Q K^T) V over the visible set with no mask:
  a chunk is denoised with two-way attention over its whole window
  ([H3-page] section 3.1.2) and its rows see every key of that window
  ([H3-page] 3.1.2 "Prefix cache").
* ``rope``       3D (t, h, w) rotary positions applied once, at the absolute
  latent-frame index of the stream ([H3-page] 3.2 Iteration 3 item 2 and
  Iteration 4).
* ``ring``       preallocated ring of W frames written in place, oldest
  evicted ([H3-page] 3.2 Iteration 3 item 2; 3.3 "Persistent KV layout").
* ``session``    one static sink bank per denoising step ([H3-page] 3.3
  "Static-context KV caching"; [teardown] "A window that slides, and a prefix
  that doesn't"), two steps then commit; chunks of any number of frames and
  a recent history of the last h committed frames; the page-faithful window
  (prefix rows see only the prefix, recomputed moving rows see everything).
* ``decoder``    the streaming decoder's window attention, one layer: windows
  of 16x16 tokens, shifted every other layer, each seeing the global tokens,
  its cached frames and its chunk ([H3-page] 3.2 Iterations 2-4).
* ``schedule``   the scheduling units (2, 1, 1, 1 latents), the 7-unit first
  window and the per-chunk plan ([teardown] "A window that slides, and a
  prefix that doesn't"; [H3-page] 3.1.2).

Every function here is pinned by ``tests/test_oracle_*.py`` against closed
forms, invariants, library routines or brute force; no function is
"parity unpinned".
"""
from .bf16 import bf16_bits_to_f64, f64_to_bf16_bits, round_bf16
from .rope import axis_split, inverse_frequencies, token_positions, rope3d
from .attention import attention, attention_rows
from .ring import RingCache
from .session import OracleSession
from .schedule import chunk_plan, latent_rgb_frames, unit_latents, units_latents

__all__ = [
    "bf16_bits_to_f64", "f64_to_bf16_bits", "round_bf16",
    "axis_split", "inverse_frequencies", "token_positions", "rope3d",
    "attention", "attention_rows", "RingCache", "OracleSession",
    "chunk_plan", "latent_rgb_frames", "unit_latents", "units_latents",
]
