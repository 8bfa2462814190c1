"""Scheduling units and the per-chunk plan of a session (test infrastructure only).

[teardown] "StreamRender-H3: the engine paints flat colours, a 33B video model
paints the rest", section "A window that slides, and a prefix that doesn't":
the video codec turns 17 RGB frames into 5 latents, the first of every five
latents covering one RGB frame and the other four covering four each; with
single-frame latents merged into their neighbour, scheduling units hold 2, 1,
1, 1 latents and the pattern repeats. The shipped configuration keeps 2 units
of sink, 2 units of recent history, 2 units per chunk, and a first window of 7
units. [H3-page] "Interactive Coding Worlds with Real-time Streaming Diffusion
Render", section 3.1.2: the first window of a stream generates seven units at
once; every later chunk is two units with two units of recent history.

Readings where the pages leave a step open:
  * the first window (chunk 0) has no recent history;
  * the recent history of chunk c >= 1 is the ``window_units`` units right
    before it, i.e. the latents of those units;
  * the sink is the first ``sink_units`` units of the stream;
  * without merging, every latent is a unit of its own.
"""


def unit_latents(u: int, merge_single_frame_units: bool = True) -> int:
    """Latents in unit u (0-based): the one-RGB-frame latent that opens
    every group of five is glued to its neighbour, so units 0, 4, 8, ... hold
    two latents and the others one."""
    if not merge_single_frame_units:
        return 1
    return 2 if u % 4 == 0 else 1


def units_latents(u0: int, n: int, merge_single_frame_units: bool = True) -> int:
    """Latents in units u0 .. u0 + n - 1."""
    return sum(unit_latents(u, merge_single_frame_units) for u in range(u0, u0 + n))


def latent_rgb_frames(latent: int) -> int:
    """RGB frames one latent covers: one for the first of every five, else four."""
    return 1 if latent % 5 == 0 else 4


def chunk_plan(c: int, bootstrap_units: int = 7, chunk_units: int = 2, window_units: int = 2,
               sink_units: int = 2, merge_single_frame_units: bool = True) -> dict:
    """Latents of chunk c: its first latent, its length, the recent history
    it sees (in latents) and the sink (in latents)."""
    if c < 0:
        raise ValueError("chunk index must be >= 0")
    m = merge_single_frame_units
    if c == 0:
        u0, nu, hist = 0, bootstrap_units, 0
    else:
        u0 = bootstrap_units + (c - 1) * chunk_units
        nu = chunk_units
        hu = min(window_units, u0)
        hist = units_latents(u0 - hu, hu, m)
    return {
        "first_latent": units_latents(0, u0, m),
        "n_frames": units_latents(u0, nu, m),
        "hist_frames": hist,
        "sink_frames": units_latents(0, sink_units, m),
    }
