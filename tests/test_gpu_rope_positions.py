"""GPU parity of the rotary positions far from the origin.

The time position of a frame is its absolute index in the stream plus the
session clock ([H3-page] "Interactive Coding Worlds with Real-time Streaming
Diffusion Render", section 3.2 Iteration 4), so it grows without bound. The
kernels reduce the angle exactly (a fixed-point phase); the oracle reduces it
in 60-digit decimal arithmetic. Checked through the C ABI: RoPE at clocks
past 2^24 (where a float position is no longer exact) and at 2^30 and
-2^31, a session restored at the last frame count the int32 slot table can
hold, which runs a whole chunk and commits it, a commit past that count being
refused, and recomputed rows rotated at stream frames 2^33 and -2^40.
"""
import numpy as np
import pytest
import torch

import synthetic as syn
from tests.gpu_common import (Twin, assert_attention_close, assert_rotated_close, device, to_dev, LSE_ABS)

pytestmark = pytest.mark.gpu

INT32_MAX = 2 ** 31 - 1


@pytest.fixture(scope="module", autouse=True)
def _built():
    from chunked_kv_cache_gb300 import build
    build.build()
    device()


@pytest.mark.parametrize("config,clock", [(1, 2 ** 24 + 3), (1, 2 ** 30), (1, -(2 ** 31)), (2, 2 ** 24 + 3),
                                          (2, 2 ** 30)])
def test_rope_at_large_clocks_matches_oracle(config, clock):
    shape = syn.SHAPES[config]
    tw = Twin(shape, config, fill=2, t_clock0=clock)
    x = syn.chunk_inputs(shape, config, chunk=3)
    q, k = to_dev(x.q[0], tw.dev), to_dev(x.k[0], tw.dev)
    tw.gpu.rope3d_qk(q, k)
    qo, ko = tw.ora.rope3d_qk(x.q[0], x.k[0])
    assert_rotated_close(syn.torch_to_bits(q), qo, f"q at clock {clock}")
    assert_rotated_close(syn.torch_to_bits(k), ko, f"k at clock {clock}")


def _restore_at(tw, shape, config, n):
    """Put both sides into the state after n committed frames: a full ring
    holding frames n-W .. n-1, each in slot g mod W."""
    W, T = shape.window_frames, shape.tokens_per_frame
    rk, rv, _ = syn.ring_prefill(shape, config, W)
    slots = np.full(W, -1, np.int64)
    for g in range(n - W, n):
        slots[g % W] = g
    tw.gpu.ring_k.copy_(to_dev(rk, tw.dev))
    tw.gpu.ring_v.copy_(to_dev(rv, tw.dev))
    tw.gpu.slot_frame.copy_(torch.from_numpy(slots.astype(np.int32)).to(tw.dev))
    tw.gpu.restore(n)
    tw.ora.load_ring(rk, rv, slots, n)


def test_chunk_at_the_last_committable_frames():
    shape = syn.TINY
    F = shape.chunk_frames
    tw = Twin(shape, 1, t_clock0=5)
    n = INT32_MAX - F                      # one more chunk fits, exactly
    _restore_at(tw, shape, 1, n)
    x = syn.chunk_inputs(shape, 1, chunk=9)
    for step in range(shape.n_steps):
        got, ref, gl, rl = tw.step(x, step, lse=True)
        assert_attention_close(got, ref, f"step {step} at n = {n}")
        assert np.abs(gl - rl).max() <= LSE_ABS
    tw.commit(x)
    torch.cuda.synchronize()
    assert tw.gpu.frames == tw.ora.n_committed == INT32_MAX
    assert np.array_equal(tw.gpu.slot_frame.cpu().numpy(), tw.ora.ring.slot_frame.astype(np.int32))
    rk, rv = tw.ring_bits()
    ok_, ov_ = tw.ora.ring_bits()
    assert np.array_equal(rv, ov_)
    assert_rotated_close(rk, ok_, "ring K")
    # the slot table cannot name frame 2^31: the next commit is refused and changes nothing
    from chunked_kv_cache_gb300 import _native as N
    before = tw.gpu.slot_frame.clone()
    with pytest.raises(N.SrError) as e:
        tw.gpu.cache_commit(to_dev(x.clean_k, tw.dev), to_dev(x.clean_v, tw.dev))
    assert e.value.status == N.SR_ERR_STATE
    torch.cuda.synchronize()
    assert tw.gpu.frames == INT32_MAX and torch.equal(before, tw.gpu.slot_frame)
    with pytest.raises(N.SrError):
        tw.gpu.restore(INT32_MAX + 1)
    assert tw.gpu.error_status() == 0


@pytest.mark.parametrize("first_frame", [2 ** 33, -(2 ** 40), 2 ** 40 - 1])
def test_rope_at_far_stream_frames_matches_oracle(first_frame):
    shape = syn.SHAPE_832x480
    tw = Twin(shape, 2, heads=[0, 13], t_clock0=-17)
    frames = 3
    x = syn.chunk_inputs(shape, 2, chunk=4, frames=frames)
    q, k = to_dev(x.q[0], tw.dev), to_dev(x.k[0], tw.dev)
    tw.gpu.rope3d_at(first_frame, frames, q, k)
    qo, ko = tw.ora.rope3d_at(first_frame, frames, tw.oh(x.q[0]), tw.oh(x.k[0]))
    assert_rotated_close(tw.oh(syn.torch_to_bits(q)), qo, f"q at frame {first_frame}")
    assert_rotated_close(tw.oh(syn.torch_to_bits(k)), ko, f"k at frame {first_frame}")
