"""Nothing is written outside the caller's buffers.

compute-sanitizer is not available on the GPU pool, so out-of-bounds writes are
caught the old way: every buffer the library writes (sink banks, ring K/V,
slot table, error word, workspace, the in-place Q/K and the outputs) sits
between two guard bands filled with a canary byte, and after a run that wraps
the ring, splits last blocks over work units and takes both denoising steps
(and one allocation-free attention call), every guard byte must still hold
the canary. The session is built through the C ABI directly so that its
buffers can be placed inside the guarded blocks."""
import numpy as np
import pytest
import torch

import synthetic as syn
from tests.gpu_common import device, to_dev

pytestmark = pytest.mark.gpu

GUARD = 4096        # bytes on each side; keeps every buffer 256-byte aligned
CANARY = 0xA5


@pytest.fixture(scope="module", autouse=True)
def _built():
    from chunked_kv_cache_gb300 import build
    build.build()
    device()


class Guarded:
    """A device buffer of nbytes between two canary-filled guard bands."""

    def __init__(self, nbytes, dev):
        self.n = nbytes
        self.block = torch.full((GUARD + nbytes + GUARD,), CANARY, dtype=torch.uint8, device=dev)
        self.inner = self.block[GUARD:GUARD + nbytes]

    def view(self, dtype, shape):
        return self.inner.view(dtype).view(shape)

    def intact(self):
        return bool(torch.all(self.block[:GUARD] == CANARY)) and bool(torch.all(self.block[GUARD + self.n:] == CANARY))


def test_nothing_written_outside_the_buffers():
    from chunked_kv_cache_gb300 import _native as N
    dev = device()
    shape = syn.TINY
    H, d, W, S, F, n_steps = (shape.n_heads, shape.head_dim, shape.window_frames, shape.n_sink,
                              shape.chunk_frames, shape.n_steps)
    T = shape.grid_h * shape.grid_w
    rows = (shape.lq, H, d)
    bf16 = torch.bfloat16
    cfg = N.SrConfig(H, d, shape.grid_h, shape.grid_w, F, W, S, n_steps, 0, shape.rope_base, 0.0, 0, 2)
    bank_k = Guarded(n_steps * S * H * d * 2, dev)
    bank_v = Guarded(n_steps * S * H * d * 2, dev)
    ring_k = Guarded(W * T * H * d * 2, dev)
    ring_v = Guarded(W * T * H * d * 2, dev)
    slots = Guarded(W * 4, dev)
    err = Guarded(4, dev)
    err.view(torch.int32, (1,)).zero_()
    ws = Guarded(N.sr_workspace_bytes(cfg), dev)
    guarded = [bank_k, bank_v, ring_k, ring_v, slots, err, ws]
    bufs = N.SrBuffers(bank_k.inner.data_ptr(), bank_v.inner.data_ptr(), ring_k.inner.data_ptr(),
                       ring_v.inner.data_ptr(), slots.inner.data_ptr(), err.inner.data_ptr(),
                       ws.inner.data_ptr(), None)
    sk, sv = syn.session_sinks(shape, 1)
    sk_d, sv_d = to_dev(sk, dev), to_dev(sv, dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    handle = N.sr_session_init(cfg, bufs, sk_d.data_ptr(), sv_d.data_ptr(), stream)
    try:
        for c in range(5):      # 10 frames through a 4-frame ring: the commits wrap
            x = syn.chunk_inputs(shape, 1, chunk=c)
            ck, cv = to_dev(x.clean_k, dev), to_dev(x.clean_v, dev)
            N.sr_cache_commit(handle, ck.data_ptr(), cv.data_ptr(), stream)
        x = syn.chunk_inputs(shape, 1, chunk=5)
        outs = []
        for st in range(n_steps):
            q, k = Guarded(shape.lq * H * d * 2, dev), Guarded(shape.lq * H * d * 2, dev)
            q.view(bf16, rows).copy_(to_dev(x.q[st], dev))
            k.view(bf16, rows).copy_(to_dev(x.k[st], dev))
            v = to_dev(x.v[st], dev)
            o = Guarded(shape.lq * H * d * 2, dev)
            lse = Guarded(H * shape.lq * 4, dev)
            guarded += [q, k, o, lse]
            N.sr_rope3d_qk(handle, q.inner.data_ptr(), k.inner.data_ptr(), stream)
            N.sr_chunk_attention(handle, st, q.inner.data_ptr(), k.inner.data_ptr(), v.data_ptr(),
                                 o.inner.data_ptr(), lse.inner.data_ptr(), stream)
            outs.append((o, lse))
        # the allocation-free entry point writes O and LSE through its own host
        # path (its scratch is the library's built-in array): guard those too
        q, k = Guarded(shape.lq * H * d * 2, dev), Guarded(shape.lq * H * d * 2, dev)
        q.view(bf16, rows).copy_(to_dev(x.q[0], dev))
        k.view(bf16, rows).copy_(to_dev(x.k[0], dev))
        v = to_dev(x.v[0], dev)
        o, lse = Guarded(shape.lq * H * d * 2, dev), Guarded(H * shape.lq * 4, dev)
        guarded += [q, k, o, lse]
        N.sr_chunk_attention_noalloc(handle, 0, q.inner.data_ptr(), k.inner.data_ptr(), v.data_ptr(),
                                     o.inner.data_ptr(), lse.inner.data_ptr(), stream)
        outs.append((o, lse))
        torch.cuda.synchronize()
        assert int(err.view(torch.int32, (1,)).item()) == 0
        for o, lse in outs:
            assert bool(torch.isfinite(o.view(bf16, rows).float()).all())
            assert bool(torch.isfinite(lse.view(torch.float32, (H, shape.lq))).all())
        assert [g.intact() for g in guarded] == [True] * len(guarded)
        # the slot table holds the last W committed frames
        got = slots.view(torch.int32, (W,)).cpu().numpy()
        assert sorted(got.tolist()) == list(range(10 - W, 10))
    finally:
        N.sr_session_free(handle)
