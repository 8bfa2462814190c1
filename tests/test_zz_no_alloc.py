"""The allocation-free chunk attention, sr_chunk_attention_noalloc.

It exists for callers that cannot allocate device memory, such as code that
runs inside a framework's fixed memory pool or a plugin that is handed only a
stream and its tensors: they cannot provide the session workspace that the key
split of a chunk's last query block uses, so this entry point takes its scratch
from an array built into the library instead.

Checked here, through the C ABI: two calls in a row agree with
sr_chunk_attention on the same inputs within the attention tolerances of the
parity tests, with the key split forced on (so the built-in scratch is really
used, and reused by the second call), and a session too large for the scratch
is refused before anything runs. This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import synthetic as syn
from tests.gpu_common import LSE_ABS, assert_attention_close, device, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from chunked_kv_cache_gb300 import build
    build.build()
    device()


def test_noalloc_matches_sr_chunk_attention_twice():
    import chunked_kv_cache_gb300 as sr
    from chunked_kv_cache_gb300 import _native as N
    dev = device()
    shape = syn.SHAPE_832x480
    sk, sv = syn.session_sinks(shape, 2)
    # no workspace of its own; the key split of the last blocks is forced to 4 parts
    s = sr.Session(shape.n_heads, shape.head_dim, shape.grid_h, shape.grid_w, shape.chunk_frames,
                   shape.window_frames, shape.n_sink, shape.n_steps, sink_k=to_dev(sk, dev), sink_v=to_dev(sv, dev),
                   tail_split=4, workspace=False, device=dev)
    rk, rv, slots = syn.ring_prefill(shape, 2, shape.window_frames)
    s.ring_k.copy_(to_dev(rk, dev))
    s.ring_v.copy_(to_dev(rv, dev))
    s.slot_frame.copy_(torch.from_numpy(slots).to(dev))
    s.restore(shape.window_frames)
    x = syn.chunk_inputs(shape, 2, chunk=5)
    q, k, v = (to_dev(b, dev) for b in (x.q[0], x.k[0], x.v[0]))
    stream = torch.cuda.current_stream(dev).cuda_stream

    ref_o = torch.empty_like(q)
    ref_l = torch.empty((shape.n_heads, shape.lq), dtype=torch.float32, device=dev)
    N.sr_chunk_attention(s.handle, 0, q.data_ptr(), k.data_ptr(), v.data_ptr(), ref_o.data_ptr(),
                         ref_l.data_ptr(), stream)
    ref = ref_o.float().cpu().numpy().astype(np.float64)
    ref_lse = ref_l.cpu().numpy().astype(np.float64)
    for call in range(2):
        o = torch.full_like(q, float("nan"))
        lse = torch.full((shape.n_heads, shape.lq), float("nan"), dtype=torch.float32, device=dev)
        N.sr_chunk_attention_noalloc(s.handle, 0, q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                     lse.data_ptr(), stream)
        torch.cuda.synchronize()
        got = o.float().cpu().numpy().astype(np.float64)
        assert_attention_close(got, ref, f"noalloc call {call}")
        assert np.abs(lse.cpu().numpy().astype(np.float64) - ref_lse).max() <= LSE_ABS
    assert s.error_status() == 0
    s.close()


def test_noalloc_refuses_sessions_beyond_its_scratch():
    import chunked_kv_cache_gb300 as sr
    from chunked_kv_cache_gb300 import _native as N
    dev = device()
    # 63 heads at head_dim 128 need just over 16 MiB of scratch
    s = sr.Session(63, 128, 1, 1, 1, 0, 0, 1, workspace=False, device=dev)
    q = torch.zeros((1, 63, 128), dtype=torch.bfloat16, device=dev)
    o = torch.empty_like(q)
    with pytest.raises(N.SrError) as e:
        N.sr_chunk_attention_noalloc(s.handle, 0, q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), 0,
                                     torch.cuda.current_stream(dev).cuda_stream)
    assert e.value.status == N.SR_ERR_UNSUPPORTED
    s.close()
