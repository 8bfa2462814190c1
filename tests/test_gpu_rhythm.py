"""The pages' unit rhythm on the GPU, through the C ABI, against the oracle.

A session runs the shipped schedule (sr_plan_chunk: a 9-latent first window,
then chunks of 3 and 2 latents with 2 and 3 latents of recent history) into a
ring too small to keep the whole first window. The commit of the first window
keeps only its last W frames, later commits wrap around the end of the ring in
the middle of a chunk, and the recent-history windows wrap too, so the visible
ring frames come in two pieces. Every chunk's attention (all rows, both steps,
and the log-sum-exp) is compared with the oracle following the same plan, the
slot table bit for bit after every commit, and the ring contents at the end.
"""
import numpy as np
import pytest
import torch

import synthetic as syn
from oracle import OracleSession, chunk_plan
from tests.gpu_common import (LSE_ABS, assert_attention_close, assert_rotated_close, device, to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from chunked_kv_cache_gb300 import build
    build.build()
    device()


SHAPES = {
    # 4 heads x 64, 60 tokens per frame: a 3-frame chunk is one single-tile block
    "tiny": syn.Shape("rhythm tiny", 4, 64, 6, 10, 3, 3, 64),
    # 2 heads x 128, 128 tokens per frame: 3 frames = 384 rows (a full block and a
    # single-tile last block), 9 frames = 1152 rows
    "d128": syn.Shape("rhythm d128", 2, 128, 8, 16, 3, 4, 200),
}


@pytest.mark.parametrize("name,W", [("tiny", 3), ("tiny", 4), ("d128", 3), ("d128", 4), ("d128", 5)])
def test_unit_rhythm_session(name, W):
    import chunked_kv_cache_gb300 as sr
    dev = device()
    base = SHAPES[name]
    sh = syn.Shape(base.name, base.n_heads, base.head_dim, base.grid_h, base.grid_w, base.chunk_frames, W,
                   base.n_sink, base.n_steps)
    T = sh.tokens_per_frame
    sk, sv = syn.session_sinks(sh, 6)
    gpu = sr.Session(sh.n_heads, sh.head_dim, sh.grid_h, sh.grid_w, sh.chunk_frames, W, sh.n_sink, sh.n_steps,
                     sink_k=to_dev(sk, dev), sink_v=to_dev(sv, dev), t_clock0=3, device=dev)
    ora = OracleSession(sh.n_heads, sh.head_dim, sh.grid_h, sh.grid_w, sh.chunk_frames, W, sh.n_sink,
                        sh.n_steps, sk, sv, t_clock0=3)
    wrapped_hist = False
    for c in range(12):
        plan = sr.plan_chunk(c)
        ref_plan = chunk_plan(c)
        F, h = plan["n_frames"], plan["hist_frames"]
        assert F == ref_plan["n_frames"] and h == ref_plan["hist_frames"]
        assert gpu.frames == ora.n_committed == plan["first_frame"]
        h = min(h, W)
        n = ora.n_committed
        if h and (n - h) % W + h > W:
            wrapped_hist = True
        x = syn.chunk_inputs(sh, 6, chunk=c, frames=F)
        for s in range(sh.n_steps):
            q, k, v = to_dev(x.q[s], dev), to_dev(x.k[s], dev), to_dev(x.v[s], dev)
            gpu.rope3d_qk(q, k, frames=F)
            o, lse = gpu.chunk_attention(s, q, k, v, lse=True, frames=F, hist=h)
            qo, ko = ora.rope3d_qk(x.q[s], x.k[s], frames=F)
            assert_rotated_close(syn.torch_to_bits(q), qo, f"chunk {c} step {s} q")
            ref, ref_lse = ora.chunk_attention(s, qo, ko, x.v[s], hist=h)
            assert_attention_close(o.float().cpu().numpy().astype(np.float64), ref, f"chunk {c} step {s}")
            assert np.abs(lse.cpu().numpy().astype(np.float64) - ref_lse).max() <= LSE_ABS
        gpu.cache_commit(to_dev(x.clean_k, dev), to_dev(x.clean_v, dev), frames=F)
        ora.cache_commit(x.clean_k, x.clean_v, frames=F)
        assert np.array_equal(gpu.slot_frame.cpu().numpy(), ora.ring.slot_frame.astype(np.int32)), f"chunk {c}"
    assert wrapped_hist, "the schedule never exercised a wrapped history window"
    rk, rv = syn.torch_to_bits(gpu.ring_k), syn.torch_to_bits(gpu.ring_v)
    ok_, ov_ = ora.ring_bits()
    assert np.array_equal(rv, ov_)
    assert_rotated_close(rk, ok_, "ring K after the rhythm")
    assert gpu.error_status() == 0
    gpu.close()


def test_frames_argument_checks():
    import chunked_kv_cache_gb300 as sr
    from chunked_kv_cache_gb300 import _native as N
    dev = device()
    sh = SHAPES["tiny"]
    gpu = sr.Session(sh.n_heads, sh.head_dim, sh.grid_h, sh.grid_w, sh.chunk_frames, 3, 0, 1, device=dev)
    q = torch.zeros((2 * sh.tokens_per_frame, sh.n_heads, sh.head_dim), dtype=torch.bfloat16, device=dev)
    st = torch.cuda.current_stream(dev).cuda_stream
    for bad_hist in (-2, 1):   # nothing committed yet: no history can be visible
        with pytest.raises(N.SrError) as e:
            N.sr_chunk_attention_frames(gpu.handle, 0, 2, bad_hist, q.data_ptr(), q.data_ptr(), q.data_ptr(),
                                        q.data_ptr(), 0, st)
        assert e.value.status == N.SR_ERR_INVALID_ARG
    for bad_frames in (0, -3):
        with pytest.raises(N.SrError):
            N.sr_rope3d_qk_frames(gpu.handle, bad_frames, q.data_ptr(), 0, st)
        with pytest.raises(N.SrError):
            N.sr_cache_commit_frames(gpu.handle, bad_frames, q.data_ptr(), q.data_ptr(), st)
    assert gpu.frames == 0
    gpu.close()
