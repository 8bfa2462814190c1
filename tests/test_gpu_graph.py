"""Device-resident chunk state and CUDA-graph replay, through the C ABI,
against the oracle.

The *_dev calls read the committed-frame count from a device counter when the
kernels run, derive the visible ring rows from it, and advance it in the
commit. Checked here:
  * eagerly, under the pages' unit rhythm (ring rows that wrap, history
    windows shorter than the ring, a first window longer than the ring), every
    chunk against the oracle following the same plan;
  * captured: one CUDA graph per chunk kind (3 latents with 2 of history, 2
    with 3), each captured once and replayed for every later chunk of its kind
    after copying that chunk's inputs into the captured buffers; every replay
    is compared with the oracle and the slot table after it bit for bit.
"""
import numpy as np
import pytest
import torch

import synthetic as syn
from oracle import OracleSession
from tests.gpu_common import assert_attention_close, device, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from chunked_kv_cache_gb300 import build
    build.build()
    device()


SHAPES = [syn.Shape("graph tiny", 4, 64, 6, 10, 3, 3, 64), syn.Shape("graph d128", 2, 128, 8, 16, 3, 4, 200)]


def _pair(sh, dev):
    import chunked_kv_cache_gb300 as sr
    sk, sv = syn.session_sinks(sh, 12)
    gpu = sr.Session(sh.n_heads, sh.head_dim, sh.grid_h, sh.grid_w, sh.chunk_frames, sh.window_frames, sh.n_sink,
                     sh.n_steps, sink_k=to_dev(sk, dev), sink_v=to_dev(sv, dev), t_clock0=2, device_state=True,
                     device=dev)
    ora = OracleSession(sh.n_heads, sh.head_dim, sh.grid_h, sh.grid_w, sh.chunk_frames, sh.window_frames,
                        sh.n_sink, sh.n_steps, sk, sv, t_clock0=2)
    return gpu, ora


def _oracle_chunk(ora, x, F, h):
    refs = []
    for s in range(len(x.q)):
        qo, ko = ora.rope3d_qk(x.q[s], x.k[s], frames=F)
        refs.append(ora.chunk_attention(s, qo, ko, x.v[s], hist=h)[0])
    ora.cache_commit(x.clean_k, x.clean_v, frames=F)
    return refs


@pytest.mark.parametrize("sh", SHAPES, ids=lambda s: s.name)
def test_device_state_calls_follow_the_rhythm(sh):
    import chunked_kv_cache_gb300 as sr
    dev = device()
    gpu, ora = _pair(sh, dev)
    for c in range(10):
        plan = sr.plan_chunk(c)
        F, h = plan["n_frames"], min(plan["hist_frames"], sh.window_frames)
        x = syn.chunk_inputs(sh, 12, chunk=c, frames=F)
        outs = []
        for s in range(sh.n_steps):
            q, k, v = to_dev(x.q[s], dev), to_dev(x.k[s], dev), to_dev(x.v[s], dev)
            gpu.rope3d_qk_dev(q, k, F)
            outs.append(gpu.chunk_attention_dev(s, q, k, v, F, h))
        gpu.cache_commit_dev(to_dev(x.clean_k, dev), to_dev(x.clean_v, dev), F)
        refs = _oracle_chunk(ora, x, F, h)
        for s in range(sh.n_steps):
            assert_attention_close(outs[s].float().cpu().numpy().astype(np.float64), refs[s], f"chunk {c} step {s}")
        assert int(gpu.frame_counter.item()) == ora.n_committed
        assert np.array_equal(gpu.slot_frame.cpu().numpy(), ora.ring.slot_frame.astype(np.int32)), f"chunk {c}"
    assert gpu.error_status() == 0
    gpu.close()


@pytest.mark.parametrize("sh", SHAPES, ids=lambda s: s.name)
def test_one_graph_per_chunk_kind_serves_every_chunk(sh):
    import chunked_kv_cache_gb300 as sr
    dev = device()
    gpu, ora = _pair(sh, dev)
    T, H, d = sh.tokens_per_frame, sh.n_heads, sh.head_dim
    # the first window (9 latents) and the first two chunks run eagerly
    c = 0
    for c in range(3):
        plan = sr.plan_chunk(c)
        F, h = plan["n_frames"], min(plan["hist_frames"], sh.window_frames)
        x = syn.chunk_inputs(sh, 12, chunk=c, frames=F)
        for s in range(sh.n_steps):
            q, k, v = to_dev(x.q[s], dev), to_dev(x.k[s], dev), to_dev(x.v[s], dev)
            gpu.rope3d_qk_dev(q, k, F)
            gpu.chunk_attention_dev(s, q, k, v, F, h)
        gpu.cache_commit_dev(to_dev(x.clean_k, dev), to_dev(x.clean_v, dev), F)
        _oracle_chunk(ora, x, F, h)
    torch.cuda.synchronize()
    # static buffers and one graph per chunk kind
    graphs, bufs = {}, {}
    for F, h in ((3, 2), (2, 3)):
        h = min(h, sh.window_frames)
        b = {n: [torch.zeros((F * T, H, d), dtype=torch.bfloat16, device=dev) for _ in range(sh.n_steps)]
             for n in ("q", "k", "v", "o")}
        b["ck"] = torch.zeros((F * T, H, d), dtype=torch.bfloat16, device=dev)
        b["cv"] = torch.zeros_like(b["ck"])
        g = torch.cuda.CUDAGraph()
        n_before = int(gpu.frame_counter.item())
        with torch.cuda.graph(g):
            for s in range(sh.n_steps):
                gpu.rope3d_qk_dev(b["q"][s], b["k"][s], F)
                gpu.chunk_attention_dev(s, b["q"][s], b["k"][s], b["v"][s], F, h, out=b["o"][s])
            gpu.cache_commit_dev(b["ck"], b["cv"], F)
        torch.cuda.synchronize()
        assert int(gpu.frame_counter.item()) == n_before      # capturing ran nothing
        graphs[F], bufs[F] = (g, h), b
    for c in range(3, 13):
        plan = sr.plan_chunk(c)
        F = plan["n_frames"]
        g, h = graphs[F]
        b = bufs[F]
        assert min(plan["hist_frames"], sh.window_frames) == h
        x = syn.chunk_inputs(sh, 12, chunk=c, frames=F)
        for s in range(sh.n_steps):
            b["q"][s].copy_(to_dev(x.q[s], dev))
            b["k"][s].copy_(to_dev(x.k[s], dev))
            b["v"][s].copy_(to_dev(x.v[s], dev))
        b["ck"].copy_(to_dev(x.clean_k, dev))
        b["cv"].copy_(to_dev(x.clean_v, dev))
        g.replay()
        refs = _oracle_chunk(ora, x, F, h)
        for s in range(sh.n_steps):
            assert_attention_close(b["o"][s].float().cpu().numpy().astype(np.float64), refs[s],
                                   f"replay chunk {c} step {s}")
        assert int(gpu.frame_counter.item()) == ora.n_committed
        assert np.array_equal(gpu.slot_frame.cpu().numpy(), ora.ring.slot_frame.astype(np.int32)), f"chunk {c}"
    assert gpu.error_status() == 0
    gpu.close()


def test_device_calls_need_a_counter():
    import chunked_kv_cache_gb300 as sr
    from chunked_kv_cache_gb300 import _native as N
    dev = device()
    sh = SHAPES[0]
    gpu = sr.Session(sh.n_heads, sh.head_dim, sh.grid_h, sh.grid_w, sh.chunk_frames, 3, 0, 1, device=dev)
    q = torch.zeros((2 * sh.tokens_per_frame, sh.n_heads, sh.head_dim), dtype=torch.bfloat16, device=dev)
    st = torch.cuda.current_stream(dev).cuda_stream
    for call in (lambda: N.sr_rope3d_qk_dev(gpu.handle, 2, q.data_ptr(), 0, st),
                 lambda: N.sr_chunk_attention_dev(gpu.handle, 0, 2, -1, q.data_ptr(), q.data_ptr(), q.data_ptr(),
                                                  q.data_ptr(), 0, st),
                 lambda: N.sr_cache_commit_dev(gpu.handle, 2, q.data_ptr(), q.data_ptr(), st)):
        with pytest.raises(N.SrError) as e:
            call()
        assert e.value.status == N.SR_ERR_STATE
    gpu.close()
