"""The streaming decoder's window attention on the GPU, through the C ABI,
against the oracle's whole-frame computation (oracle/decoder.py).

A layer of windows (plain and shifted, so edge windows are partial) runs a
stream of chunks from an empty cache: the first chunks see a cache that is
still filling (its empty slots are simply not visited), later ones the full
four frames. Every window's rows of every chunk are compared with the oracle.
"""
import numpy as np
import pytest
import torch

import synthetic as syn
from oracle.decoder import DecoderLayerOracle
from oracle import f64_to_bf16_bits
from tests.gpu_common import assert_attention_close, assert_rotated_close, device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from chunked_kv_cache_gb300 import build
    build.build()
    device()


def _bits_dev(bits, dev):
    return torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)


@pytest.mark.parametrize("gh,gw,H,d", [(40, 40, 4, 64), (21, 37, 2, 128)])
@pytest.mark.parametrize("shifted", [False, True])
def test_decoder_layer_stream(gh, gw, H, d, shifted):
    """Frame-major inputs through the layer calls: one gather + RoPE launch, one
    batched attention launch, one commit launch per chunk."""
    from chunked_kv_cache_gb300.decoder import DecoderWindowLayer
    dev = device()
    G, F = 5, 2
    lay = DecoderWindowLayer(gh, gw, H, d, G, shifted=shifted, t_clock0=4, device=dev)
    ora = DecoderLayerOracle(gh, gw, 16, shifted, H, d, cache_frames=4, t_clock0=4)
    assert [(w.row0, w.col0, w.rows, w.cols) for w in lay.windows] == ora.windows
    idx = lay.packing_index().numpy()
    rng = np.random.default_rng(gh + shifted)
    for c in range(4):
        q, k, v, ck, cv = (syn.normal_bf16_bits((F, gh, gw, H, d), rng) for _ in range(5))
        gk, gv = syn.normal_bf16_bits((G, H, d), rng), syn.normal_bf16_bits((G, H, d), rng)
        qd, kd, vd, ckd, cvd = (_bits_dev(b, dev) for b in (q, k, v, ck, cv))
        lay.set_global(_bits_dev(gk, dev), _bits_dev(gv, dev))
        qp, kp, vp = lay.gather_rope(qd, kd, vd)
        o = lay.attention(qp, kp, vp)
        lay.commit(ckd, cvd)
        ref = ora.step(q, k, v, gk, gv)
        ora.commit(ck, cv)
        got = np.empty((F * gh * gw, H, d))
        got[idx] = o.float().cpu().numpy()
        assert_attention_close(got, ref.reshape(-1, H, d), f"chunk {c} (cache {min(2 * c, 4)} frames)")
        # the packed V is a plain gather of the frame-major V
        assert np.array_equal(syn.torch_to_bits(vp), v.reshape(-1, H, d)[idx])
    # every window's ring holds its cached frames: K rotated like the oracle's, V copied
    for s, (r0, c0, nr, nc) in zip(lay.sessions, ora.windows):
        rk, rv = syn.torch_to_bits(s.ring_k), syn.torch_to_bits(s.ring_v)
        slots = s.slot_frame.cpu().numpy()
        T = nr * nc
        for g, ok_, ov_ in ora.cache:
            slot = g % 4
            assert slots[slot] == g
            want_k = f64_to_bf16_bits(ok_[r0:r0 + nr, c0:c0 + nc]).reshape(T, H, d)
            want_v = f64_to_bf16_bits(ov_[r0:r0 + nr, c0:c0 + nc]).reshape(T, H, d)
            assert np.array_equal(rv[slot * T:(slot + 1) * T], want_v)
            assert_rotated_close(rk[slot * T:(slot + 1) * T], want_k, f"ring K of window ({r0}, {c0}) frame {g}")
    assert lay.error_status() == 0
    lay.close()


def test_layer_calls_match_per_window_calls_bit_for_bit():
    """The one-launch gather + RoPE and commit of a layer give the same bits as
    the per-window calls on a gather done by indexing (the same arithmetic)."""
    import chunked_kv_cache_gb300 as sr
    from chunked_kv_cache_gb300.decoder import DecoderWindowLayer
    dev = device()
    gh, gw, H, d, G, F = 45, 80, 3, 128, 5, 2
    for shifted in (False, True):
        lay = DecoderWindowLayer(gh, gw, H, d, G, shifted=shifted, t_clock0=9, device=dev)
        ref = DecoderWindowLayer(gh, gw, H, d, G, shifted=shifted, t_clock0=9, device=dev)
        idx = lay.packing_index().to(dev)
        rng = np.random.default_rng(40 + shifted)
        for c in range(3):   # 6 frames through 4-frame rings: the commits wrap
            q, k, v, ck, cv = (_bits_dev(syn.normal_bf16_bits((F, gh, gw, H, d), rng), dev) for _ in range(5))
            qp, kp, vp = lay.gather_rope(q, k, v)
            flat = lambda t: t.reshape(F * gh * gw, H, d)[idx].contiguous()
            rq, rk_, rv = flat(q), flat(k), flat(v)
            for i, s in enumerate(ref.sessions):
                a, b = ref.offsets[i], ref.offsets[i + 1]
                s.rope3d_qk(rq[a:b], rk_[a:b])
            assert torch.equal(qp, rq) and torch.equal(kp, rk_) and torch.equal(vp, rv)
            lay.commit(ck, cv)
            pck, pcv = flat(ck), flat(cv)
            for i, s in enumerate(ref.sessions):
                a, b = ref.offsets[i], ref.offsets[i + 1]
                s.cache_commit(pck[a:b], pcv[a:b])
            torch.cuda.synchronize()
            for s1, s2 in zip(lay.sessions, ref.sessions):
                assert s1.frames == s2.frames == F * (c + 1)
                assert torch.equal(s1.slot_frame, s2.slot_frame)
                # the slots written so far (the others hold whatever the allocator left)
                rows = torch.repeat_interleave(s1.slot_frame >= 0, s1.T)
                assert torch.equal(s1.ring_k[rows], s2.ring_k[rows]) and torch.equal(s1.ring_v[rows], s2.ring_v[rows])
        # only the packed rows were written: the frame-major inputs are untouched
        q0 = _bits_dev(syn.normal_bf16_bits((F, gh, gw, H, d), rng), dev)
        keep = q0.clone()
        lay.gather_rope(q0, q0.clone())
        assert torch.equal(q0, keep)
        assert lay.error_status() == 0 and ref.error_status() == 0
        lay.close()
        ref.close()


@pytest.mark.parametrize("gh,gw,window,F,C,d", [
    (176, 176, 16, 2, 4, 64),    # 121 windows: two gather / commit launches of at most 96 windows
    (20, 24, 8, 1, 3, 64),       # one-frame chunks into 3-frame caches (commits wrap every 3 chunks)
    (16, 24, 8, 3, 0, 128),      # no cache: the commit only advances the frame counts
])
def test_layer_calls_edge_shapes_match_per_window_calls(gh, gw, window, F, C, d):
    from chunked_kv_cache_gb300.decoder import DecoderWindowLayer
    dev = device()
    H, G = 2, 5
    lay = DecoderWindowLayer(gh, gw, H, d, G, window=window, chunk_frames=F, cache_frames=C, t_clock0=3, device=dev)
    ref = DecoderWindowLayer(gh, gw, H, d, G, window=window, chunk_frames=F, cache_frames=C, t_clock0=3, device=dev)
    idx = lay.packing_index().to(dev)
    rng = np.random.default_rng(gh + F + C)
    flat = lambda t: t.reshape(F * gh * gw, H, d)[idx].contiguous()
    for c in range(4):
        q, k, v, ck, cv = (_bits_dev(syn.normal_bf16_bits((F, gh, gw, H, d), rng), dev) for _ in range(5))
        qp, kp, vp = lay.gather_rope(q, k, v)
        rq, rk_, rv = flat(q), flat(k), flat(v)
        for i, s in enumerate(ref.sessions):
            a, b = ref.offsets[i], ref.offsets[i + 1]
            s.rope3d_qk(rq[a:b], rk_[a:b])
        assert torch.equal(qp, rq) and torch.equal(kp, rk_) and torch.equal(vp, rv), c
        lay.commit(ck, cv)
        pck, pcv = flat(ck), flat(cv)
        for i, s in enumerate(ref.sessions):
            a, b = ref.offsets[i], ref.offsets[i + 1]
            s.cache_commit(pck[a:b], pcv[a:b])
        torch.cuda.synchronize()
        for s1, s2 in zip(lay.sessions, ref.sessions):
            assert s1.frames == s2.frames == F * (c + 1)
            if C > 0:
                assert torch.equal(s1.slot_frame, s2.slot_frame)
                rows = torch.repeat_interleave(s1.slot_frame >= 0, s1.T)
                assert torch.equal(s1.ring_k[rows], s2.ring_k[rows]) and torch.equal(s1.ring_v[rows], s2.ring_v[rows])
    assert lay.error_status() == 0 and ref.error_status() == 0
    lay.close()
    ref.close()


def test_decoder_layer_graph_replay_matches_eager():
    """A layer's launches captured in a CUDA graph (persistent launches whose
    work counter the last CTA clears) replay to the eager result, bit for bit:
    the unit order changes nothing in the arithmetic."""
    from chunked_kv_cache_gb300.decoder import DecoderWindowLayer
    dev = device()
    H, d, G = 4, 128, 5
    for shifted in (False, True):
        lay = DecoderWindowLayer(45, 80, H, d, G, shifted=shifted, device=dev)
        rng = np.random.default_rng(7 + shifted)
        mk = lambda: _bits_dev(syn.normal_bf16_bits((lay.rows, H, d), rng), dev)
        q, k, v, ck, cv = mk(), mk(), mk(), mk(), mk()
        lay.set_global(_bits_dev(syn.normal_bf16_bits((G, H, d), rng), dev),
                       _bits_dev(syn.normal_bf16_bits((G, H, d), rng), dev))
        for _ in range(2):
            lay.commit(ck, cv)
        o = torch.empty_like(q)
        lay.attention(q, k, v, out=o)
        torch.cuda.synchronize()
        want = o.clone()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            lay.attention(q, k, v, out=o)
        for _ in range(3):
            o.zero_()
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(o, want)
        assert lay.error_status() == 0
        lay.close()
