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
from tests.gpu_common import assert_attention_close, device

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
    from chunked_kv_cache_gb300.decoder import DecoderWindowLayer
    dev = device()
    G, F = 5, 2
    lay = DecoderWindowLayer(gh, gw, H, d, G, shifted=shifted, t_clock0=4, device=dev)
    ora = DecoderLayerOracle(gh, gw, 16, shifted, H, d, cache_frames=4, t_clock0=4)
    assert [(w.row0, w.col0, w.rows, w.cols) for w in lay.windows] == ora.windows
    idx = lay.packing_index().to(dev)
    rng = np.random.default_rng(gh + shifted)
    for c in range(4):
        q, k, v, ck, cv = (syn.normal_bf16_bits((F, gh, gw, H, d), rng) for _ in range(5))
        gk, gv = syn.normal_bf16_bits((G, H, d), rng), syn.normal_bf16_bits((G, H, d), rng)
        pk = lambda b: _bits_dev(b, dev).reshape(F * gh * gw, H, d)[idx].contiguous()
        qd, kd, vd, ckd, cvd = pk(q), pk(k), pk(v), pk(ck), pk(cv)
        lay.set_global(_bits_dev(gk, dev), _bits_dev(gv, dev))
        lay.rope(qd, kd)
        o = lay.attention(qd, kd, vd)
        lay.commit(ckd, cvd)
        ref = ora.step(q, k, v, gk, gv)
        ora.commit(ck, cv)
        got = np.empty((F * gh * gw, H, d))
        got[idx.cpu().numpy()] = o.float().cpu().numpy()
        assert_attention_close(got, ref.reshape(-1, H, d), f"chunk {c} (cache {min(2 * c, 4)} frames)")
    assert lay.error_status() == 0
    lay.close()


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
