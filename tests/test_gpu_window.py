"""The page-faithful window on the GPU, through the C ABI, against the oracle.

sr_window_attention computes the prefix rows (which see only the bank of the
step) and the moving rows (recomputed history and the chunk, which see the
bank and themselves) in one launch; sr_rope3d_qk_at gives recomputed history
rows their own frame times. Compared with the oracle's window_attention and
rope3d_at on the same bits: every row at small shapes, sampled rows and heads
at the 832x480 frame size (2072 prefix rows, 5 moving frames of 1560 tokens).
"""
import numpy as np
import pytest
import torch

import synthetic as syn
from oracle import OracleSession
from tests.gpu_common import LSE_ABS, assert_attention_close, assert_rotated_close, device, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from chunked_kv_cache_gb300 import build
    build.build()
    device()


def _pair(sh, dev, W=3):
    import chunked_kv_cache_gb300 as sr
    sk, sv = syn.session_sinks(sh, 11)
    gpu = sr.Session(sh.n_heads, sh.head_dim, sh.grid_h, sh.grid_w, sh.chunk_frames, W, sh.n_sink, sh.n_steps,
                     sink_k=to_dev(sk, dev), sink_v=to_dev(sv, dev), t_clock0=5, device=dev)
    ora = OracleSession(sh.n_heads, sh.head_dim, sh.grid_h, sh.grid_w, sh.chunk_frames, W, sh.n_sink, sh.n_steps,
                        sk, sv, t_clock0=5)
    return gpu, ora


SMALL = [syn.Shape("window tiny", 4, 64, 6, 10, 3, 3, 64),
         syn.Shape("window d128", 2, 128, 8, 16, 3, 3, 200)]


@pytest.mark.parametrize("sh", SMALL, ids=lambda s: s.name)
@pytest.mark.parametrize("with_prefix", [True, False])
@pytest.mark.parametrize("moving", [5, 4, 1])
def test_window_attention_small(sh, with_prefix, moving):
    dev = device()
    gpu, ora = _pair(sh, dev)
    T, S = sh.tokens_per_frame, sh.n_sink
    P = S if with_prefix else 0
    g = np.random.default_rng(moving + 10 * with_prefix)
    bits = lambda rows: syn.normal_bf16_bits((rows, sh.n_heads, sh.head_dim), g)
    for step in range(sh.n_steps):
        q, km, vm = bits(P + moving * T), bits(moving * T), bits(moving * T)
        o, lse = gpu.window_attention(step, to_dev(q, dev), to_dev(km, dev), to_dev(vm, dev), moving,
                                      with_prefix=with_prefix, lse=True)
        ref, ref_lse = ora.window_attention(step, q, km, vm, with_prefix)
        assert_attention_close(o.float().cpu().numpy().astype(np.float64), ref,
                               f"{sh.name} step {step} prefix {with_prefix} moving {moving}")
        assert np.abs(lse.cpu().numpy().astype(np.float64) - ref_lse).max() <= LSE_ABS
    assert gpu.error_status() == 0 and gpu.frames == 0
    gpu.close()


def test_window_attention_832x480_sampled():
    dev = device()
    base = syn.SHAPE_832x480
    gpu, _ = _pair(base, dev)
    heads = [3, 17]
    T, S, H, d = base.tokens_per_frame, base.n_sink, base.n_heads, base.head_dim
    M = 5 * T
    # the oracle follows two heads, with those heads' bank bits
    sk, sv = syn.session_sinks(base, 11)
    ora = OracleSession(len(heads), d, base.grid_h, base.grid_w, base.chunk_frames, 3, S, base.n_steps,
                        np.ascontiguousarray(sk[:, :, heads]), np.ascontiguousarray(sv[:, :, heads]), t_clock0=5)
    g = np.random.default_rng(7)
    q = syn.normal_bf16_bits((S + M, H, d), g)
    km = syn.normal_bf16_bits((M, H, d), g)
    vm = syn.normal_bf16_bits((M, H, d), g)
    o = gpu.window_attention(1, to_dev(q, dev), to_dev(km, dev), to_dev(vm, dev), 5, with_prefix=True)
    got = o.float().cpu().numpy()[:, heads].astype(np.float64)
    hb = lambda b: np.ascontiguousarray(b[:, heads])
    # every prefix row (cheap: 2072 keys), and a sample of moving rows
    mv = np.unique(np.concatenate([np.arange(0, 40), np.arange(M - 40, M), g.integers(0, M, 200)]))
    ref, _ = ora.window_attention(1, np.concatenate([hb(q)[:S], hb(q)[S + mv]]), hb(km), hb(vm), True)
    assert_attention_close(got[:S], ref[:S], "832x480 window, prefix rows")
    assert_attention_close(got[S + mv], ref[S:], "832x480 window, sampled moving rows")
    assert gpu.error_status() == 0
    gpu.close()


@pytest.mark.parametrize("first", [0, 7, 1000])
def test_rope3d_at_matches_oracle(first):
    dev = device()
    sh = SMALL[1]
    gpu, ora = _pair(sh, dev)
    g = np.random.default_rng(first)
    frames = 5
    q = syn.normal_bf16_bits((frames * sh.tokens_per_frame, sh.n_heads, sh.head_dim), g)
    k = syn.normal_bf16_bits((frames * sh.tokens_per_frame, sh.n_heads, sh.head_dim), g)
    qd, kd = to_dev(q, dev), to_dev(k, dev)
    gpu.rope3d_at(first, frames, qd, kd)
    qo, ko = ora.rope3d_at(first, frames, q, k)
    assert_rotated_close(syn.torch_to_bits(qd), qo, "q")
    assert_rotated_close(syn.torch_to_bits(kd), ko, "k")
    gpu.close()


def test_page_faithful_chunk_loop():
    # the pages' per-chunk computation: the moving rows (last h frames of history,
    # recomputed, then the chunk) are rotated at their own frame times and attend
    # over the bank and themselves; the ring path is not involved
    import chunked_kv_cache_gb300 as sr
    dev = device()
    sh = SMALL[0]
    gpu, ora = _pair(sh, dev)
    T = sh.tokens_per_frame
    g = np.random.default_rng(21)
    frame = 9                                      # after the 9-latent first window
    for c in range(1, 7):
        plan = sr.plan_chunk(c)
        h, F = plan["hist_frames"], plan["n_frames"]
        assert plan["first_frame"] == frame
        moving = h + F
        for step in range(sh.n_steps):
            q, k, v = (syn.normal_bf16_bits((moving * T, sh.n_heads, sh.head_dim), g) for _ in range(3))
            qd, kd = to_dev(q, dev), to_dev(k, dev)
            gpu.rope3d_at(frame - h, moving, qd, kd)
            qo, ko = ora.rope3d_at(frame - h, moving, q, k)
            o = gpu.window_attention(step, qd, kd, to_dev(v, dev), moving)
            ref, _ = ora.window_attention(step, qo, ko, v, False)
            assert_attention_close(o.float().cpu().numpy().astype(np.float64), ref, f"chunk {c} step {step}")
        frame += F
    assert gpu.error_status() == 0
    gpu.close()
