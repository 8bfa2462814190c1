"""Seeded random shapes through the whole chunk path, against the float64 oracle.

Each case draws a session shape (heads, head dim 64 or 128, latent grid, chunk
frames, ring frames, sink tokens, steps, clock, workspace and key split) and
runs several chunks of it from a partly filled ring: RoPE-3D on both steps'
Q and K, both steps' attention (with LSE), and the ring commit, comparing the
rotated values, the outputs, the LSE, the ring and the slot table with the
oracle after every chunk. The shapes are small enough for the oracle to follow
every head and row, and mixed enough to reach tiles that straddle segment ends,
single-tile last blocks, rings that wrap and empty key segments. A second
test packs several random sessions of one head shape into one batched launch,
and a third runs chunks of random frame counts with random history windows
through the variable-length and the device-state calls.
"""
import numpy as np
import pytest
import torch

import synthetic as syn
from tests.gpu_common import (LSE_ABS, Twin, assert_attention_close, assert_rotated_close, device, to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from chunked_kv_cache_gb300 import build
    build.build()
    device()


def _draw_shape(rng, case):
    d = int(rng.choice([64, 128]))
    H = int(rng.integers(1, 5))
    gh, gw = int(rng.integers(1, 13)), int(rng.integers(1, 17))
    F = int(rng.integers(1, 4))
    W = int(rng.choice([0, F, F + 1, 2 * F + 1]))
    S = int(rng.choice([0, 1, 37, 128, 200]))
    steps = int(rng.integers(1, 3))
    return syn.Shape(f"fuzz {case}", H, d, gh, gw, F, W, S, steps)


@pytest.mark.parametrize("case", range(96))
def test_random_session_shapes_match_oracle(case):
    rng = np.random.default_rng(1000 + case)
    shape = _draw_shape(rng, case)
    fill = int(rng.integers(0, shape.window_frames + 1)) if shape.window_frames else 0
    clock = int(rng.choice([0, 9, -5, 2 ** 24 + 1]))
    workspace = bool(rng.random() < 0.7)
    split = int(rng.choice([0, 1, 2, 4]))
    tw = Twin(shape, 6, fill=fill, session=case, t_clock0=clock, workspace=workspace, tail_split=split)
    for c in range(3):
        x = syn.chunk_inputs(shape, 6, session=case, chunk=c)
        for st in range(shape.n_steps):
            q, k = to_dev(x.q[st], tw.dev), to_dev(x.k[st], tw.dev)
            tw.gpu.rope3d_qk(q, k)
            qo, ko = tw.ora.rope3d_qk(x.q[st], x.k[st])
            assert_rotated_close(syn.torch_to_bits(q), qo, f"{shape.name} chunk {c} q")
            assert_rotated_close(syn.torch_to_bits(k), ko, f"{shape.name} chunk {c} k")
            o, lse = tw.gpu.chunk_attention(st, q, k, to_dev(x.v[st], tw.dev), lse=True)
            ref, ref_lse = tw.ora.chunk_attention(st, qo, ko, x.v[st])
            what = f"{shape.name} (H={shape.n_heads} d={shape.head_dim} grid={shape.grid_h}x{shape.grid_w} " \
                   f"F={shape.chunk_frames} W={shape.window_frames} S={shape.n_sink} fill={fill}) chunk {c} step {st}"
            assert_attention_close(o.float().cpu().numpy(), ref, what)
            assert np.abs(lse.cpu().numpy().astype(np.float64) - ref_lse).max() <= LSE_ABS, what
        tw.commit(x)
        torch.cuda.synchronize()
        assert tw.gpu.frames == tw.ora.n_committed
        if shape.window_frames:
            assert np.array_equal(tw.gpu.slot_frame.cpu().numpy(), tw.ora.ring.slot_frame.astype(np.int32))
            rk, rv = tw.ring_bits()
            ok_, ov_ = tw.ora.ring_bits()
            occ = np.repeat(tw.ora.ring.slot_frame >= 0, shape.tokens_per_frame)
            assert np.array_equal(rv[occ], ov_[occ])
            assert_rotated_close(rk[occ], ok_[occ], f"{shape.name} ring K")
    assert tw.gpu.error_status() == 0


@pytest.mark.parametrize("case", range(24))
def test_random_batches_match_single_calls_and_oracle(case):
    import chunked_kv_cache_gb300 as sr
    rng = np.random.default_rng(2000 + case)
    H, d = int(rng.integers(1, 4)), int(rng.choice([64, 128]))
    n = int(rng.integers(2, 7))
    twins, xs = [], []
    for i in range(n):
        gh, gw, F = int(rng.integers(1, 11)), int(rng.integers(1, 13)), int(rng.integers(1, 3))
        W = int(rng.choice([0, F, 2 * F]))
        shape = syn.Shape(f"batch {case}.{i}", H, d, gh, gw, F, W, int(rng.choice([0, 64, 150])), 1)
        fill = int(rng.integers(0, W + 1)) if W else 0
        twins.append(Twin(shape, 7, fill=fill, session=10 * case + i, tail_split=1))
        xs.append(syn.chunk_inputs(shape, 7, session=10 * case + i))
    dev = twins[0].dev
    qs, ks, vs = [], [], []
    for tw, x in zip(twins, xs):
        q, k = to_dev(x.q[0], dev), to_dev(x.k[0], dev)
        tw.gpu.rope3d_qk(q, k)
        qs.append(q), ks.append(k), vs.append(to_dev(x.v[0], dev))
    O, L = sr.chunk_attention_batch([t.gpu for t in twins], 0, torch.cat(qs), torch.cat(ks), torch.cat(vs), lse=True)
    row = 0
    for i, (tw, x) in enumerate(zip(twins, xs)):
        lq = tw.sh.lq
        single, sl = tw.gpu.chunk_attention(0, qs[i], ks[i], vs[i], lse=True)
        assert torch.equal(O[row:row + lq], single), f"case {case} session {i}"
        assert torch.equal(L[:, row:row + lq], sl)
        qo, ko = tw.ora.rope3d_qk(x.q[0], x.k[0])
        ref, _ = tw.ora.chunk_attention(0, qo, ko, x.v[0])
        assert_attention_close(single.float().cpu().numpy(), ref, f"batch case {case} session {i}")
        row += lq
    for tw in twins:
        assert tw.gpu.error_status() == 0


@pytest.mark.parametrize("case", range(24))
@pytest.mark.parametrize("device_state", [False, True])
def test_random_frame_counts_and_history_windows_match_oracle(case, device_state):
    """Chunks of 1 to 5 frames with random visible-history windows through the
    *_frames calls (host state) or the *_dev calls (frame count on the device),
    so that commits longer than the ring and history windows that wrap around
    its end both occur."""
    import chunked_kv_cache_gb300 as sr
    from oracle import OracleSession
    rng = np.random.default_rng(3000 + case)
    dev = device()
    H, d = int(rng.integers(1, 4)), int(rng.choice([64, 128]))
    gh, gw = int(rng.integers(1, 9)), int(rng.integers(1, 11))
    W = int(rng.integers(2, 6))
    S = int(rng.choice([0, 33, 128]))
    sh = syn.Shape(f"frames {case}", H, d, gh, gw, 2, W, S, 2)
    sk, sv = syn.session_sinks(sh, 8, case)
    gpu = sr.Session(H, d, gh, gw, 2, W, S, 2, sink_k=to_dev(sk, dev) if S else None,
                     sink_v=to_dev(sv, dev) if S else None, t_clock0=7, device_state=device_state, device=dev)
    ora = OracleSession(H, d, gh, gw, 2, W, S, 2, sk, sv, t_clock0=7)
    for c in range(8):
        F = int(rng.integers(1, 6))
        n = ora.n_committed
        occupied = min(n, W)
        h = int(rng.integers(0, occupied + 1))
        x = syn.chunk_inputs(sh, 8, session=case, chunk=c, frames=F)
        for s in range(2):
            q, k, v = to_dev(x.q[s], dev), to_dev(x.k[s], dev), to_dev(x.v[s], dev)
            if device_state:
                gpu.rope3d_qk_dev(q, k, F)
                lse = torch.empty((H, F * gh * gw), dtype=torch.float32, device=dev)
                o = gpu.chunk_attention_dev(s, q, k, v, F, h, lse=lse)
            else:
                gpu.rope3d_qk(q, k, frames=F)
                o, lse = gpu.chunk_attention(s, q, k, v, lse=True, frames=F, hist=h)
            qo, ko = ora.rope3d_qk(x.q[s], x.k[s], frames=F)
            assert_rotated_close(syn.torch_to_bits(q), qo, f"case {case} chunk {c} step {s} q")
            ref, ref_lse = ora.chunk_attention(s, qo, ko, x.v[s], hist=h)
            what = f"case {case} (H={H} d={d} {gh}x{gw} W={W} S={S}) chunk {c} F={F} n={n} hist={h} step {s}"
            assert_attention_close(o.float().cpu().numpy(), ref, what)
            assert np.abs(lse.cpu().numpy().astype(np.float64) - ref_lse).max() <= LSE_ABS, what
        if device_state:
            gpu.cache_commit_dev(to_dev(x.clean_k, dev), to_dev(x.clean_v, dev), F)
        else:
            gpu.cache_commit(to_dev(x.clean_k, dev), to_dev(x.clean_v, dev), frames=F)
        ora.cache_commit(x.clean_k, x.clean_v, frames=F)
        torch.cuda.synchronize()
        assert np.array_equal(gpu.slot_frame.cpu().numpy(), ora.ring.slot_frame.astype(np.int32)), f"case {case} chunk {c}"
        if device_state:
            assert int(gpu.frame_counter.item()) == ora.n_committed
    occ = np.repeat(ora.ring.slot_frame >= 0, sh.tokens_per_frame)
    rk, rv = syn.torch_to_bits(gpu.ring_k), syn.torch_to_bits(gpu.ring_v)
    ok_, ov_ = ora.ring_bits()
    assert np.array_equal(rv[occ], ov_[occ])
    assert_rotated_close(rk[occ], ok_[occ], f"case {case} ring K")
    assert gpu.error_status() == 0
    gpu.close()


@pytest.mark.parametrize("case", range(30))
def test_random_decoder_layers_match_oracle(case):
    """Random latent grids, window sizes, shifts, chunk lengths and cache depths
    through a decoder layer's three launches (gather + RoPE, batched attention,
    commit), against the oracle's whole-frame layer."""
    from chunked_kv_cache_gb300.decoder import DecoderWindowLayer
    from oracle.decoder import DecoderLayerOracle
    rng = np.random.default_rng(4000 + case)
    dev = device()
    H, d = int(rng.integers(1, 4)), int(rng.choice([64, 128]))
    window = int(rng.choice([4, 8, 16]))
    gh, gw = int(rng.integers(window // 2 + 1, 25)), int(rng.integers(window // 2 + 1, 25))
    shifted = bool(rng.random() < 0.5)
    F = int(rng.integers(1, 4))
    C = int(rng.choice([0, F, 2 * F]))
    G = int(rng.choice([1, 5]))
    lay = DecoderWindowLayer(gh, gw, H, d, G, window=window, shifted=shifted, chunk_frames=F, cache_frames=C,
                             t_clock0=11, device=dev)
    ora = DecoderLayerOracle(gh, gw, window, shifted, H, d, cache_frames=C, t_clock0=11)
    idx = lay.packing_index().numpy()
    bits = lambda b: torch.from_numpy(b.view(np.int16)).to(dev).view(torch.bfloat16)
    for c in range(3):
        q, k, v, ck, cv = (syn.normal_bf16_bits((F, gh, gw, H, d), rng) for _ in range(5))
        gk, gv = syn.normal_bf16_bits((G, H, d), rng), syn.normal_bf16_bits((G, H, d), rng)
        lay.set_global(bits(gk), bits(gv))
        qp, kp, vp = lay.gather_rope(bits(q), bits(k), bits(v))
        o = lay.attention(qp, kp, vp)
        lay.commit(bits(ck), bits(cv))
        ref = ora.step(q, k, v, gk, gv)
        ora.commit(ck, cv)
        got = np.empty((F * gh * gw, H, d))
        got[idx] = o.float().cpu().numpy()
        what = f"case {case}: {gh}x{gw} window {window} shifted={shifted} F={F} C={C} H={H} d={d} G={G} chunk {c}"
        assert_attention_close(got, ref.reshape(-1, H, d), what)
    assert lay.error_status() == 0
    lay.close()


@pytest.mark.parametrize("case", range(24))
def test_random_page_faithful_windows_match_oracle(case):
    """The page-faithful window on random shapes: prefix rows over the bank of
    the step alone and moving rows (1 to 5 frames) over the bank and
    themselves, in one launch, with and without a workspace (persistent or one
    unit per CTA), against the oracle's window_attention."""
    import chunked_kv_cache_gb300 as sr
    from oracle import OracleSession
    rng = np.random.default_rng(5000 + case)
    d = int(rng.choice([64, 128]))
    H = int(rng.integers(1, 5))
    gh, gw = int(rng.integers(1, 13)), int(rng.integers(1, 17))
    S = int(rng.choice([1, 37, 128, 200, 300]))
    steps = int(rng.integers(1, 3))
    sh = syn.Shape(f"window fuzz {case}", H, d, gh, gw, 3, 3, S, steps)
    moving = int(rng.integers(1, 6))
    with_prefix = bool(rng.random() < 0.6)
    workspace = bool(rng.random() < 0.7)
    dev = device()
    sk, sv = syn.session_sinks(sh, 11 + case)
    gpu = sr.Session(H, d, gh, gw, sh.chunk_frames, sh.window_frames, S, steps, sink_k=to_dev(sk, dev),
                     sink_v=to_dev(sv, dev), t_clock0=5, workspace=workspace, device=dev)
    ora = OracleSession(H, d, gh, gw, sh.chunk_frames, sh.window_frames, S, steps, sk, sv, t_clock0=5)
    T = gh * gw
    P = S if with_prefix else 0
    for step in range(steps):
        q, km, vm = (syn.normal_bf16_bits((rows, H, d), rng) for rows in (P + moving * T, moving * T, moving * T))
        o, lse = gpu.window_attention(step, to_dev(q, dev), to_dev(km, dev), to_dev(vm, dev), moving,
                                      with_prefix=with_prefix, lse=True)
        ref, ref_lse = ora.window_attention(step, q, km, vm, with_prefix)
        assert_attention_close(o.float().cpu().numpy().astype(np.float64), ref,
                               f"{sh.name} step {step} prefix {with_prefix} moving {moving}")
        assert np.abs(lse.cpu().numpy().astype(np.float64) - ref_lse).max() <= LSE_ABS
    assert gpu.error_status() == 0
    gpu.close()
