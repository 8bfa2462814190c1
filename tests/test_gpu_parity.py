"""GPU parity: the CUDA library (through the C ABI) against the float64 oracle
on the same seeded inputs. Gates: attention max-abs <= 2e-2, mean-abs <= 2e-3
and relative rms <= 1e-2 on bf16 outputs; ring K within 1 bf16 ulp, ring V
and the slot table bit-exact."""
import numpy as np
import pytest
import torch

import synthetic as syn
from tests.gpu_common import (Twin, assert_attention_close, assert_rotated_close, device, to_dev, LSE_ABS)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from chunked_kv_cache_gb300 import build
    build.build()
    device()


# ------------------------------------------------------------------ RoPE / commit

@pytest.mark.parametrize("config,fill,clock", [(1, 0, 0), (1, 3, 7), (1, 2, 123457), (2, 6, 0), (2, 2, 1000)])
def test_rope3d_qk_matches_oracle(config, fill, clock):
    shape = syn.SHAPES[config]
    tw = Twin(shape, config, fill=fill, t_clock0=clock)
    x = syn.chunk_inputs(shape, config, chunk=fill)
    q, k = to_dev(x.q[0], tw.dev), to_dev(x.k[0], tw.dev)
    tw.gpu.rope3d_qk(q, k)
    qo, ko = tw.ora.rope3d_qk(x.q[0], x.k[0])
    for name, g, o in (("q", q, qo), ("k", k, ko)):
        assert_rotated_close(syn.torch_to_bits(g), o, name)


def test_rope3d_single_tensor_rotates_once():
    shape = syn.TINY
    tw = Twin(shape, 1)
    x = syn.chunk_inputs(shape, 1)
    q = to_dev(x.q[0], tw.dev)
    k = to_dev(x.k[0], tw.dev)
    q2, k2 = q.clone(), k.clone()
    tw.gpu.rope3d_qk(q, k)
    tw.gpu.rope3d_qk(q2, None)
    tw.gpu.rope3d_qk(None, k2)
    assert torch.equal(q, q2) and torch.equal(k, k2)


@pytest.mark.parametrize("config,fill,chunks,clock", [(1, 0, 5, 0), (1, 3, 4, 11), (2, 0, 4, 0), (2, 5, 2, 100)])
def test_cache_commit_matches_oracle(config, fill, chunks, clock):
    shape = syn.SHAPES[config]
    tw = Twin(shape, config, fill=fill, t_clock0=clock)
    for c in range(chunks):
        x = syn.chunk_inputs(shape, config, chunk=100 + c)
        tw.commit(x)
        torch.cuda.synchronize()
        assert tw.gpu.frames == tw.ora.n_committed
        assert np.array_equal(tw.gpu.slot_frame.cpu().numpy(), tw.ora.ring.slot_frame.astype(np.int32))
    rk, rv = tw.ring_bits()
    ok_, ov_ = tw.ora.ring_bits()
    occupied = np.repeat(tw.ora.ring.slot_frame >= 0, shape.tokens_per_frame)
    assert np.array_equal(rv[occupied], ov_[occupied])                    # V is a copy
    assert_rotated_close(rk[occupied], ok_[occupied], "ring K")
    # slots never written keep the NaN canary of the synthetic prefill
    assert np.all(rk[~occupied] == 0x7FC0) and np.all(rv[~occupied] == 0x7FC0)
    assert tw.gpu.error_status() == 0


ODD_SHAPES = [
    # (heads, d, grid_h, grid_w, F, W): 16-byte vectors per token 8 .. 80, frames
    # that do not divide a copy chunk, a single token per frame
    (1, 64, 5, 7, 3, 4),
    (5, 128, 7, 9, 2, 3),
    (3, 64, 1, 1, 2, 5),
    (2, 128, 13, 29, 2, 2),
]


@pytest.mark.parametrize("H,d,gh,gw,F,W", ODD_SHAPES)
def test_rope_and_commit_odd_shapes(H, d, gh, gw, F, W):
    shape = syn.Shape(f"odd {H}x{d} {gh}x{gw}", H, d, gh, gw, F, W, 16)
    tw = Twin(shape, 1, fill=0, t_clock0=5)
    for c in range(4):   # past one wrap of the ring
        x = syn.chunk_inputs(shape, 1, chunk=200 + c)
        q, k = to_dev(x.q[0], tw.dev), to_dev(x.k[0], tw.dev)
        tw.gpu.rope3d_qk(q, k)
        qo, ko = tw.ora.rope3d_qk(x.q[0], x.k[0])
        assert_rotated_close(syn.torch_to_bits(q), qo, "q")
        assert_rotated_close(syn.torch_to_bits(k), ko, "k")
        tw.commit(x)
        torch.cuda.synchronize()
        assert tw.gpu.frames == tw.ora.n_committed
        assert np.array_equal(tw.gpu.slot_frame.cpu().numpy(), tw.ora.ring.slot_frame.astype(np.int32))
    rk, rv = tw.ring_bits()
    ok_, ov_ = tw.ora.ring_bits()
    occupied = np.repeat(tw.ora.ring.slot_frame >= 0, shape.tokens_per_frame)
    assert np.array_equal(rv[occupied], ov_[occupied])
    assert_rotated_close(rk[occupied], ok_[occupied], "ring K")
    assert tw.gpu.error_status() == 0


# ------------------------------------------------------------------ attention

@pytest.mark.parametrize("fill", [0, 1, 3, 4])
@pytest.mark.parametrize("step", [0, 1])
def test_attention_tiny(fill, step):
    shape = syn.TINY
    tw = Twin(shape, 1, fill=fill)
    x = syn.chunk_inputs(shape, 1, chunk=fill)
    got, ref, gl, rl = tw.step(x, step, lse=True)
    assert_attention_close(got, ref, f"tiny fill={fill} step={step}")
    assert np.abs(gl - rl).max() <= LSE_ABS


@pytest.mark.parametrize("fill", [6, 0])
def test_attention_832x480_full(fill):
    shape = syn.SHAPE_832x480
    tw = Twin(shape, 2, fill=fill)
    x = syn.chunk_inputs(shape, 2, chunk=7)
    got, ref, gl, rl = tw.step(x, 1, lse=True)
    assert_attention_close(got, ref, f"832x480 fill={fill}")
    assert np.abs(gl - rl).max() <= LSE_ABS


@pytest.mark.parametrize("gh,gw", [
    (8, 16),    # Lq 256: one block of two tiles, no last-block units
    (10, 16),   # Lq 320: a single-tile last block of 64 rows
    (12, 16),   # Lq 384: a single-tile last block of exactly 128 rows
    (13, 16),   # Lq 416: a last block of two tiles (128 + 32 rows) runs as a whole block
    (16, 32),   # Lq 1024: four whole blocks per head, side by side
])
@pytest.mark.parametrize("workspace", [True, False])
def test_attention_block_shapes(gh, gw, workspace):
    shape = syn.Shape(f"blocks {gh}x{gw}", 3, 128, gh, gw, 2, 2, 40)
    tw = Twin(shape, 1, fill=2, workspace=workspace)
    x = syn.chunk_inputs(shape, 1, chunk=3)
    got, ref, gl, rl = tw.step(x, 0, lse=True)
    assert_attention_close(got, ref, f"blocks {gh}x{gw}")
    assert np.abs(gl - rl).max() <= LSE_ABS
    assert tw.gpu.error_status() == 0


def _edge_rows(lq):
    base = [0, 1, 126, 127, 128, 129, 255, 256, 257, 511, 512, lq // 2, lq - 129, lq - 128, lq - 2, lq - 1]
    rng = np.random.default_rng(5)
    return sorted(set([r for r in base if 0 <= r < lq] + list(rng.choice(lq, 48, replace=False))))


@pytest.mark.parametrize("fill", [8, 3])
def test_attention_720p_sampled(fill):
    shape = syn.SHAPE_720P
    tw = Twin(shape, 3, fill=fill, heads=[0, 17, 39])
    x = syn.chunk_inputs(shape, 3, chunk=2)
    rows = _edge_rows(shape.lq)
    got, ref, gl, rl = tw.step(x, 0, rows=rows, lse=True)
    assert_attention_close(got, ref, f"720p fill={fill}")
    assert np.abs(gl - rl).max() <= LSE_ABS


@pytest.mark.parametrize("config", [1, 2])
def test_attention_peaky(config):
    # scaled queries plus planted dominant keys: exercises the running-max
    # rescale of the online softmax
    shape = syn.SHAPES[config]
    tw = Twin(shape, config, fill=shape.window_frames, heads=None if config == 1 else [3, 11])
    x = syn.chunk_inputs(shape, config, chunk=3, q_scale=4.0)
    for s in range(shape.n_steps):
        x.k[s] = syn.plant_keys(x.q[s], x.k[s], every=37, gain=3.0)
    rows = None if config == 1 else _edge_rows(shape.lq)
    got, ref, _, _ = tw.step(x, 0, rows=rows)
    assert_attention_close(got, ref, f"peaky config {config}")


@pytest.mark.parametrize("S,W,fill", [(0, 4, 4), (64, 0, 0), (0, 0, 0), (3, 4, 2)])
def test_attention_degenerate_windows(S, W, fill):
    shape = syn.TINY
    tw = Twin(shape, 1, fill=fill, n_sink=S, window_frames=W)
    x = syn.chunk_inputs(shape, 1, chunk=1)
    got, ref, _, _ = tw.step(x, 1)
    assert_attention_close(got, ref, f"S={S} W={W} fill={fill}")


def test_attention_single_key_is_exact():
    # one token per frame, one frame per chunk, no sinks, no history: every
    # query sees exactly one key, so O equals that key's value exactly
    import chunked_kv_cache_gb300 as sr
    dev = device()
    for d in (64, 128):
        s = sr.Session(3, d, 1, 1, 1, 0, 0, 1, device=dev)
        g = np.random.default_rng(d)
        q, k, v = (torch.from_numpy(g.standard_normal((1, 3, d)).astype(np.float32)).to(torch.bfloat16).to(dev)
                   for _ in range(3))
        o = s.chunk_attention(0, q, k, v)
        assert torch.equal(o, v)


def test_attention_is_deterministic_and_bank_per_step():
    shape = syn.TINY
    tw = Twin(shape, 1, fill=4)
    x = syn.chunk_inputs(shape, 1)
    q, k, v = (to_dev(b, tw.dev) for b in (x.q[0], x.k[0], x.v[0]))
    o1 = tw.gpu.chunk_attention(0, q, k, v)
    o2 = tw.gpu.chunk_attention(0, q, k, v)
    o3 = tw.gpu.chunk_attention(1, q, k, v)
    assert torch.equal(o1, o2)
    assert not torch.equal(o1, o3)


def test_evicted_frames_give_bit_identical_output():
    shape = syn.TINY
    a = Twin(shape, 1)
    b = Twin(shape, 1)
    for c in range(4):
        xa = syn.chunk_inputs(shape, 1, chunk=c)
        xb = syn.chunk_inputs(shape, 1, chunk=c + 50) if c == 0 else xa
        a.commit(xa)
        b.commit(xb)
    x = syn.chunk_inputs(shape, 1, chunk=9)
    oa, *_ = a.step(x, 0)
    ob, *_ = b.step(x, 0)
    assert np.array_equal(oa, ob)


def test_checkpoint_and_resume_continue_bit_for_bit():
    # A session's state is its sink banks, ring, slot table and frame count. A
    # session built from copies of them (the count through sr_session_restore)
    # continues bit for bit: same outputs, same ring, same slot table.
    import chunked_kv_cache_gb300 as sr
    shape = syn.TINY
    a = Twin(shape, 1)
    for c in range(5):      # 10 frames through a 4-frame ring: the ring has wrapped
        a.commit(syn.chunk_inputs(shape, 1, chunk=c))
    g = a.gpu
    b = sr.Session(shape.n_heads, shape.head_dim, shape.grid_h, shape.grid_w, shape.chunk_frames,
                   shape.window_frames, shape.n_sink, shape.n_steps, sink_k=g.sink_k.clone(),
                   sink_v=g.sink_v.clone(), device=a.dev)
    b.ring_k.copy_(g.ring_k)
    b.ring_v.copy_(g.ring_v)
    b.slot_frame.copy_(g.slot_frame)
    b.restore(g.frames)
    assert b.frames == g.frames == 10
    for c in range(5, 8):
        x = syn.chunk_inputs(shape, 1, chunk=c)
        for st in range(shape.n_steps):
            q, k, v = to_dev(x.q[st], a.dev), to_dev(x.k[st], a.dev), to_dev(x.v[st], a.dev)
            q2, k2 = q.clone(), k.clone()
            g.rope3d_qk(q, k)
            b.rope3d_qk(q2, k2)
            assert torch.equal(g.chunk_attention(st, q, k, v), b.chunk_attention(st, q2, k2, v))
        ck, cv = to_dev(x.clean_k, a.dev), to_dev(x.clean_v, a.dev)
        g.cache_commit(ck, cv)
        b.cache_commit(ck, cv)
    assert torch.equal(g.ring_k, b.ring_k) and torch.equal(g.ring_v, b.ring_v)
    assert torch.equal(g.slot_frame, b.slot_frame)
    assert b.frames == g.frames == 16
    assert g.error_status() == 0 and b.error_status() == 0


def test_clock_shift_invariance_without_sinks():
    shape = syn.TINY
    outs = []
    for clock in (0, 100, 1000):
        tw = Twin(shape, 1, n_sink=0, t_clock0=clock)
        for c in range(3):
            tw.commit(syn.chunk_inputs(shape, 1, chunk=c))
        got, ref, _, _ = tw.step(syn.chunk_inputs(shape, 1, chunk=5), 0)
        assert_attention_close(got, ref, f"clock {clock}")
        outs.append(got)
    # equal up to the bf16 rounding of keys rotated at other absolute angles
    assert np.abs(outs[0] - outs[1]).max() <= 2e-2 and np.abs(outs[0] - outs[2]).max() <= 2e-2


# ------------------------------------------------------------------ key-split last blocks

@pytest.mark.parametrize("k", [1, 2, 3, 4])
def test_key_split_last_block_832x480(k):
    # rows 3072..3119 form a single-tile last block per head; its key range is
    # spread over k CTAs whose partial results the last one merges
    shape = syn.SHAPE_832x480
    tw = Twin(shape, 2, fill=6, heads=[1, 22], tail_split=k)
    x = syn.chunk_inputs(shape, 2, chunk=11)
    rows = sorted(set(list(range(3072, 3120)) + [0, 255, 3071]))
    for rep in range(2):      # a second call exercises the next epoch of the arrival counters
        got, ref, gl, rl = tw.step(x, 0, rows=rows, lse=True)
        assert_attention_close(got, ref, f"key split {k}, call {rep}")
        assert np.abs(gl - rl).max() <= LSE_ABS


@pytest.mark.parametrize("k", [2, 3, 4])
def test_key_split_tiny_all_units_split(k):
    # Lq = 120: every unit is a single-tile block; with 4 key tiles and k = 4 each
    # part walks one tile and its second softmax group has nothing to do
    shape = syn.TINY
    tw = Twin(shape, 1, fill=4, tail_split=k)
    x = syn.chunk_inputs(shape, 1, chunk=2)
    got, ref, gl, rl = tw.step(x, 1, lse=True)
    assert_attention_close(got, ref, f"tiny key split {k}")
    assert np.abs(gl - rl).max() <= LSE_ABS


def test_key_split_needs_workspace():
    # without a workspace the split is off and results still match
    shape = syn.TINY
    tw = Twin(shape, 1, fill=2, tail_split=4, workspace=False)
    got, ref, _, _ = tw.step(syn.chunk_inputs(shape, 1, chunk=3), 0)
    assert_attention_close(got, ref, "no workspace")


# ------------------------------------------------------------------ multi-session batch

def test_batch_matches_single_and_oracle():
    import chunked_kv_cache_gb300 as sr
    shape = syn.SHAPE_832x480
    # a fixed key split of the last blocks, so that batch and single calls run the same parts
    twins = [Twin(shape, 5, fill=f, session=i, heads=[0, 13], tail_split=2) for i, f in enumerate(syn.BATCH_FILLS)]
    xs = [syn.chunk_inputs(shape, 5, session=i) for i in range(len(twins))]
    dev = twins[0].dev
    step = 1
    qs, ks, vs = [], [], []
    for tw, x in zip(twins, xs):
        q, k = to_dev(x.q[step], dev), to_dev(x.k[step], dev)
        tw.gpu.rope3d_qk(q, k)
        qs.append(q), ks.append(k), vs.append(to_dev(x.v[step], dev))
    Q, K, V = torch.cat(qs), torch.cat(ks), torch.cat(vs)
    O, L = sr.chunk_attention_batch([t.gpu for t in twins], step, Q, K, V, lse=True)
    lq = shape.lq
    rows = _edge_rows(lq)
    for i, (tw, x) in enumerate(zip(twins, xs)):
        single, sl = tw.gpu.chunk_attention(step, qs[i], ks[i], vs[i], lse=True)
        assert torch.equal(O[i * lq:(i + 1) * lq], single)          # same tiles, same order
        assert torch.equal(L[:, i * lq:(i + 1) * lq], sl)
        qo, ko = tw.ora.rope3d_qk(tw.oh(x.q[step]), tw.oh(x.k[step]))
        ref, _ = tw.ora.chunk_attention(step, qo, ko, tw.oh(x.v[step]), rows=rows)
        got = single.float().cpu().numpy()[:, tw.heads][rows]
        assert_attention_close(got, ref, f"batch session {i}")


# ------------------------------------------------------------------ long session

def test_long_session_240_chunks():
    # 240 consecutive chunks from an empty ring; inputs drawn on the device
    # (the oracle follows two heads, fed the same bits of those heads)
    shape = syn.SHAPE_832x480
    heads = [5, 20]
    tw = Twin(shape, 4, heads=heads)
    dev = tw.dev
    rows = _edge_rows(shape.lq)[::3]
    n_chunks = syn.LONG_SESSION_CHUNKS
    checkpoints = set(range(5)) | set(range(0, n_chunks, 40)) | {n_chunks - 1}
    hb = lambda t: syn.torch_to_bits(t[:, heads])
    for c in range(n_chunks):
        x = syn.chunk_inputs_device(shape, 4, dev, chunk=c, with_steps=c in checkpoints)
        if c in checkpoints:
            for s in range(shape.n_steps):
                q, k, v = x["q"][s], x["k"][s], x["v"][s]
                qh, kh, vh = hb(q), hb(k), hb(v)
                tw.gpu.rope3d_qk(q, k)
                o = tw.gpu.chunk_attention(s, q, k, v)
                qo, ko = tw.ora.rope3d_qk(qh, kh)
                ref, _ = tw.ora.chunk_attention(s, qo, ko, vh, rows=rows)
                got = o.float().cpu().numpy()[:, heads][rows]
                assert_attention_close(got, ref, f"long session chunk {c} step {s}")
        tw.gpu.cache_commit(x["clean_k"], x["clean_v"])
        tw.ora.cache_commit(hb(x["clean_k"]), hb(x["clean_v"]))
        slots = tw.gpu.slot_frame.cpu().numpy()
        assert np.array_equal(slots, tw.ora.ring.slot_frame.astype(np.int32)), f"chunk {c}"
    rk, rv = tw.ring_bits()
    ok_, ov_ = tw.ora.ring_bits()
    assert np.array_equal(rv, ov_)
    assert_rotated_close(rk, ok_, "ring K after 240 chunks")
    assert tw.gpu.frames == 2 * n_chunks
    assert tw.gpu.error_status() == 0


# ------------------------------------------------------------------ failure detection

def test_bounded_wait_reports_timeout_and_context_survives():
    import chunked_kv_cache_gb300 as sr
    from chunked_kv_cache_gb300 import _native as N
    dev = device()
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    sr.sr_debug_wait_timeout(err.data_ptr(), 2_000_000, torch.cuda.current_stream(dev).cuda_stream)
    torch.cuda.synchronize()
    code = int(err.item())
    assert code == (N.SR_DEVERR_WAIT_TIMEOUT | (0xFF << 8))
    assert sr.sr_device_error_status(code) == N.SR_ERR_TIMEOUT
    # the context is still usable afterwards
    test_attention_tiny(4, 0)
