"""The allocation-free chunk attention, sr_chunk_attention_noalloc.

It exists for callers that cannot allocate device memory, such as code that
runs inside a framework's fixed memory pool or a plugin that is handed only a
stream and its tensors: they cannot provide the session workspace that the key
split of a chunk's last query block uses, so this entry point takes its scratch
from an array built into the library instead.

Checked here, through the C ABI, on two calls in a row with the key split
forced on (so the built-in scratch is really used, and reused by the second
call): the output against the float64 oracle within the attention tolerances
of the parity tests, and bit for bit against sr_chunk_attention on a twin
session that has its own workspace and the same forced split (the same plan,
so the same arithmetic); and the same two checks on twelve random session
shapes with forced splits of 1, 2 or 4 parts. A session too large for the
scratch is refused before anything runs. This file is collected last on
purpose.
"""
import numpy as np
import pytest
import torch

import synthetic as syn
from tests.gpu_common import LSE_ABS, Twin, assert_attention_close, device, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from chunked_kv_cache_gb300 import build
    build.build()
    device()


def _edge_rows(lq):
    # both query tiles of the first and last blocks, the rows around the
    # single-tile last block (3120 = 12 * 256 + 48 rows), and a random sample
    base = [0, 1, 127, 128, 255, 256, 1537, lq - 49, lq - 48, lq - 47, lq - 2, lq - 1]
    rng = np.random.default_rng(11)
    return sorted(set(base + [int(r) for r in rng.choice(lq, 40, replace=False)]))


def test_noalloc_matches_oracle_and_sr_chunk_attention_twice():
    from chunked_kv_cache_gb300 import _native as N
    shape = syn.SHAPE_832x480
    heads = [0, 13]
    fill = shape.window_frames
    # the allocation-free session: no workspace of its own, last blocks forced into 4 key parts
    tw = Twin(shape, 2, fill=fill, heads=heads, tail_split=4, workspace=False)
    # its twin with a workspace and the same split, for the bit-for-bit check
    twin = Twin(shape, 2, fill=fill, heads=heads, tail_split=4, workspace=True)
    dev = tw.dev
    x = syn.chunk_inputs(shape, 2, chunk=5)
    q, k, v = (to_dev(b, dev) for b in (x.q[0], x.k[0], x.v[0]))
    tw.gpu.rope3d_qk(q, k)                     # both sessions are at the same frame count
    qo, ko = tw.ora.rope3d_qk(tw.oh(x.q[0]), tw.oh(x.k[0]))
    rows = _edge_rows(shape.lq)
    ref, ref_lse = tw.ora.chunk_attention(0, qo, ko, tw.oh(x.v[0]), rows=rows)
    stream = torch.cuda.current_stream(dev).cuda_stream

    same_o = torch.empty_like(q)
    same_l = torch.empty((shape.n_heads, shape.lq), dtype=torch.float32, device=dev)
    N.sr_chunk_attention(twin.gpu.handle, 0, q.data_ptr(), k.data_ptr(), v.data_ptr(), same_o.data_ptr(),
                         same_l.data_ptr(), stream)
    for call in range(2):
        o = torch.full_like(q, float("nan"))
        lse = torch.full((shape.n_heads, shape.lq), float("nan"), dtype=torch.float32, device=dev)
        N.sr_chunk_attention_noalloc(tw.gpu.handle, 0, q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                     lse.data_ptr(), stream)
        torch.cuda.synchronize()
        got = o.float().cpu().numpy().astype(np.float64)[:, heads][rows]
        assert_attention_close(got, ref, f"noalloc call {call} against the oracle")
        got_lse = lse.cpu().numpy().astype(np.float64)[heads][:, rows]
        assert np.abs(got_lse - ref_lse).max() <= LSE_ABS
        assert torch.equal(o, same_o), f"noalloc call {call} differs from sr_chunk_attention with a workspace"
        assert torch.equal(lse, same_l)
    assert tw.gpu.error_status() == 0 and twin.gpu.error_status() == 0


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


@pytest.mark.parametrize("case", range(12))
def test_noalloc_random_shapes_match_oracle_and_workspace_twin(case):
    """Random session shapes (1-4 heads of 64 or 128, small grids, 1-3 chunk
    frames, rings of 0 to 2F+1 frames partly filled, 0-200 sink tokens) with a
    forced key split of 1, 2 or 4 parts: the allocation-free call against the
    oracle, and bit for bit against sr_chunk_attention on a twin session with a
    workspace of its own and the same split."""
    from chunked_kv_cache_gb300 import _native as N
    rng = np.random.default_rng(6000 + case)
    d = int(rng.choice([64, 128]))
    H = int(rng.integers(1, 5))
    gh, gw = int(rng.integers(1, 13)), int(rng.integers(1, 17))
    F = int(rng.integers(1, 4))
    W = int(rng.choice([0, F, F + 1, 2 * F + 1]))
    S = int(rng.choice([0, 1, 37, 128, 200]))
    shape = syn.Shape(f"noalloc fuzz {case}", H, d, gh, gw, F, W, S, 1)
    fill = int(rng.integers(0, W + 1)) if W else 0
    split = int(rng.choice([1, 2, 4]))
    tw = Twin(shape, 7, fill=fill, session=case, tail_split=split, workspace=False)
    twin = Twin(shape, 7, fill=fill, session=case, tail_split=split, workspace=True)
    dev = tw.dev
    x = syn.chunk_inputs(shape, 7, session=case, chunk=1)
    q, k, v = (to_dev(b, dev) for b in (x.q[0], x.k[0], x.v[0]))
    tw.gpu.rope3d_qk(q, k)
    qo, ko = tw.ora.rope3d_qk(x.q[0], x.k[0])
    ref, ref_lse = tw.ora.chunk_attention(0, qo, ko, x.v[0])
    stream = torch.cuda.current_stream(dev).cuda_stream
    same_o = torch.empty_like(q)
    same_l = torch.empty((H, shape.lq), dtype=torch.float32, device=dev)
    N.sr_chunk_attention(twin.gpu.handle, 0, q.data_ptr(), k.data_ptr(), v.data_ptr(), same_o.data_ptr(),
                         same_l.data_ptr(), stream)
    o = torch.full_like(q, float("nan"))
    lse = torch.full((H, shape.lq), float("nan"), dtype=torch.float32, device=dev)
    N.sr_chunk_attention_noalloc(tw.gpu.handle, 0, q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                 lse.data_ptr(), stream)
    torch.cuda.synchronize()
    assert_attention_close(o.float().cpu().numpy().astype(np.float64), ref, f"{shape.name} against the oracle")
    assert np.abs(lse.cpu().numpy().astype(np.float64) - ref_lse).max() <= LSE_ABS
    assert torch.equal(o, same_o) and torch.equal(lse, same_l), f"{shape.name}: differs from the workspace twin"
    assert tw.gpu.error_status() == 0 and twin.gpu.error_status() == 0
