"""The library's chunk planner (sr_plan_chunk, host arithmetic in libsr.so)
against the oracle's scheduling units, on the CPU: the C restatement and the
oracle's must agree on every chunk of several unit configurations, and the C
entry point must reject what it documents as invalid. Also the argument checks
of the *_frames calls that need no GPU."""
import pytest

from oracle import chunk_plan


@pytest.fixture(scope="module")
def sr():
    import chunked_kv_cache_gb300 as m
    from chunked_kv_cache_gb300 import _native
    try:
        _native.lib()
    except OSError:
        pytest.skip("libsr.so is not built")
    return m


@pytest.mark.parametrize("boot,cu,wu,su,merge", [(7, 2, 2, 2, True), (7, 2, 5, 4, True), (3, 1, 2, 1, True),
                                                 (7, 2, 2, 2, False), (9, 3, 4, 2, True), (1, 1, 0, 0, True)])
def test_c_planner_matches_oracle(sr, boot, cu, wu, su, merge):
    for c in range(60):
        got = sr.plan_chunk(c, boot, cu, wu, su, merge)
        want = chunk_plan(c, boot, cu, wu, su, merge)
        assert got == {"first_frame": want["first_latent"], "n_frames": want["n_frames"],
                       "hist_frames": want["hist_frames"], "sink_frames": want["sink_frames"]}, c


def test_c_planner_rejects_invalid(sr):
    from chunked_kv_cache_gb300 import _native as N
    for args in [(-1, 7, 2, 2, 2, 1), (0, 0, 2, 2, 2, 1), (1, 7, 0, 2, 2, 1), (1, 7, 2, -1, 2, 1),
                 (1, 7, 2, 2, -1, 1), (2 ** 30, 7, 2, 2, 2, 1)]:
        with pytest.raises(N.SrError) as e:
            N.sr_plan_chunk(*args)
        assert e.value.status == N.SR_ERR_INVALID_ARG


def test_frames_calls_reject_bad_counts_without_a_gpu(sr):
    from chunked_kv_cache_gb300 import _native as N
    # a NULL session handle is rejected before anything else
    with pytest.raises(N.SrError):
        N.sr_rope3d_qk_frames(0, 3, 0, 0, 0)
    with pytest.raises(N.SrError):
        N.sr_chunk_attention_frames(0, 0, 3, -1, 16, 16, 16, 16, 0, 0)
    with pytest.raises(N.SrError):
        N.sr_cache_commit_frames(0, 3, 16, 16, 0)


@pytest.mark.parametrize("gh,gw,window", [(45, 80, 16), (40, 40, 16), (48, 84, 16), (10, 7, 4), (16, 16, 16)])
@pytest.mark.parametrize("shifted", [False, True])
def test_c_window_planner_matches_oracle(sr, gh, gw, window, shifted):
    from chunked_kv_cache_gb300 import _native as N
    from oracle.decoder import window_partition
    want = window_partition(gh, gw, window, shifted)
    n = N.sr_window_count(gh, gw, window, shifted)
    assert n == len(want)
    got = [N.sr_plan_window(gh, gw, window, shifted, i) for i in range(n)]
    assert [(w.row0, w.col0, w.rows, w.cols) for w in got] == want


def test_c_window_planner_rejects_invalid(sr):
    import ctypes
    from chunked_kv_cache_gb300 import _native as N
    for args in [(0, 8, 4, 0), (8, 8, 1, 0), (2, 8, 8, 1)]:
        with pytest.raises(N.SrError):
            N.sr_window_count(*args)
    n = ctypes.c_int32()
    assert N.lib().sr_window_count(8, 8, 4, 2, ctypes.byref(n)) == N.SR_ERR_INVALID_ARG   # shifted must be 0 or 1
    with pytest.raises(N.SrError):
        N.sr_plan_window(8, 8, 4, 0, 4)


# ---------------------------------------------------------------- attention launch plan

def _dispatch(costs, sms):
    """Longest-first list scheduling: each unit to the SM that frees up first."""
    import heapq
    free = [0.0] * sms
    for c in costs:
        t = heapq.heappop(free)
        heapq.heappush(free, t + c)
    return max(free)


def _plan_model(H, lq, tiles, ws, forced, sms):
    """The plan restated: whole blocks, then single-tile units, then last-block parts."""
    import math
    rem = lq % 256
    single = 0 < rem <= 128
    whole = H * ((lq + 255) // 256 - (1 if single else 0))
    ks = [1]
    if single and ws:
        cap = min(4, tiles)
        ks = [max(1, min(forced, cap))] if forced else list(range(1, cap + 1))
    left = whole % sms if whole >= sms and whole % sms <= sms // 2 else 0
    best = None
    for c in ([0, left] if left else [0]):
        for k in ks:
            costs = [float(tiles)] * (whole - c) + [math.ceil(tiles / 2) * 1.33 + 0.5] * (2 * c)
            if single:
                costs += [math.ceil(math.ceil(tiles / k) / 2) * 1.33 + 0.5 + (0.5 if k > 1 else 0)] * (H * k)
            t = _dispatch(costs, sms)
            if best is None or (c == best[2] and t < best[0] * 0.995) or (c != best[2] and t < best[0] * 0.98):
                best = (t, k, c)
    _, k, c = best
    return {"parts": k, "whole_as_tiles": c, "n_units": whole + c + (H * k if single else 0)}


@pytest.mark.parametrize("H,lq,tiles,want", [
    (24, 3120, 114, {"parts": 2, "whole_as_tiles": 0, "n_units": 288 + 48}),     # 832x480, ring full
    (40, 7200, 315, {"parts": 1, "whole_as_tiles": 56, "n_units": 1120 + 56 + 40}),   # 720p: 1120 = 7 x 152 + 56
    (24, 4680, 78, {"parts": 1, "whole_as_tiles": 0, "n_units": 432 + 24}),
])
def test_attention_plan_workloads(sr, H, lq, tiles, want):
    from chunked_kv_cache_gb300 import _native as N
    assert N.sr_plan_attention(H, lq, tiles, True, 0, 152) == want
    assert _plan_model(H, lq, tiles, True, 0, 152) == want


def test_attention_plan_matches_model_on_small_launches(sr):
    from chunked_kv_cache_gb300 import _native as N
    import random
    rng = random.Random(3)
    for _ in range(300):
        H, lq, tiles = rng.randint(1, 12), rng.randint(1, 2000), rng.randint(1, 40)
        ws, forced, sms = rng.random() < 0.7, rng.choice([0, 0, 1, 2, 3, 4]), rng.choice([4, 16, 152])
        assert N.sr_plan_attention(H, lq, tiles, ws, forced, sms) == _plan_model(H, lq, tiles, ws, forced, sms), \
            (H, lq, tiles, ws, forced, sms)


def test_attention_plan_without_workspace_and_invalid(sr):
    from chunked_kv_cache_gb300 import _native as N
    assert N.sr_plan_attention(24, 3120, 114, False, 0, 152)["parts"] == 1
    assert N.sr_plan_attention(24, 3120, 114, True, 3, 152)["parts"] == 3
    assert N.sr_plan_attention(24, 3120, 2, True, 4, 152)["parts"] == 2          # clamped to the key tiles
    for args in [(0, 3120, 114), (24, 0, 114), (24, 3120, 0)]:
        with pytest.raises(RuntimeError):
            N.sr_plan_attention(*args)
    with pytest.raises(RuntimeError):
        N.sr_plan_attention(24, 3120, 114, True, 5, 152)
