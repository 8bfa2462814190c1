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
