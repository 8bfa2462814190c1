"""ctypes binding of libsr.so: the C ABI of include/sr.h, argument marshalling only.

Every function keeps the C name and takes plain integers for device pointers
and for the CUDA stream. No computation happens here; if the library is
missing, loading raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libsr.so")

SR_OK = 0
SR_ERR_INVALID_ARG = -1
SR_ERR_UNSUPPORTED = -2
SR_ERR_ALIGN = -3
SR_ERR_STATE = -4
SR_ERR_CUDA = -5
SR_ERR_TIMEOUT = -6
SR_DEVERR_WAIT_TIMEOUT = 1
SR_MAX_BATCH = 24
SR_MAX_LAYER_WINDOWS = 96

# every extern "C" symbol that include/sr.h declares
EXPORTS = (
    "sr_session_init", "sr_session_restore", "sr_session_frames", "sr_rope3d_qk",
    "sr_chunk_attention", "sr_cache_commit", "sr_session_free", "sr_chunk_attention_batch",
    "sr_device_error_status", "sr_debug_wait_timeout", "sr_status_string", "sr_workspace_bytes",
    "sr_chunk_attention_noalloc", "sr_plan_chunk", "sr_rope3d_qk_frames", "sr_chunk_attention_frames",
    "sr_cache_commit_frames", "sr_window_attention", "sr_rope3d_qk_at", "sr_rope3d_qk_dev",
    "sr_chunk_attention_dev", "sr_cache_commit_dev", "sr_window_count", "sr_plan_window",
    "sr_plan_attention", "sr_rope_angle", "sr_layer_rope_gather", "sr_layer_commit",
)


class SrConfig(ctypes.Structure):
    _fields_ = [
        ("n_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("grid_h", ctypes.c_int32), ("grid_w", ctypes.c_int32),
        ("chunk_frames", ctypes.c_int32), ("window_frames", ctypes.c_int32),
        ("n_sink", ctypes.c_int32), ("n_steps", ctypes.c_int32),
        ("t_clock0", ctypes.c_int32), ("rope_base", ctypes.c_float),
        ("softmax_scale", ctypes.c_float), ("wait_timeout_ns", ctypes.c_uint64),
        ("tail_split", ctypes.c_int32),
    ]


class SrBuffers(ctypes.Structure):
    _fields_ = [
        ("sink_k", ctypes.c_void_p), ("sink_v", ctypes.c_void_p),
        ("ring_k", ctypes.c_void_p), ("ring_v", ctypes.c_void_p),
        ("slot_frame", ctypes.c_void_p), ("err_word", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p), ("frame_counter", ctypes.c_void_p),
    ]


class SrChunkPlan(ctypes.Structure):
    _fields_ = [
        ("first_frame", ctypes.c_int32), ("n_frames", ctypes.c_int32),
        ("hist_frames", ctypes.c_int32), ("sink_frames", ctypes.c_int32),
    ]


class SrWindow(ctypes.Structure):
    _fields_ = [("row0", ctypes.c_int32), ("col0", ctypes.c_int32), ("rows", ctypes.c_int32),
                ("cols", ctypes.c_int32)]


class SrError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


_lib = None


def lib() -> ctypes.CDLL:
    """Load libsr.so once (raises OSError if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise OSError(f"{LIB_PATH} is missing: build it with `python -m chunked_kv_cache_gb300.build` "
                          "(there is no fallback implementation)")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64, u64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64
        L.sr_session_init.argtypes = [ctypes.POINTER(SrConfig), ctypes.POINTER(SrBuffers), vp, vp, vp,
                                      ctypes.POINTER(vp)]
        L.sr_session_restore.argtypes = [vp, i64]
        L.sr_session_frames.argtypes = [vp, ctypes.POINTER(i64)]
        L.sr_rope3d_qk.argtypes = [vp, vp, vp, vp]
        L.sr_chunk_attention.argtypes = [vp, i32, vp, vp, vp, vp, vp, vp]
        L.sr_cache_commit.argtypes = [vp, vp, vp, vp]
        L.sr_chunk_attention_noalloc.argtypes = [vp, i32, vp, vp, vp, vp, vp, vp]
        L.sr_session_free.argtypes = [vp]
        L.sr_plan_chunk.argtypes = [i32, i32, i32, i32, i32, i32, ctypes.POINTER(SrChunkPlan)]
        L.sr_rope3d_qk_frames.argtypes = [vp, i32, vp, vp, vp]
        L.sr_chunk_attention_frames.argtypes = [vp, i32, i32, i32, vp, vp, vp, vp, vp, vp]
        L.sr_cache_commit_frames.argtypes = [vp, i32, vp, vp, vp]
        L.sr_window_attention.argtypes = [vp, i32, i32, i32, vp, vp, vp, vp, vp, vp]
        L.sr_rope3d_qk_at.argtypes = [vp, i64, i32, vp, vp, vp]
        L.sr_rope3d_qk_dev.argtypes = [vp, i32, vp, vp, vp]
        L.sr_chunk_attention_dev.argtypes = [vp, i32, i32, i32, vp, vp, vp, vp, vp, vp]
        L.sr_cache_commit_dev.argtypes = [vp, i32, vp, vp, vp]
        L.sr_window_count.argtypes = [i32, i32, i32, i32, ctypes.POINTER(i32)]
        L.sr_plan_window.argtypes = [i32, i32, i32, i32, i32, ctypes.POINTER(SrWindow)]
        L.sr_chunk_attention_batch.argtypes = [ctypes.POINTER(vp), i32, i32, vp, vp, vp,
                                               ctypes.POINTER(i64), vp, vp, vp]
        L.sr_plan_attention.argtypes = [i32, i64, i64, i32, i32, i32, ctypes.POINTER(i32), ctypes.POINTER(i32),
                                        ctypes.POINTER(i64)]
        L.sr_rope_angle.argtypes = [ctypes.POINTER(SrConfig), i32, i64, ctypes.POINTER(ctypes.c_float)]
        L.sr_layer_rope_gather.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(SrWindow), i32, i32, i32, vp, vp, vp,
                                           vp, vp, vp, vp]
        L.sr_layer_commit.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(SrWindow), i32, i32, i32, vp, vp, vp]
        L.sr_device_error_status.argtypes = [i32]
        L.sr_debug_wait_timeout.argtypes = [vp, u64, vp]
        L.sr_workspace_bytes.argtypes = [ctypes.POINTER(SrConfig), ctypes.POINTER(ctypes.c_uint64)]
        L.sr_status_string.argtypes = [ctypes.c_int]
        L.sr_status_string.restype = ctypes.c_char_p
        for name in EXPORTS:
            if name != "sr_status_string":
                getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def status_string(st: int) -> str:
    return lib().sr_status_string(int(st)).decode()


def _check(st: int, what: str) -> None:
    if st != SR_OK:
        raise SrError(st, what)


def sr_session_init(cfg: SrConfig, bufs: SrBuffers, sink_k_src: int, sink_v_src: int, stream: int) -> int:
    out = ctypes.c_void_p()
    _check(lib().sr_session_init(ctypes.byref(cfg), ctypes.byref(bufs), sink_k_src or None,
                                 sink_v_src or None, stream or None, ctypes.byref(out)), "sr_session_init")
    return out.value


def sr_workspace_bytes(cfg: SrConfig) -> int:
    n = ctypes.c_uint64()
    _check(lib().sr_workspace_bytes(ctypes.byref(cfg), ctypes.byref(n)), "sr_workspace_bytes")
    return n.value


def sr_session_restore(handle: int, n_committed: int) -> None:
    _check(lib().sr_session_restore(handle, int(n_committed)), "sr_session_restore")


def sr_session_frames(handle: int) -> int:
    n = ctypes.c_int64()
    _check(lib().sr_session_frames(handle, ctypes.byref(n)), "sr_session_frames")
    return n.value


def sr_rope3d_qk(handle: int, q: int, k: int, stream: int) -> None:
    _check(lib().sr_rope3d_qk(handle, q or None, k or None, stream or None), "sr_rope3d_qk")


def sr_chunk_attention(handle: int, step: int, q: int, k: int, v: int, o: int, lse: int, stream: int) -> None:
    _check(lib().sr_chunk_attention(handle, int(step), q, k, v, o, lse or None, stream or None),
           "sr_chunk_attention")


def sr_plan_chunk(chunk_index: int, bootstrap_units: int = 7, chunk_units: int = 2, window_units: int = 2,
                  sink_units: int = 2, merge_single_frame_units: bool = True) -> SrChunkPlan:
    out = SrChunkPlan()
    _check(lib().sr_plan_chunk(int(chunk_index), int(bootstrap_units), int(chunk_units), int(window_units),
                               int(sink_units), 1 if merge_single_frame_units else 0, ctypes.byref(out)),
           "sr_plan_chunk")
    return out


def sr_plan_attention(n_heads: int, lq: int, key_tiles: int, has_workspace: bool = True, tail_split: int = 0,
                      sm_count: int = 0) -> dict:
    """The attention launch plan of one query group (host arithmetic)."""
    parts, conv, units = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int64()
    _check(lib().sr_plan_attention(int(n_heads), int(lq), int(key_tiles), 1 if has_workspace else 0, int(tail_split),
                                   int(sm_count), ctypes.byref(parts), ctypes.byref(conv), ctypes.byref(units)),
           "sr_plan_attention")
    return {"parts": parts.value, "whole_as_tiles": conv.value, "n_units": units.value}


def sr_rope3d_qk_frames(handle: int, n_frames: int, q: int, k: int, stream: int) -> None:
    _check(lib().sr_rope3d_qk_frames(handle, int(n_frames), q or None, k or None, stream or None),
           "sr_rope3d_qk_frames")


def sr_chunk_attention_frames(handle: int, step: int, n_frames: int, hist_frames: int, q: int, k: int, v: int,
                              o: int, lse: int, stream: int) -> None:
    _check(lib().sr_chunk_attention_frames(handle, int(step), int(n_frames), int(hist_frames), q, k, v, o,
                                           lse or None, stream or None), "sr_chunk_attention_frames")


def sr_cache_commit_frames(handle: int, n_frames: int, k_raw: int, v: int, stream: int) -> None:
    _check(lib().sr_cache_commit_frames(handle, int(n_frames), k_raw, v, stream or None), "sr_cache_commit_frames")


def sr_window_attention(handle: int, step: int, moving_frames: int, with_prefix: bool, q: int, k_moving: int,
                        v_moving: int, o: int, lse: int, stream: int) -> None:
    _check(lib().sr_window_attention(handle, int(step), int(moving_frames), 1 if with_prefix else 0, q, k_moving,
                                     v_moving, o, lse or None, stream or None), "sr_window_attention")


def sr_rope3d_qk_at(handle: int, first_frame: int, n_frames: int, q: int, k: int, stream: int) -> None:
    _check(lib().sr_rope3d_qk_at(handle, int(first_frame), int(n_frames), q or None, k or None, stream or None),
           "sr_rope3d_qk_at")


def sr_rope3d_qk_dev(handle: int, n_frames: int, q: int, k: int, stream: int) -> None:
    _check(lib().sr_rope3d_qk_dev(handle, int(n_frames), q or None, k or None, stream or None), "sr_rope3d_qk_dev")


def sr_chunk_attention_dev(handle: int, step: int, n_frames: int, hist_frames: int, q: int, k: int, v: int, o: int,
                           lse: int, stream: int) -> None:
    _check(lib().sr_chunk_attention_dev(handle, int(step), int(n_frames), int(hist_frames), q, k, v, o, lse or None,
                                        stream or None), "sr_chunk_attention_dev")


def sr_cache_commit_dev(handle: int, n_frames: int, k_raw: int, v: int, stream: int) -> None:
    _check(lib().sr_cache_commit_dev(handle, int(n_frames), k_raw, v, stream or None), "sr_cache_commit_dev")


def sr_window_count(grid_h: int, grid_w: int, window: int, shifted: bool) -> int:
    n = ctypes.c_int32()
    _check(lib().sr_window_count(int(grid_h), int(grid_w), int(window), 1 if shifted else 0, ctypes.byref(n)),
           "sr_window_count")
    return n.value


def sr_plan_window(grid_h: int, grid_w: int, window: int, shifted: bool, index: int) -> SrWindow:
    out = SrWindow()
    _check(lib().sr_plan_window(int(grid_h), int(grid_w), int(window), 1 if shifted else 0, int(index),
                                ctypes.byref(out)), "sr_plan_window")
    return out


def sr_chunk_attention_noalloc(handle: int, step: int, q: int, k: int, v: int, o: int, lse: int,
                               stream: int) -> None:
    """sr_chunk_attention with the library's built-in scratch instead of a workspace,
    for callers that cannot allocate device memory."""
    _check(lib().sr_chunk_attention_noalloc(handle, int(step), q, k, v, o, lse or None, stream or None),
           "sr_chunk_attention_noalloc")


def sr_cache_commit(handle: int, k_raw: int, v: int, stream: int) -> None:
    _check(lib().sr_cache_commit(handle, k_raw, v, stream or None), "sr_cache_commit")


def sr_session_free(handle: int) -> None:
    _check(lib().sr_session_free(handle), "sr_session_free")


def sr_chunk_attention_batch(handles, step: int, q: int, k: int, v: int, q_off, o: int, lse: int,
                             stream: int) -> None:
    n = len(handles)
    arr = (ctypes.c_void_p * n)(*handles)
    offs = (ctypes.c_int64 * (n + 1))(*[int(x) for x in q_off])
    _check(lib().sr_chunk_attention_batch(arr, n, int(step), q, k, v, offs, o, lse or None, stream or None),
           "sr_chunk_attention_batch")


def sr_rope_angle(cfg: SrConfig, pair: int, position: int) -> float:
    """The reduced rotation angle (radians, float) the kernels apply to one pair (host arithmetic)."""
    a = ctypes.c_float()
    _check(lib().sr_rope_angle(ctypes.byref(cfg), int(pair), int(position), ctypes.byref(a)), "sr_rope_angle")
    return a.value


def _layer_args(handles, windows):
    n = len(handles)
    arr = (ctypes.c_void_p * n)(*handles)
    wins = (SrWindow * n)(*[SrWindow(w.row0, w.col0, w.rows, w.cols) for w in windows])
    return arr, wins, n


def sr_layer_rope_gather(handles, windows, frame_h: int, frame_w: int, q: int, k: int, v: int, q_packed: int,
                         k_packed: int, v_packed: int, stream: int) -> None:
    """A decoder layer's window gather with RoPE (q, k) and copy (v, optional), one launch."""
    arr, wins, n = _layer_args(handles, windows)
    _check(lib().sr_layer_rope_gather(arr, wins, n, int(frame_h), int(frame_w), q, k, v or None, q_packed, k_packed,
                                      v_packed or None, stream or None), "sr_layer_rope_gather")


def sr_layer_commit(handles, windows, frame_h: int, frame_w: int, k_raw: int, v: int, stream: int) -> None:
    """Every window's ring commit of a decoder layer, one launch."""
    arr, wins, n = _layer_args(handles, windows)
    _check(lib().sr_layer_commit(arr, wins, n, int(frame_h), int(frame_w), k_raw, v, stream or None),
           "sr_layer_commit")


def sr_device_error_status(value: int) -> int:
    return lib().sr_device_error_status(int(value))


def sr_debug_wait_timeout(err_word: int, timeout_ns: int, stream: int) -> None:
    _check(lib().sr_debug_wait_timeout(err_word, int(timeout_ns), stream or None), "sr_debug_wait_timeout")
