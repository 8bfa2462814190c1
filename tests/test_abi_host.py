"""C-ABI checks that need no GPU: the library builds, loads, exports every
symbol include/sr.h declares, and rejects bad arguments before launching
anything (so these calls never touch a device)."""
import ctypes
import os
import re

import pytest

from chunked_kv_cache_gb300 import _native as N
from chunked_kv_cache_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return N.lib()


def _header_functions():
    src = open(os.path.join(ROOT, "include", "sr.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(sr_[a-z_0-9]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    declared = _header_functions()
    assert set(declared) == set(N.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name


def test_no_other_symbols_leak(lib):
    # internal kernels and helpers are hidden; only the C ABI is visible
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", N.LIB_PATH], capture_output=True, text=True).stdout
    names = {l.split()[-1] for l in out.splitlines() if " T " in l}
    ours = {n for n in names if n.startswith("sr_")}
    assert ours == set(N.EXPORTS)


def test_status_strings(lib):
    assert N.status_string(0) == "ok"
    assert "timed out" in N.status_string(N.SR_ERR_TIMEOUT)
    assert N.status_string(-99) == "unknown status"
    assert N.sr_device_error_status(0) == N.SR_OK
    assert N.sr_device_error_status(N.SR_DEVERR_WAIT_TIMEOUT | (5 << 8)) == N.SR_ERR_TIMEOUT


def _cfg(**kw):
    base = dict(n_heads=4, head_dim=64, grid_h=6, grid_w=10, chunk_frames=2, window_frames=4, n_sink=64,
                n_steps=2, t_clock0=0, rope_base=10000.0, softmax_scale=0.0, wait_timeout_ns=0)
    base.update(kw)
    return N.SrConfig(**base)


def _bufs(**kw):
    base = dict(sink_k=0x10000, sink_v=0x20000, ring_k=0x30000, ring_v=0x40000, slot_frame=0x50000,
                err_word=0x60000)
    base.update(kw)
    return N.SrBuffers(**base)


def _init(cfg, bufs):
    out = ctypes.c_void_p(0x1234)
    st = N.lib().sr_session_init(ctypes.byref(cfg), ctypes.byref(bufs), None, None, None, ctypes.byref(out))
    return st, out.value


@pytest.mark.parametrize("field,value,status", [
    ("head_dim", 96, N.SR_ERR_UNSUPPORTED),
    ("head_dim", 256, N.SR_ERR_UNSUPPORTED),
    ("n_heads", 0, N.SR_ERR_INVALID_ARG),
    ("grid_h", 0, N.SR_ERR_INVALID_ARG),
    ("chunk_frames", 0, N.SR_ERR_INVALID_ARG),
    ("window_frames", -1, N.SR_ERR_INVALID_ARG),
    ("window_frames", 1, N.SR_ERR_INVALID_ARG),       # 0 < W < F would overwrite within one commit
    ("n_sink", -5, N.SR_ERR_INVALID_ARG),
    ("n_steps", 0, N.SR_ERR_INVALID_ARG),
    ("rope_base", 1.0, N.SR_ERR_INVALID_ARG),
    ("rope_base", float("nan"), N.SR_ERR_INVALID_ARG),
    ("softmax_scale", float("inf"), N.SR_ERR_INVALID_ARG),
    ("grid_w", 1 << 20, N.SR_ERR_INVALID_ARG),         # too many tokens
])
def test_invalid_config_rejected_before_launch(lib, field, value, status):
    st, out = _init(_cfg(**{field: value}), _bufs())
    assert st == status
    assert out is None


@pytest.mark.parametrize("field,value,status", [
    ("sink_k", 0, N.SR_ERR_INVALID_ARG),
    ("ring_v", 0, N.SR_ERR_INVALID_ARG),
    ("slot_frame", 0, N.SR_ERR_INVALID_ARG),
    ("err_word", 0, N.SR_ERR_INVALID_ARG),
    ("sink_k", 0x10008, N.SR_ERR_ALIGN),
    ("ring_k", 0x30001, N.SR_ERR_ALIGN),
    ("err_word", 0x60002, N.SR_ERR_ALIGN),
])
def test_bad_buffers_rejected_before_launch(lib, field, value, status):
    st, out = _init(_cfg(), _bufs(**{field: value}))
    assert st == status and out is None


def test_null_arguments(lib):
    L = N.lib()
    assert L.sr_session_init(None, None, None, None, None, None) == N.SR_ERR_INVALID_ARG
    assert L.sr_chunk_attention(None, 0, 16, 16, 16, 16, None, None) == N.SR_ERR_INVALID_ARG
    assert L.sr_cache_commit(None, 16, 16, None) == N.SR_ERR_INVALID_ARG
    assert L.sr_rope3d_qk(None, 16, 16, None) == N.SR_ERR_INVALID_ARG
    assert L.sr_session_restore(None, 0) == N.SR_ERR_INVALID_ARG
    assert L.sr_session_frames(None, None) == N.SR_ERR_INVALID_ARG
    assert L.sr_session_free(None) == N.SR_OK
    assert L.sr_debug_wait_timeout(None, 1000, None) == N.SR_ERR_INVALID_ARG
    offs = (ctypes.c_int64 * 2)(0, 120)
    assert L.sr_chunk_attention_batch(None, 1, 0, 16, 16, 16, offs, 16, None, None) == N.SR_ERR_INVALID_ARG
    arr = (ctypes.c_void_p * 1)(None)
    assert L.sr_chunk_attention_batch(arr, 0, 0, 16, 16, 16, offs, 16, None, None) == N.SR_ERR_INVALID_ARG
    assert L.sr_chunk_attention_batch(arr, 17, 0, 16, 16, 16, offs, 16, None, None) == N.SR_ERR_INVALID_ARG


def test_layer_calls_reject_bad_arguments(lib):
    L = N.lib()
    arr = (ctypes.c_void_p * 1)(None)
    wins = (N.SrWindow * 1)(N.SrWindow(0, 0, 16, 16))
    # NULL sessions / windows, a NULL session inside, n out of range, empty frame
    assert L.sr_layer_rope_gather(None, wins, 1, 16, 16, 16, 16, None, 16, 16, None, None) == N.SR_ERR_INVALID_ARG
    assert L.sr_layer_rope_gather(arr, None, 1, 16, 16, 16, 16, None, 16, 16, None, None) == N.SR_ERR_INVALID_ARG
    assert L.sr_layer_rope_gather(arr, wins, 1, 16, 16, 16, 16, None, 16, 16, None, None) == N.SR_ERR_INVALID_ARG
    assert L.sr_layer_rope_gather(arr, wins, 0, 16, 16, 16, 16, None, 16, 16, None, None) == N.SR_ERR_INVALID_ARG
    assert L.sr_layer_rope_gather(arr, wins, N.SR_MAX_LAYER_WINDOWS + 1, 16, 16, 16, 16, None, 16, 16, None,
                                  None) == N.SR_ERR_INVALID_ARG
    assert L.sr_layer_rope_gather(arr, wins, 1, 0, 16, 16, 16, None, 16, 16, None, None) == N.SR_ERR_INVALID_ARG
    # v without v_packed
    assert L.sr_layer_rope_gather(arr, wins, 1, 16, 16, 16, 16, 16, 16, 16, None, None) == N.SR_ERR_INVALID_ARG
    # a misaligned pointer is refused before the sessions are looked at
    assert L.sr_layer_rope_gather(arr, wins, 1, 16, 16, 24, 16, None, 16, 16, None, None) == N.SR_ERR_ALIGN
    assert L.sr_layer_commit(None, wins, 1, 16, 16, 16, 16, None) == N.SR_ERR_INVALID_ARG
    assert L.sr_layer_commit(arr, wins, 1, 16, 16, None, 16, None) == N.SR_ERR_INVALID_ARG
    assert L.sr_layer_commit(arr, wins, 1, 16, 16, 16, 8, None) == N.SR_ERR_ALIGN


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(N, "_lib", None)
    monkeypatch.setattr(N, "LIB_PATH", str(tmp_path / "libsr.so"))
    with pytest.raises(OSError, match="no fallback"):
        N.lib()


def test_workspace_bytes_closed_form(lib):
    n = N.sr_workspace_bytes(_cfg(n_heads=24, head_dim=128))
    # counters (24 x 4 B, padded to 256) + 24 heads x 4 parts x 128 rows x (128 + 4) floats
    assert n == 256 + 24 * 4 * 128 * 132 * 4
    assert N.sr_workspace_bytes(_cfg(n_heads=100, head_dim=64)) == 512 + 100 * 4 * 128 * 68 * 4


@pytest.mark.parametrize("value", [-1, 5])
def test_tail_split_out_of_range(lib, value):
    st, out = _init(_cfg(tail_split=value), _bufs())
    assert st == N.SR_ERR_INVALID_ARG and out is None


def test_misaligned_workspace(lib):
    st, out = _init(_cfg(), _bufs(workspace=0x70080))
    assert st == N.SR_ERR_ALIGN and out is None
