"""Shared helpers for the GPU parity tests: build twin sessions (CUDA library
and float64 oracle) from the same seeded synthetic inputs, and compare."""
import numpy as np
import pytest
import torch

import synthetic as syn
from oracle import OracleSession, bf16_bits_to_f64

# spec gates on bf16 outputs, plus a relative gate (outputs are small:
# softmax over thousands of near-uniform keys)
MAX_ABS = 2e-2
MEAN_ABS = 2e-3
REL_RMS = 1e-2
LSE_ABS = 5e-3


def device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda", 0)


def to_dev(bits, dev):
    return syn.bits_to_torch(bits).to(dev)


def bf16_ordinal(bits: np.ndarray) -> np.ndarray:
    """Map bf16 bit patterns to integers whose difference counts ulps."""
    b = bits.astype(np.int64)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def ulp_distance(a_bits, b_bits) -> np.ndarray:
    return np.abs(bf16_ordinal(np.asarray(a_bits)) - bf16_ordinal(np.asarray(b_bits)))


def assert_rotated_close(gpu_bits, ref_bits, what=""):
    """Rotated bf16 values: within one bf16 ulp of the oracle's correctly
    rounded value, plus the fp32 evaluation error of the rotation, which is
    absolute (bounded by 2^-19 times the pair's norm) and so exceeds an ulp
    only for outputs that nearly cancel. Almost every element must match
    bit for bit: all but 0.1 %, or all but two in a tensor of fewer than
    2000 elements. An element whose exact value lies within the fp32
    evaluation error of a bf16 rounding midpoint may round to the other
    neighbour, a few in 10^5 of them; in a 256-element tensor one such flip
    is 0.4 %."""
    g = bf16_bits_to_f64(np.asarray(gpu_bits))
    r = bf16_bits_to_f64(np.asarray(ref_bits))
    pair = np.sqrt(r[..., 0::2] ** 2 + r[..., 1::2] ** 2)
    pair = np.repeat(pair, 2, axis=-1)
    mag = np.maximum(np.abs(r), 2.0 ** -126)
    ulp = 2.0 ** (np.floor(np.log2(mag)) - 7)
    err = np.abs(g - r)
    bound = ulp + 2.0 ** -19 * pair
    worst = np.argmax(err - bound)
    assert np.all(err <= bound), (f"{what}: |gpu-ref| {err.flat[worst]:.3e} > bound {bound.flat[worst]:.3e} "
                                  f"(ref {r.flat[worst]:.4e}, gpu {g.flat[worst]:.4e})")
    n_diff = int((np.asarray(gpu_bits) != np.asarray(ref_bits)).sum())
    n = np.asarray(gpu_bits).size
    assert n_diff <= max(1e-3 * n, 2), f"{what}: {n_diff} of {n} elements not bit-identical"


def assert_attention_close(got: np.ndarray, ref: np.ndarray, what: str = ""):
    got = np.asarray(got, np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    rel = np.sqrt(np.mean(err ** 2)) / max(np.sqrt(np.mean(ref ** 2)), 1e-30)
    assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS and rel <= REL_RMS, (
        f"{what}: max {err.max():.3e} mean {err.mean():.3e} rel-rms {rel:.3e}")


class Twin:
    """A CUDA session and an oracle session in the same state."""

    def __init__(self, shape: syn.Shape, config: int, fill: int = 0, session: int = 0, t_clock0: int = 0,
                 n_sink=None, window_frames=None, dev=None, heads=None, tail_split: int = 0,
                 workspace: bool = True):
        import chunked_kv_cache_gb300 as sr
        self.dev = dev or device()
        self.shape = shape
        S = shape.n_sink if n_sink is None else n_sink
        W = shape.window_frames if window_frames is None else window_frames
        sh = syn.Shape(shape.name, shape.n_heads, shape.head_dim, shape.grid_h, shape.grid_w,
                       shape.chunk_frames, W, S, shape.n_steps, shape.rope_base)
        self.sh = sh
        sk, sv = syn.session_sinks(sh, config, session)
        self.gpu = sr.Session(sh.n_heads, sh.head_dim, sh.grid_h, sh.grid_w, sh.chunk_frames, W, S, sh.n_steps,
                              sink_k=to_dev(sk, self.dev), sink_v=to_dev(sv, self.dev), t_clock0=t_clock0,
                              tail_split=tail_split, workspace=workspace, device=self.dev)
        # the oracle may follow only a subset of heads (heads are independent)
        self.heads = None if heads is None else np.asarray(heads)
        hs = slice(None) if heads is None else self.heads
        osk = sk[:, :, hs] if heads is not None else sk
        osv = sv[:, :, hs] if heads is not None else sv
        nh = sh.n_heads if heads is None else len(heads)
        self.ora = OracleSession(nh, sh.head_dim, sh.grid_h, sh.grid_w, sh.chunk_frames, W, S, sh.n_steps,
                                 osk, osv, t_clock0=t_clock0)
        if W > 0:
            rk, rv, slots = syn.ring_prefill(sh, config, fill, session)
            self.gpu.ring_k.copy_(to_dev(rk, self.dev))
            self.gpu.ring_v.copy_(to_dev(rv, self.dev))
            self.gpu.slot_frame.copy_(torch.from_numpy(slots).to(self.dev))
            self.gpu.restore(fill)
            self.ora.load_ring(rk[:, hs] if heads is not None else rk, rv[:, hs] if heads is not None else rv,
                               slots, fill)

    def oh(self, bits):
        """Slice host bits to the oracle's heads."""
        return bits if self.heads is None else np.ascontiguousarray(bits[:, self.heads])

    def step(self, x: syn.ChunkInputs, step: int, rows=None, lse=False):
        """Run RoPE + attention on both sides; returns (gpu_o [sampled], ref_o, gpu_lse, ref_lse)."""
        q, k, v = to_dev(x.q[step], self.dev), to_dev(x.k[step], self.dev), to_dev(x.v[step], self.dev)
        self.gpu.rope3d_qk(q, k)
        res = self.gpu.chunk_attention(step, q, k, v, lse=lse)
        o, l = res if lse else (res, None)
        qo, ko = self.ora.rope3d_qk(self.oh(x.q[step]), self.oh(x.k[step]))
        ref, ref_lse = self.ora.chunk_attention(step, qo, ko, self.oh(x.v[step]), rows=rows)
        got = o.float().cpu().numpy()
        if self.heads is not None:
            got = got[:, self.heads]
        if rows is not None:
            got = got[np.asarray(rows)]
        gl = None
        if l is not None:
            gl = l.cpu().numpy().astype(np.float64)
            if self.heads is not None:
                gl = gl[self.heads]
            if rows is not None:
                gl = gl[:, np.asarray(rows)]
        return got.astype(np.float64), ref, gl, ref_lse

    def commit(self, x: syn.ChunkInputs):
        self.gpu.cache_commit(to_dev(x.clean_k, self.dev), to_dev(x.clean_v, self.dev))
        self.ora.cache_commit(self.oh(x.clean_k), self.oh(x.clean_v))

    def ring_bits(self):
        rk = syn.torch_to_bits(self.gpu.ring_k)
        rv = syn.torch_to_bits(self.gpu.ring_v)
        if self.heads is not None:
            rk, rv = rk[:, self.heads], rv[:, self.heads]
        return rk, rv
