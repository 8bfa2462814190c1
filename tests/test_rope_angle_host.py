"""The library's rotary angle against the oracle's exact one (CPU only).

sr_rope_angle runs, on the host, the fixed-point phase arithmetic the RoPE and
commit kernels run: each pair's turns per position step held as a 96-bit
binary fraction, the phase of a position formed modulo one turn in integer
arithmetic, then scaled to radians and rounded to float. The oracle forms the
same angle, position * base**(-2i/d_axis) reduced modulo 2*pi, in 60-digit
decimal arithmetic ([H3-page] "Interactive Coding Worlds with Real-time
Streaming Diffusion Render", section 3.2 Iteration 4: the time position is the
absolute frame index of the stream, unbounded). They must agree to the float
rounding of the result at every position the ABI accepts, up to 2^42.
"""
import math

import numpy as np
import pytest

from chunked_kv_cache_gb300 import _native as N
from chunked_kv_cache_gb300 import build as B
from oracle import axis_split
from oracle.rope import reduced_angle


@pytest.fixture(scope="module")
def lib():
    B.build()
    return N.lib()


def _cfg(head_dim, base):
    return N.SrConfig(n_heads=1, head_dim=head_dim, grid_h=1, grid_w=1, chunk_frames=1, window_frames=0, n_sink=0,
                      n_steps=1, t_clock0=0, rope_base=base, softmax_scale=0.0, wait_timeout_ns=0)


def _pair_axis(d):
    """(axis length d_a, index i inside the axis) of every pair of a head."""
    out = []
    for d_a in axis_split(d):
        out += [(d_a, i) for i in range(d_a // 2)]
    return out


POSITIONS = [0, 1, -1, 7, 44, 79, 1000, 123457, 2 ** 24 - 1, 2 ** 24, 2 ** 24 + 1, 2 ** 24 + 3, 2 ** 30,
             2 ** 31 - 1, 2 ** 32 + 5, 2 ** 33, -(2 ** 33) + 11, 2 ** 40, 2 ** 40 + 2 ** 31 + 2 ** 30,
             -(2 ** 40) - 3, 2 ** 42 - 1, -(2 ** 42) + 1]


@pytest.mark.parametrize("head_dim,base", [(128, 10000.0), (64, 500.0), (128, 1.5), (64, 1.0001), (128, 1.0e6)])
def test_library_angle_matches_the_exact_reduction(lib, head_dim, base):
    cfg = _cfg(head_dim, base)
    rng = np.random.default_rng(head_dim)
    positions = POSITIONS + [int(x) for x in rng.integers(-(2 ** 42) + 1, 2 ** 42, size=12)]
    worst = 0.0
    for pair, (d_a, i) in enumerate(_pair_axis(head_dim)):
        for p in positions:
            got = N.sr_rope_angle(cfg, pair, p)
            ref = reduced_angle(p, i, d_a, float(np.float32(base)))
            assert -math.pi <= got <= math.pi
            err = abs((got - ref + math.pi) % (2 * math.pi) - math.pi)
            # the float rounding of the result, and nothing else
            bound = 0.5 * float(np.spacing(np.float32(max(abs(ref), 2.0 ** -126)))) + 1e-12
            assert err <= bound, (pair, p, got, ref, err, bound)
            worst = max(worst, err)
    assert worst < 2.4e-7


def test_angle_arguments_checked(lib):
    cfg = _cfg(128, 10000.0)
    for pair, pos in ((-1, 0), (64, 0), (0, 2 ** 42), (0, -(2 ** 42))):
        with pytest.raises(N.SrError) as e:
            N.sr_rope_angle(cfg, pair, pos)
        assert e.value.status == N.SR_ERR_INVALID_ARG
    bad = _cfg(96, 10000.0)
    with pytest.raises(N.SrError) as e:
        N.sr_rope_angle(bad, 0, 0)
    assert e.value.status == N.SR_ERR_UNSUPPORTED


def test_float_product_would_fail_this_test():
    # what the bound rules out: at p = 2^24 + 1 the float product p * 1.0 rounds
    # to 2^24, a full radian short of the exact angle of a frequency-one pair
    p = 2 ** 24 + 1
    naive = float(np.float32(p)) * 1.0
    exact = reduced_angle(p, 0, 44, 10000.0)
    err = abs((math.fmod(naive, 2 * math.pi) - exact + math.pi) % (2 * math.pi) - math.pi)
    assert err > 0.5
