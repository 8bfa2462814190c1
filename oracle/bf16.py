"""bf16 <-> float64 for the oracle (test infrastructure only).

bf16 is the top half of an IEEE binary32: 1 sign, 8 exponent, 7 fraction
bits. Widening is exact. Narrowing rounds the exact float64 value to the
nearest bf16 with ties to even, which is where the API stores bf16: roped Q/K
and the ring's K/V.
"""
import numpy as np

_BF16_MAX = float.fromhex("0x1.fep127")      # largest finite bf16
_MIN_NORMAL_EXP = -126                      # 2**-126, smallest normal
_SUBNORMAL_STEP = 2.0 ** -133               # spacing below 2**-126


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 value (ties to even), as float64."""
    x = np.asarray(x, dtype=np.float64)
    out = np.empty_like(x)
    finite = np.isfinite(x)
    out[~finite] = x[~finite]
    xf = x[finite]
    mant, exp = np.frexp(xf)                 # xf = mant * 2**exp, |mant| in [0.5, 1)
    # a bf16 normal carries 8 significant bits: mant*2**8 rounded to an integer
    step_exp = np.maximum(exp - 8, _MIN_NORMAL_EXP - 7)   # 2**-133 below the normals
    r = np.rint(np.ldexp(xf, -step_exp))     # np.rint: round half to even
    y = np.ldexp(r, step_exp)
    y[np.abs(y) > _BF16_MAX] = np.copysign(np.inf, y[np.abs(y) > _BF16_MAX])
    out[finite] = y
    return out


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round to bf16 (ties to even) and return the uint16 bit patterns."""
    y = round_bf16(x).astype(np.float32)     # exact: y is a bf16 value
    return (y.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
