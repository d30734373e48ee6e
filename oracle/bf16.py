"""bfloat16 conversions for the oracle (test infrastructure only).

bfloat16 keeps the sign, the 8 exponent bits and the top 7 fraction bits of an IEEE
binary32 value.  Widening appends 16 zero bits (exact).  Narrowing rounds the
discarded 16 bits to nearest, ties to even; NaN stays a quiet NaN.
"""
import numpy as np


def to_bf16(x) -> np.ndarray:
    """fp32 (or anything castable to fp32) -> bf16 bit patterns (uint16), RNE."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    bits = f.view(np.uint32).astype(np.uint64)
    upper = bits >> np.uint64(16)
    lower = bits & np.uint64(0xFFFF)
    round_up = (lower > 0x8000) | ((lower == 0x8000) & ((upper & np.uint64(1)) == 1))
    out = (upper + round_up.astype(np.uint64)) & np.uint64(0xFFFF)
    out = out.astype(np.uint16)
    nan = np.isnan(f)
    if nan.any():
        out[nan] = (upper[nan].astype(np.uint16) & np.uint16(0x8000)) | np.uint16(0x7FC0)
    return out


def bf16_to_f64(b) -> np.ndarray:
    """bf16 bit patterns -> float64 (exact)."""
    u = np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def bf16_to_f32(b) -> np.ndarray:
    u = np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32)


def f64_to_bf16(x) -> np.ndarray:
    """float64 -> bf16 bit patterns, correctly rounded (nearest, ties to even).

    Goes through fp32 with round-to-odd (truncate toward zero, set the last bit when
    anything was discarded), which keeps the final RNE step free of double rounding
    because fp32 carries 16 more fraction bits than bf16.
    """
    d = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    f = d.astype(np.float32)
    back = f.astype(np.float64)
    inexact = back != d
    overshoot = inexact & (np.abs(back) > np.abs(d))
    f = np.where(overshoot, np.nextafter(f, np.float32(0)), f).astype(np.float32)
    bits = f.view(np.uint32).copy()
    bits[inexact] |= np.uint32(1)
    return to_bf16(bits.view(np.float32))


def round_to_bf16_f64(x) -> np.ndarray:
    """Round float64 values to the nearest bf16 value and return it as float64."""
    return bf16_to_f64(f64_to_bf16(x))
