"""Floating-point helpers of the oracle (numpy only).

fp16 rounding uses numpy's float32 -> float16 cast, which rounds to nearest
even.  bf16 rounding is written out on the float32 bit pattern (round to
nearest even, NaN kept quiet).
"""
import numpy as np


def to_fp16(x) -> np.ndarray:
    """float32 -> float16, round to nearest even."""
    return np.asarray(x, dtype=np.float32).astype(np.float16)


def bf16_round(x) -> np.ndarray:
    """float32 -> bf16 value (returned as float32 holding the bf16 number), RNE."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    is_nan = np.isnan(x)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)) & np.uint64(0xFFFF)
    r = np.where(is_nan, (u >> np.uint64(16)) | np.uint64(0x40), r)
    return (r.astype(np.uint32) << np.uint32(16)).view(np.float32).reshape(x.shape)


def bf16_bits(x) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), RNE."""
    return (bf16_round(x).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def bits_to_f32(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float32 values."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_ulp(v) -> np.ndarray:
    """Spacing of bf16 numbers at |v| (8 significant bits); 2^-133 at zero."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -126.0)
    ulp = np.exp2(e - 7.0)
    return np.where(a > 0, ulp, 2.0 ** -133)
