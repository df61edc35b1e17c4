"""Asymmetric round-to-nearest group quantizer Q_b (oracle).

The GPTQ page (intro and "İddia ve Gerçeklik: GPTQ") names round-to-nearest
(RTN) as the baseline quantizer of a weight group; the SpQR page ("İddia ve
Gerçeklik: SpQR") quantizes groups of 16 -- and their statistics -- to 3 bits.
Neither page writes the quantizer out.  Reading taken: min-max asymmetric RTN
whose range always contains 0, with an fp16 scale and an integer zero point:

    lo = min(0, min v)     hi = max(0, max v)
    hi == lo  ->  scale = 1, z = 0
    otherwise     scale = fp16((hi - lo) / (2^b - 1))   (fp32 divide, RNE to fp16)
                  scale == 0 -> scale = 2^-24
                  z = clamp(rint(-lo / scale), 0, 2^b - 1)
    q_i = clamp(rint(v_i / scale) + z, 0, 2^b - 1)
    dequant  w_hat_i = (q_i - z) * scale   (exact in fp32)

All arithmetic that decides a code is fp32 with IEEE division and
round-half-to-even ``rint``.  A scale that overflows fp16 is an input error.
"""
import numpy as np

from .fp import to_fp16


def quantize_groups(v, bits: int, valid=None):
    """Applies Q_b to every row of ``v`` ([G, n] float32).

    ``valid`` ([G, n] bool, optional) restricts the min/max to the marked
    entries (the SpQR first level excludes outliers); codes are still produced
    for every entry.  A row without valid entries has lo = hi = 0, so it gets
    scale 1 and zero 0.

    Returns (q int64 [G, n], scale float16 [G], zero float16 [G]).
    """
    v = np.asarray(v, dtype=np.float32)
    qmax = np.float32(2 ** bits - 1)
    if valid is None:
        vmin = v.min(axis=1)
        vmax = v.max(axis=1)
    else:
        vmin = np.where(valid, v, np.float32(np.inf)).min(axis=1)
        vmax = np.where(valid, v, np.float32(-np.inf)).max(axis=1)
        vmin = np.where(np.isfinite(vmin), vmin, np.float32(0))
        vmax = np.where(np.isfinite(vmax), vmax, np.float32(0))
    lo = np.minimum(np.float32(0), vmin).astype(np.float32)
    hi = np.maximum(np.float32(0), vmax).astype(np.float32)
    flat = hi == lo
    with np.errstate(over="ignore"):
        scale16 = to_fp16((hi - lo) / qmax)
    if not np.all(np.isfinite(scale16)):
        raise ValueError("group range too large: scale overflows fp16")
    scale16 = np.where(scale16 == 0, np.float16(2.0 ** -24), scale16).astype(np.float16)
    scale16 = np.where(flat, np.float16(1.0), scale16).astype(np.float16)
    scale = scale16.astype(np.float32)
    z = np.clip(np.rint(-lo / scale), 0, qmax)
    z = np.where(flat, np.float32(0), z).astype(np.float32) + np.float32(0)  # -0.0 -> +0.0
    q = np.clip(np.rint(v / scale[:, None]) + z[:, None], 0, qmax)
    return q.astype(np.int64), scale16, z.astype(np.float16)


def dequantize_groups(q, scale16, zero16) -> np.ndarray:
    """w_hat = (q - z) * scale per group, fp32 (exact: |q - z| < 2^8, scale has 11 bits)."""
    qf = np.asarray(q).astype(np.float32)
    z = np.asarray(zero16).astype(np.float32)[:, None]
    s = np.asarray(scale16).astype(np.float32)[:, None]
    return ((qf - z) * s).astype(np.float32)
