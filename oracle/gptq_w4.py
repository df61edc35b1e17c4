"""W4 g128: 4-bit weights in 128-wide K groups with an fp16 scale and zero (oracle).

GPTQ page: weights quantized to 4 bits in blocks of 128 ("İddia ve Gerçeklik:
GPTQ", second paragraph), weight-only, activations stay 16-bit (third
paragraph).  The codes here come from round-to-nearest (the baseline quantizer
the GPTQ page contrasts with its error-compensating one); the packed format is
what GPTQ-format checkpoints hold, so kernels are the same either way.

Canonical layout (the format ``qlin_export`` hands back):
  codes  uint32 [N, K/8]   nibble i (bits 4i..4i+3) of word j holds k = 8j + i
  scale  float16 [N, K/128]
  zero   float16 [N, K/128]   integer valued, 0..15
"""
import numpy as np

from . import rtn

GROUP = 128


def quantize(W):
    """RTN 4-bit per (row, 128-group).  Returns (q int64 [N, K], scale f16 [N, K/128], zero f16)."""
    W = np.asarray(W, dtype=np.float32)
    N, K = W.shape
    if K % GROUP:
        raise ValueError("K must be a multiple of 128")
    if not np.all(np.isfinite(W)):
        raise ValueError("W must be finite")
    G = K // GROUP
    q, s, z = rtn.quantize_groups(W.reshape(N * G, GROUP), 4)
    return q.reshape(N, K), s.reshape(N, G), z.reshape(N, G)


def pack_codes(q) -> np.ndarray:
    """[N, K] codes in 0..15 -> uint32 [N, K/8], nibble i of word j = code 8j + i."""
    q = np.asarray(q, dtype=np.uint32)
    N, K = q.shape
    q8 = q.reshape(N, K // 8, 8)
    words = np.zeros((N, K // 8), dtype=np.uint32)
    for i in range(8):
        words |= q8[:, :, i] << np.uint32(4 * i)
    return words


def unpack_codes(words) -> np.ndarray:
    words = np.asarray(words, dtype=np.uint32)
    N, W8 = words.shape
    out = np.empty((N, W8, 8), dtype=np.int64)
    for i in range(8):
        out[:, :, i] = (words >> np.uint32(4 * i)) & np.uint32(0xF)
    return out.reshape(N, W8 * 8)


def dequantize(q, scale16, zero16) -> np.ndarray:
    """fp32 W_hat [N, K] = (q - z_g) * s_g."""
    q = np.asarray(q)
    N, K = q.shape
    G = K // GROUP
    w = rtn.dequantize_groups(q.reshape(N * G, GROUP), np.asarray(scale16).reshape(-1),
                              np.asarray(zero16).reshape(-1))
    return w.reshape(N, K)


def pack(W):
    """Full oracle pack: dict with canonical arrays and the fp32 dequantized matrix."""
    q, s, z = quantize(W)
    return {"codes": pack_codes(q), "scale": s, "zero": z, "q": q, "w_hat": dequantize(q, s, z)}


def packed_bytes(N: int, K: int) -> int:
    """Bytes of the canonical layout: N*K/2 code bytes + 2 fp16 per 128-group."""
    return N * K // 2 + N * (K // GROUP) * 4
