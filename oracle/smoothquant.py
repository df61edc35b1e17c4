"""SmoothQuant W8A8 (oracle).

SmoothQuant page, "İddia ve Gerçeklik: SmoothQuant": the layer is rewritten
as Y = (X diag(s)^-1)(diag(s) W); the per-channel vector s divides the
activation peaks and is folded into the weights offline; activations are then
quantized per token and weights per output channel to int8 and fed to an int8
GEMM; the migration strength alpha is usually 0.8-0.85; the activation maxima
come from a calibration set.

The smoothing formula s_j = max|X_j|^alpha / max|W_j|^(1-alpha) is the
method's published one (the pages name the vector and alpha but do not print
the formula).  Readings taken:

* act_absmax[k] (the calibration statistic) is an input; the tests pass the
  per-channel max |x| of the same synthetic X.
* s_k = fp32( max(ax_k, 1e-5)^alpha / max(aw_k, 1e-5)^(1-alpha) ) in float64,
  aw_k = max_n |W[n, k]|, alpha = float64 of the fp32 argument.  The 1e-5
  floor keeps s finite on dead channels.  pow is the C library's, called per
  element.
* s_inv_k = 1 / s_k in fp32.
* W'[n, k] = W[n, k] * s_k (fp32); sw_n = max_k |W'[n, k]| / 127 (1 if that is 0);
  qw = clamp(rint(W' / sw_n), -127, 127).
* x'[m, k] = x[m, k] * s_inv_k (fp32); sx_m = max_k |x'[m, k]| / 127 (1 if 0);
  qx = clamp(rint(x' / sx_m), -127, 127).  IEEE division, not a reciprocal.
* acc[m, n] = sum_k qx * qw exactly (int64 here; it must fit int32).
* y = bf16( (fp32(acc) * sx_m) * sw_n ), two fp32 multiplies in that order.
"""
import math

import numpy as np

from .fp import bf16_round


def smoothing_factors(act_absmax, W, alpha: float):
    """Returns (s fp32 [K], s_inv fp32 [K])."""
    W = np.asarray(W, dtype=np.float32)
    ax = np.asarray(act_absmax, dtype=np.float32)
    aw = np.abs(W).max(axis=0)
    a = float(np.float32(alpha))
    s = np.empty(ax.shape[0], dtype=np.float32)
    for k in range(ax.shape[0]):
        num = math.pow(max(float(ax[k]), 1e-5), a)
        den = math.pow(max(float(aw[k]), 1e-5), 1.0 - a)
        s[k] = np.float32(num / den)
    s_inv = (np.float32(1.0) / s).astype(np.float32)
    return s, s_inv


def fold_weights(W, s) -> np.ndarray:
    """diag(s) folded into W along the input channel: W'[n, k] = W[n, k] * s_k (fp32)."""
    return (np.asarray(W, dtype=np.float32) * np.asarray(s, dtype=np.float32)[None, :]).astype(np.float32)


def scale_activations(x, s_inv) -> np.ndarray:
    """X diag(s)^-1 as an fp32 multiply by s_inv: x'[m, k] = x[m, k] * s_inv_k."""
    return (np.asarray(x, dtype=np.float32) * np.asarray(s_inv, dtype=np.float32)[None, :]).astype(np.float32)


def quantize_rows_int8(a):
    """Symmetric per-row int8: scale = max|a_row| / 127 (1 if 0), q = clamp(rint(a / scale), +-127)."""
    a = np.asarray(a, dtype=np.float32)
    amax = np.abs(a).max(axis=1)
    scale = (amax / np.float32(127)).astype(np.float32)
    scale = np.where(amax == 0, np.float32(1), scale).astype(np.float32)
    q = np.clip(np.rint(a / scale[:, None]), -127, 127).astype(np.int8)
    return q, scale


def quantize_weights(W, act_absmax, alpha: float):
    """Offline part: smoothing factors, folded weights, per-channel int8."""
    s, s_inv = smoothing_factors(act_absmax, W, alpha)
    qw, sw = quantize_rows_int8(fold_weights(W, s))
    return {"s": s, "s_inv": s_inv, "qw": qw, "sw": sw}


def quantize_activations(x, s_inv):
    """Run-time part: per-token int8 codes and fp32 scales of X diag(s)^-1."""
    return quantize_rows_int8(scale_activations(x, s_inv))


def accumulate(qx, qw) -> np.ndarray:
    """Exact integer accumulators acc[m, n] = sum_k qx[m, k] * qw[n, k] (int64)."""
    return np.asarray(qx, dtype=np.int64) @ np.asarray(qw, dtype=np.int64).T


def epilogue(acc, sx, sw) -> np.ndarray:
    """y = bf16((fp32(acc) * sx_m) * sw_n), returned as float32 bf16 values."""
    a = np.asarray(acc).astype(np.float32)
    y = (a * np.asarray(sx, dtype=np.float32)[:, None]).astype(np.float32)
    y = (y * np.asarray(sw, dtype=np.float32)[None, :]).astype(np.float32)
    return bf16_round(y)


def forward(x, packed):
    """Full W8A8 forward; returns (y bf16-valued fp32 [M, N], acc int64, qx, sx)."""
    qx, sx = quantize_activations(x, packed["s_inv"])
    acc = accumulate(qx, packed["qw"])
    return epilogue(acc, sx, packed["sw"]), acc, qx, sx


def packed_bytes(N: int, K: int) -> int:
    """int8 weights, fp32 per-channel scale, fp32 s_inv per input channel."""
    return N * K + 4 * N + 4 * K
