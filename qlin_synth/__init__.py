"""Seeded synthetic inputs for the quantized linear layer (tests and benchmark).

This module is shared by the oracle side and the GPU side.  It holds no
quantization or matrix arithmetic: it draws numbers from a counter-based
generator (``gen.c``) and shapes them into the workloads the SpQR, GPTQ and
SmoothQuant pages talk about:

* weights ~ N(0, 0.02^2) (GPTQ / SmoothQuant layers) or 0.02 * Student-t(3)
  (heavy-tailed SpQR layer, so that a ~1% outlier set exists);
* activations ~ N(0, 1) in bf16, optionally with 1% of the channels scaled
  by 100 (the activation outlier channels of the SmoothQuant page, "Claim vs
  reality" section);
* the per-channel activation maxima a calibration pass would collect.

Stream keys: X = 1, W = 2, outlier channels = 3, chi-square draws = 4, calibration
block factors = 5.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

KEY_X = 1
KEY_W = 2
KEY_CHANNELS = 3
KEY_CHI = 4
KEY_CALIB = 5

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB_PATH = os.path.join(_HERE, "libqlin_synth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compiles gen.c into libqlin_synth.so next to it (plain gcc, no GPU)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-std=c11", "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            i64, u64, f32 = ctypes.c_int64, ctypes.c_uint64, ctypes.c_float
            vp = ctypes.c_void_p
            lib.qs_normal_f32.argtypes = [u64, u64, f32, i64, vp]
            lib.qs_normal_f32.restype = None
            lib.qs_student_t3_f32.argtypes = [u64, u64, u64, f32, i64, vp]
            lib.qs_student_t3_f32.restype = None
            lib.qs_pick_channels.argtypes = [u64, u64, ctypes.c_int32, ctypes.c_int32, vp]
            lib.qs_pick_channels.restype = ctypes.c_int
            lib.qs_activations_bf16.argtypes = [u64, u64, i64, i64, f32, vp, ctypes.c_int32, f32, vp]
            lib.qs_activations_bf16.restype = ctypes.c_int
            lib.qs_f32_to_bf16.argtypes = [vp, i64, vp]
            lib.qs_f32_to_bf16.restype = None
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def normal(seed: int, key: int, sigma: float, shape) -> np.ndarray:
    """float32 array of sigma * N(0, 1) draws, element i of the flattened shape = draw i."""
    out = np.empty(shape, dtype=np.float32)
    _load().qs_normal_f32(seed, key, sigma, out.size, _ptr(out))
    return out


def student_t3(seed: int, scale: float, shape, key_z: int = KEY_W, key_chi: int = KEY_CHI) -> np.ndarray:
    """float32 array of scale * Student-t(nu=3) draws."""
    out = np.empty(shape, dtype=np.float32)
    _load().qs_student_t3_f32(seed, key_z, key_chi, scale, out.size, _ptr(out))
    return out


def pick_channels(seed: int, K: int, count: int, key: int = KEY_CHANNELS) -> np.ndarray:
    """Sorted int32 array of `count` distinct channel indices in [0, K)."""
    out = np.empty(count, dtype=np.int32)
    rc = _load().qs_pick_channels(seed, key, K, count, _ptr(out))
    if rc != 0:
        raise ValueError("pick_channels: bad arguments")
    return out


def activations_bf16(seed: int, M: int, K: int, sigma: float = 1.0, boosted=None, boost: float = 100.0,
                     key: int = KEY_X) -> np.ndarray:
    """uint16 array [M, K] holding bf16 bit patterns of sigma * N(0, 1), boosted channels x boost."""
    out = np.empty((M, K), dtype=np.uint16)
    if boosted is not None and len(boosted):
        ch = np.ascontiguousarray(boosted, dtype=np.int32)
        rc = _load().qs_activations_bf16(seed, key, M, K, sigma, _ptr(ch), len(ch), boost, _ptr(out))
    else:
        rc = _load().qs_activations_bf16(seed, key, M, K, sigma, None, 0, boost, _ptr(out))
    if rc != 0:
        raise ValueError("activations_bf16: bad arguments")
    return out


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widens bf16 bit patterns (uint16) to float32 values (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """Rounds float32 values to bf16 bit patterns (round to nearest even)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().qs_f32_to_bf16(_ptr(x), x.size, _ptr(out))
    return out


def outlier_channel_count(K: int) -> int:
    """floor(0.01 * K): the 1% of activation channels that carry outliers."""
    return (K * 1) // 100


def channel_absmax(x_bits: np.ndarray) -> np.ndarray:
    """Per-channel max |x| over the rows of a bf16 activation matrix (a calibration pass)."""
    return np.abs(bf16_to_f32(x_bits)).max(axis=0).astype(np.float32)


# -- workload recipes ------------------------------------------------------------------------------

def gptq_layer(N: int, K: int, M: int, seed: int = 0):
    """W4g128 workload: W ~ N(0, 0.02^2) fp32 [N, K]; X ~ N(0, 1) bf16 [M, K]."""
    W = normal(seed, KEY_W, 0.02, (N, K))
    X = activations_bf16(seed, M, K)
    return W, X


def spqr_layer(N: int, K: int, M: int, seed: int = 0):
    """SpQR workload: W ~ 0.02 * Student-t(3) fp32 [N, K]; X ~ N(0, 1) bf16 [M, K]."""
    W = student_t3(seed, 0.02, (N, K))
    X = activations_bf16(seed, M, K)
    return W, X


def spqr_quiet_group_layer(N: int, K: int, seed: int = 0):
    """An SpQR test layer with one near-silent 16-group per row.

    W ~ N(0, 0.02^2); in row r the entries of 16-group (5 r) mod (K / 16) are scaled by 1e-3,
    except one (entry r mod 16 of the group), which is set to 1 + r 2^-10 -- larger than every
    other weight, distinct per row.  With N outliers the large values are exactly the outlier
    set, and the group's other entries are far below its supergroup's scales (the case where
    a group's 3-bit scale code is 0).
    """
    W = normal(seed, KEY_W, 0.02, (N, K))
    G = K // 16
    for r in range(N):
        g = (5 * r) % G
        W[r, 16 * g:16 * g + 16] *= np.float32(1e-3)
        W[r, 16 * g + r % 16] = np.float32(1.0 + r * 2.0 ** -10)
    return W.astype(np.float32)


def gptq_calibration(S: int, K: int, seed: int = 0, block: int = 16) -> np.ndarray:
    """Calibration rows for the GPTQ packer: fp32 [S, K] of bf16 values.

    x[s, k] = z[s, k] + c[s, k // block] with z, c ~ N(0, 1) on their own streams, so the
    channels of a block are correlated as real layer inputs are (an identity covariance would
    leave nothing to compensate); rounded to bf16, and |x| < 2^-8 set to 0, so that every
    product of two inputs is a multiple of 2^-30 and X^T X is exact in fp64 whatever the
    summation order (for S * max|x|^2 < 2^23).
    """
    z = normal(seed, KEY_X, 1.0, (S, K))
    c = normal(seed, KEY_CALIB, 1.0, (S, (K + block - 1) // block))
    x = bf16_to_f32(f32_to_bf16(z + np.repeat(c, block, axis=1)[:, :K]))
    return np.where(np.abs(x) < np.float32(2.0 ** -8), np.float32(0), x).astype(np.float32)


def smoothquant_layer(N: int, K: int, M: int, seed: int = 0):
    """W8A8 workload: W ~ N(0, 0.02^2); X ~ N(0, 1) bf16 with floor(0.01 K) channels x100.

    Returns (W, X, act_absmax, channels); act_absmax is the per-channel max |X| of the same X,
    standing in for the calibration set.
    """
    W = normal(seed, KEY_W, 0.02, (N, K))
    ch = pick_channels(seed, K, outlier_channel_count(K))
    X = activations_bf16(seed, M, K, boosted=ch, boost=100.0)
    return W, X, channel_absmax(X), ch
