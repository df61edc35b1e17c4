"""fp64 reference forward, the tolerance bound and bits per parameter (oracle).

Forward (all formats with a dequantized matrix): y_ref[m, n] = sum_k x[m, k] * w_hat[n, k]
in float64 (x from bf16, w_hat the fp32 dequantized weights).

Tolerance of a bf16 output y (from the stated target): |y - y_ref| <= 1e-2 * B[m, n] + ulp_bf16(y_ref),
with B[m, n] = sum_k |x[m, k] * w_hat[n, k]|.
"""
import numpy as np

from .fp import bf16_ulp


def reference(x, w_hat):
    """Returns (y_ref float64 [M, N], B float64 [M, N])."""
    x64 = np.asarray(x, dtype=np.float64)
    w64 = np.asarray(w_hat, dtype=np.float64)
    return x64 @ w64.T, np.abs(x64) @ np.abs(w64).T


def reference_rows(x, w_hat, rows):
    """Same as ``reference`` on a subset of the rows of x (large-M sampling)."""
    return reference(np.asarray(x)[rows], w_hat)


def tolerance(y_ref, bound, rel: float = 1e-2):
    return rel * np.asarray(bound) + bf16_ulp(y_ref)


def within_tolerance(y, y_ref, bound, rel: float = 1e-2):
    """Elementwise check; returns (ok bool, worst ratio |err| / tol)."""
    err = np.abs(np.asarray(y, dtype=np.float64) - y_ref)
    tol = tolerance(y_ref, bound, rel)
    ratio = err / tol
    return bool(np.all(err <= tol)), float(ratio.max()) if ratio.size else 0.0


def bits_per_param(packed_bytes: int, N: int, K: int) -> float:
    return 8.0 * packed_bytes / (N * K)
