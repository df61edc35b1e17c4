"""SpQR-style layer: 3-bit g16 dense part with bi-level statistics + fp16 CSR outliers (oracle).

SpQR page, "İddia ve Gerçeklik: SpQR": about 1% of the weights are outliers
kept at fp16 in a sparse matrix; the remaining weights are quantized to 3 bits
in groups of 16 with two-level ("bi-level") quantization; the average storage
is 3.36-4.75 bits per parameter; at run time the dense codes are unpacked
while the sparse fp16 product is applied.

Readings taken where the page is silent (each is restated in the design notes):

1. Outlier choice.  The page selects outliers by Hessian sensitivity, which
   needs calibration data and a model; here the outliers are the
   nnz = floor(f * N * K) entries of largest |w| over the whole matrix
   (f as float64 of the fp32 argument), ties going to the smaller linear
   index n*K + k.
2. First level.  Q_3 (see ``rtn``) over the non-outlier entries of every
   16-wide group gives an fp16 scale s_g and an integer zero z_g; a group
   whose entries are all outliers gets s_g = 1, z_g = 0.
3. Second level ("per 16 groups").  For the 16 consecutive groups of a row
   (a 256-wide supergroup), Q_3 over the 16 values s_g gives (ss, zs, qs_g)
   and Q_3 over the 16 values z_g gives (sz, zz, qz_g): four fp16 numbers per
   supergroup, 3-bit qs and qz per group.
4. Dequantized statistics  s^_g = (qs_g - zs) * ss,  z^_g = (qz_g - zz) * sz
   (fp32, both exact).
5. Dense codes for every entry, outliers included:
   q = 0 if s^_g == 0 else clamp(rint(w / s^_g + z^_g), 0, 7)   (fp32).
6. Dense value D = s^_g * (q - z^_g), fp32, subtraction first, no fused multiply-add.
7. Outlier value val = fp16(w - D) (the residual), so W_hat = D + S is one
   pass with no mask.  At an outlier w_hat = D + float(val) in fp32.
8. CSR rows hold columns in ascending order; columns are int16, so K <= 32768.

Canonical layout (what ``qlin_export`` hands back):
  codes   uint8 [N, 3K/8]        LSB-first bitstream per row, code k at bits 3k..3k+2
  qs, qz  uint8 [N, 3(K/16)/8]   same bitstream form, one 3-bit code per 16-group
  stats   float16 [N, K/256, 4]  (ss, zs, sz, zz) per supergroup
  rowptr int32 [N+1], col int16 [nnz], val float16 [nnz]
"""
import math

import numpy as np

from . import rtn
from .fp import to_fp16

GROUP = 16
SUPER = 256


def outlier_count(N: int, K: int, frac: float) -> int:
    """floor(float64(f) * (N*K)) with f the fp32 outlier fraction."""
    return int(math.floor(float(np.float32(frac)) * float(N * K)))


def select_outliers(W, frac: float) -> np.ndarray:
    """Boolean mask of the nnz largest |w| (ties: smaller linear index first)."""
    W = np.asarray(W, dtype=np.float32)
    N, K = W.shape
    nnz = outlier_count(N, K, frac)
    mask = np.zeros(N * K, dtype=bool)
    if nnz > 0:
        order = np.argsort(-np.abs(W).ravel(), kind="stable")
        mask[order[:nnz]] = True
    return mask.reshape(N, K)


def select_outliers_by_threshold(W, frac: float) -> np.ndarray:
    """Same set as ``select_outliers`` for large matrices: the nnz-th largest |w| found by
    partition, every |w| above it taken, and the entries equal to it taken in index order
    until nnz are chosen."""
    W = np.asarray(W, dtype=np.float32)
    N, K = W.shape
    nnz = outlier_count(N, K, frac)
    a = np.abs(W).ravel()
    mask = np.zeros(a.size, dtype=bool)
    if nnz > 0:
        T = np.partition(a, a.size - nnz)[a.size - nnz]
        above = a > T
        mask |= above
        need = nnz - int(above.sum())
        ties = np.flatnonzero(a == T)[:need]
        mask[ties] = True
    return mask.reshape(N, K)


def pack_bits3(codes) -> np.ndarray:
    """[N, L] 3-bit codes -> uint8 [N, 3L/8] LSB-first bitstream per row."""
    c = np.asarray(codes, dtype=np.uint8)
    N, L = c.shape
    bits = np.stack([(c >> b) & 1 for b in range(3)], axis=-1).reshape(N, 3 * L)
    return np.packbits(bits, axis=1, bitorder="little")


def unpack_bits3(stream, L: int) -> np.ndarray:
    s = np.asarray(stream, dtype=np.uint8)
    N = s.shape[0]
    bits = np.unpackbits(s, axis=1, bitorder="little")[:, : 3 * L].reshape(N, L, 3).astype(np.int64)
    return bits[:, :, 0] | (bits[:, :, 1] << 1) | (bits[:, :, 2] << 2)


def quantize(W, frac: float):
    """Runs readings 1-7.  Returns a dict of intermediate and canonical arrays."""
    W = np.asarray(W, dtype=np.float32)
    _check_shape(W)
    return quantize_with_mask(W, select_outliers(W, frac))


def quantize_rows(W, frac: float, rows):
    """Readings 1-7 for a subset of rows of a large matrix: the outlier set is chosen over the
    whole matrix (reading 1), everything after it is row-local.  Rows come back in the order
    given, as a smaller layer."""
    W = np.asarray(W, dtype=np.float32)
    _check_shape(W)
    mask = select_outliers_by_threshold(W, frac)
    rows = np.asarray(rows)
    return quantize_with_mask(W[rows], mask[rows])


def _check_shape(W):
    N, K = W.shape
    if K % SUPER:
        raise ValueError("K must be a multiple of 256")
    if K > 32768:
        raise ValueError("K must be <= 32768 (int16 CSR columns)")
    if not np.all(np.isfinite(W)):
        raise ValueError("W must be finite")


def quantize_with_mask(W, out_mask):
    """Readings 2-7 given the outlier mask."""
    W = np.asarray(W, dtype=np.float32)
    N, K = W.shape
    G = K // GROUP
    S = K // SUPER

    # first level over the non-outlier entries of each 16-group
    _, s_g, z_g = rtn.quantize_groups(W.reshape(N * G, GROUP), 3, valid=~out_mask.reshape(N * G, GROUP))
    s_g = s_g.reshape(N, G)
    z_g = z_g.reshape(N, G)

    # second level: Q_3 over the 16 scales and over the 16 zeros of each supergroup
    qs, ss, zs = rtn.quantize_groups(s_g.astype(np.float32).reshape(N * S, 16), 3)
    qz, sz, zz = rtn.quantize_groups(z_g.astype(np.float32).reshape(N * S, 16), 3)
    qs = qs.reshape(N, G)
    qz = qz.reshape(N, G)
    ss, zs, sz, zz = (a.reshape(N, S) for a in (ss, zs, sz, zz))

    # dequantized first-level statistics, one per 16-group
    rep = lambda a: np.repeat(a.astype(np.float32), 16, axis=1)  # noqa: E731  supergroup -> group
    s_hat = ((qs.astype(np.float32) - rep(zs)) * rep(ss)).astype(np.float32)
    z_hat = ((qz.astype(np.float32) - rep(zz)) * rep(sz)).astype(np.float32)

    # dense codes and values for every entry
    sh = np.repeat(s_hat, GROUP, axis=1)
    zh = np.repeat(z_hat, GROUP, axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        t = np.rint(W / sh + zh)
    q = np.where(sh == 0, np.float32(0), np.clip(t, 0, 7)).astype(np.int64)
    D = ((q.astype(np.float32) - zh) * sh).astype(np.float32)

    # sparse residuals at the outlier positions, CSR with ascending columns
    rows, cols = np.nonzero(out_mask)
    with np.errstate(over="ignore"):
        val = to_fp16(W[rows, cols] - D[rows, cols])
    if not np.all(np.isfinite(val)):
        raise ValueError("outlier residual overflows fp16")
    rowptr = np.zeros(N + 1, dtype=np.int32)
    np.add.at(rowptr, rows + 1, 1)
    rowptr = np.cumsum(rowptr).astype(np.int32)

    stats = np.stack([ss, zs, sz, zz], axis=-1).astype(np.float16)
    return {
        "mask": out_mask,
        "q": q,
        "s_g": s_g, "z_g": z_g,
        "qs": qs, "qz": qz,
        "s_hat": s_hat, "z_hat": z_hat,
        "D": D,
        "codes": pack_bits3(q),
        "qs_bits": pack_bits3(qs),
        "qz_bits": pack_bits3(qz),
        "stats": stats,
        "rowptr": rowptr,
        "col": cols.astype(np.int16),
        "val": val,
    }


def dequantize(packed) -> np.ndarray:
    """fp32 W_hat = D with D + float(val) at the outlier positions."""
    D = packed["D"].copy()
    rowptr = packed["rowptr"]
    rows = np.repeat(np.arange(len(rowptr) - 1), np.diff(rowptr))
    cols = packed["col"].astype(np.int64)
    D[rows, cols] = (D[rows, cols] + packed["val"].astype(np.float32)).astype(np.float32)
    return D


def dequantize_canonical(N: int, K: int, codes, qs_bits, qz_bits, stats, rowptr, col, val) -> np.ndarray:
    """Dequantizes from the canonical arrays alone (used to check an exported layout)."""
    G = K // GROUP
    q = unpack_bits3(codes, K)
    qs = unpack_bits3(qs_bits, G)
    qz = unpack_bits3(qz_bits, G)
    st = np.asarray(stats, dtype=np.float16).astype(np.float32)
    rep = lambda a: np.repeat(a, 16, axis=1)  # noqa: E731
    s_hat = ((qs.astype(np.float32) - rep(st[:, :, 1])) * rep(st[:, :, 0])).astype(np.float32)
    z_hat = ((qz.astype(np.float32) - rep(st[:, :, 3])) * rep(st[:, :, 2])).astype(np.float32)
    sh = np.repeat(s_hat, GROUP, axis=1)
    zh = np.repeat(z_hat, GROUP, axis=1)
    D = ((q.astype(np.float32) - zh) * sh).astype(np.float32)
    rows = np.repeat(np.arange(N), np.diff(np.asarray(rowptr)))
    cols = np.asarray(col).astype(np.int64)
    D[rows, cols] = (D[rows, cols] + np.asarray(val, dtype=np.float16).astype(np.float32)).astype(np.float32)
    return D


def pack(W, frac: float):
    p = quantize(W, frac)
    p["w_hat"] = dequantize(p)
    return p


def packed_bytes(N: int, K: int, nnz: int) -> int:
    """Canonical bytes: 3-bit codes, 3-bit qs and qz per group, 4 fp16 per supergroup, CSR."""
    return N * (3 * K // 8) + 2 * N * (3 * (K // GROUP) // 8) + N * (K // SUPER) * 8 + 4 * (N + 1) + 4 * nnz
