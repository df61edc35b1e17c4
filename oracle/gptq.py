"""GPTQ error-compensating W4 g128 quantizer (oracle).

GPTQ page, "Makale Bülteni — GPTQ" (intro) and "İddia ve Gerçeklik: GPTQ"
(second paragraph): the layer is quantized with a second-order (Taylor / OBS)
view of its output error.  The inverse Hessian comes from the covariance of the
layer's inputs and is made stable through a Cholesky decomposition; weights are
quantized column after column, in blocks of 128, and the rounding error of each
quantized column is spread at once over the columns not yet quantized, so that
it does not pile up.

The page names the steps, not the formulae.  Readings taken:

1. H = Xcal^T Xcal in fp64 over the calibration rows (a constant factor in front
   of H changes nothing below).
2. A column with H_kk == 0 (an input that is always zero) gets H_kk = 1 and its
   weights are set to 0 before quantization: it never reaches the output.
3. Damping, for the Cholesky decomposition: H += damp * mean(diag H) * I with
   damp = 0.01.
4. U is the upper Cholesky factor of H^-1 (H^-1 = U^T U).
5. Columns k = 0 .. K-1 in order.  At the first column of each 128-wide group
   the group's fp16 scale and integer zero come from the round-to-nearest
   quantizer Q_4 (oracle.rtn) applied to the group's current, already updated
   weights cast to fp32.  Column k is quantized with them exactly as Q_4 does
   (fp32, IEEE division, round half to even, clamp to 0..15); with
   e = (w_k - w_hat_k) / U_kk, every later column j of the row becomes
   w_j - e * U_kj (fp64, a product then a difference).
   The page batches the updates of a 128-block for speed; this is the same
   arithmetic column by column, without the batching.
6. The result is the W4 g128 canonical layout of oracle.gptq_w4 (codes, scale,
   zero), read by the same kernels as round-to-nearest codes.

With H = I, every U_kj with j > k is 0, no weight moves, and the codes are the
round-to-nearest codes bit for bit.

Act-order (GPTQ page, "İddia ve Gerçeklik: GPTQ", last paragraph: columns sorted by
activation size, at the price of irregular groups at run time).  Reading: the column order
is perm = the columns by decreasing diag(H) (after reading 2, ties to the smaller index);
the layer W[:, perm] is quantized as above under H[perm][:, perm], so its 128-groups are
contiguous in the permuted order; the forward then multiplies by X[:, perm].  With diag(H)
already non-increasing, perm is the identity and nothing changes.
"""
import numpy as np

from . import gptq_w4, rtn

GROUP = gptq_w4.GROUP


def hessian(Xcal) -> np.ndarray:
    """H = Xcal^T Xcal, fp64 [K, K] (reading 1)."""
    X = np.asarray(Xcal, dtype=np.float64)
    return X.T @ X


def inverse_cholesky_upper(H, damp: float = 0.01):
    """Readings 2-4: returns (U upper-triangular fp64 [K, K], dead bool [K])."""
    H = np.array(H, dtype=np.float64)
    K = H.shape[0]
    dead = np.diag(H) == 0
    H[dead, dead] = 1.0
    H = H + damp * np.mean(np.diag(H)) * np.eye(K)
    Hinv = np.linalg.inv(H)
    L = np.linalg.cholesky(Hinv)  # Hinv = L L^T, L lower
    return L.T, dead


def quantize(W, H, damp: float = 0.01):
    """GPTQ W4 g128 of W (fp32 [N, K]) under Hessian H [K, K].

    Returns (q int64 [N, K], scale f16 [N, K/128], zero f16 [N, K/128]).
    """
    W = np.array(W, dtype=np.float32)
    N, K = W.shape
    if K % GROUP:
        raise ValueError("K must be a multiple of 128")
    if not np.all(np.isfinite(W)):
        raise ValueError("W must be finite")
    U, dead = inverse_cholesky_upper(H, damp)
    Wd = W.astype(np.float64)
    Wd[:, dead] = 0.0
    G = K // GROUP
    q = np.zeros((N, K), dtype=np.int64)
    scale = np.zeros((N, G), dtype=np.float16)
    zero = np.zeros((N, G), dtype=np.float16)
    for k in range(K):
        g = k // GROUP
        if k % GROUP == 0:
            _, s_g, z_g = rtn.quantize_groups(Wd[:, k:k + GROUP].astype(np.float32), 4)
            scale[:, g], zero[:, g] = s_g, z_g
        s32 = scale[:, g].astype(np.float32)
        z32 = zero[:, g].astype(np.float32)
        w32 = Wd[:, k].astype(np.float32)
        qk = np.clip(np.rint(w32 / s32) + z32, np.float32(0), np.float32(15))
        q[:, k] = qk.astype(np.int64)
        w_hat = ((qk - z32) * s32).astype(np.float32)
        e = (Wd[:, k] - w_hat.astype(np.float64)) / U[k, k]
        Wd[:, k + 1:] -= e[:, None] * U[k, k + 1:][None, :]
    return q, scale, zero


def act_order(H) -> np.ndarray:
    """perm: the columns by decreasing diag(H), dead columns counted as 1, ties to the smaller index."""
    d = np.array(np.diag(np.asarray(H, dtype=np.float64)))
    d[d == 0] = 1.0
    return np.argsort(-d, kind="stable").astype(np.int32)


def pack(W, Xcal, damp: float = 0.01, act: bool = False):
    """Canonical arrays (as oracle.gptq_w4.pack) plus the fp32 dequantized matrix.

    act: act-order; then codes/scale/zero are those of W[:, perm], "perm" is returned, and
    "w_hat" is in the original column order (w_hat[:, perm] = the permuted dequantization).
    """
    H = hessian(Xcal)
    if not act:
        q, s, z = quantize(W, H, damp)
        return {"codes": gptq_w4.pack_codes(q), "scale": s, "zero": z, "q": q,
                "w_hat": gptq_w4.dequantize(q, s, z)}
    perm = act_order(H)
    q, s, z = quantize(np.asarray(W, dtype=np.float32)[:, perm], H[np.ix_(perm, perm)], damp)
    w_perm = gptq_w4.dequantize(q, s, z)
    w_hat = np.empty_like(w_perm)
    w_hat[:, perm] = w_perm
    return {"codes": gptq_w4.pack_codes(q), "scale": s, "zero": z, "q": q, "perm": perm,
            "w_hat_perm": w_perm, "w_hat": w_hat}


def output_error(W, w_hat, Xcal) -> float:
    """||(W - W_hat) Xcal^T||_F^2 in fp64: the layer-output error GPTQ lowers."""
    D = np.asarray(W, dtype=np.float64) - np.asarray(w_hat, dtype=np.float64)
    R = D @ np.asarray(Xcal, dtype=np.float64).T
    return float(np.sum(R * R))
