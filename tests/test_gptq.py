"""GPTQ error-compensating W4 g128 quantizer: oracle pins and the host packer (CPU only).

GPTQ page, "İddia ve Gerçeklik: GPTQ": inverse Hessian from the layer-input covariance,
Cholesky-stabilised; columns quantized in order with each column's rounding error spread
over the columns not yet quantized.  Pins, each aimed at a plausible slip:

* H = c I: no cross-column term, so the codes are the round-to-nearest codes bit for bit
  (an update that leaks through the diagonal, or a mis-scaled U, fails it);
* two correlated inputs, everything else identity: after column 0 is quantized, column 1
  moves by (w0 - w_hat0) * b / (c + d) -- the second-order update written out by hand from
  the 2 x 2 inverse (a wrong sign, a transposed U or a missing damping term fails it);
* the purpose the page gives: the layer-output error on the calibration rows drops well
  below round-to-nearest's;
* an always-zero input column quantizes its weights to exactly 0;
* the packer (C++) agrees with the oracle code for code on seeded layers.
"""
import numpy as np
import pytest

import qlin_synth as synth
from oracle import gptq, gptq_w4


def _f16_bits(a):
    return np.asarray(a).view(np.uint16)


@pytest.mark.parametrize("c", [1.0, 3.5])
def test_identity_hessian_gives_rtn(c):
    K = 256
    W = synth.normal(11, synth.KEY_W, 0.02, (48, K))
    q, s, z = gptq.quantize(W, c * np.eye(K))
    q0, s0, z0 = gptq_w4.quantize(W)
    assert np.array_equal(q, q0)
    assert np.array_equal(_f16_bits(s), _f16_bits(s0)) and np.array_equal(_f16_bits(z), _f16_bits(z0))


def test_two_correlated_inputs_closed_form():
    K, N, damp = 128, 64, 0.01
    a, b, c = 1.0, 0.5, 1.25
    H = np.eye(K)
    H[0, 0], H[0, 1], H[1, 0], H[1, 1] = a, b, b, c
    W = synth.normal(5, synth.KEY_W, 0.02, (N, K))
    q, s, z = gptq.quantize(W, H, damp)
    # by hand: the group statistics are fixed at column 0 from the original weights
    q_rtn, s0, z0 = gptq_w4.quantize(W)
    assert np.array_equal(_f16_bits(s), _f16_bits(s0)) and np.array_equal(_f16_bits(z), _f16_bits(z0))
    s32, z32 = s0[:, 0].astype(np.float32), z0[:, 0].astype(np.float32)
    d = damp * (a + c + (K - 2)) / K
    w0_hat = (q_rtn[:, 0].astype(np.float32) - z32) * s32
    w1 = W[:, 1].astype(np.float64) + (W[:, 0].astype(np.float64) - w0_hat.astype(np.float64)) * b / (c + d)
    q1 = np.clip(np.rint(w1.astype(np.float32) / s32) + z32, 0, 15).astype(np.int64)
    assert np.array_equal(q[:, 0], q_rtn[:, 0])
    assert np.array_equal(q[:, 1], q1)
    assert np.any(q1 != q_rtn[:, 1])  # the update does move codes
    assert np.array_equal(q[:, 2:], q_rtn[:, 2:])  # uncorrelated columns are untouched


def test_lowers_calibration_output_error():
    N, K, S = 64, 256, 512
    W = synth.normal(9, synth.KEY_W, 0.02, (N, K))
    X = synth.gptq_calibration(S, K, seed=9)
    g = gptq.pack(W, X)
    r = gptq_w4.pack(W)
    assert gptq.output_error(W, g["w_hat"], X) < 0.5 * gptq.output_error(W, r["w_hat"], X)
    # and every weight still sits on its group's grid (same format as round-to-nearest)
    assert np.array_equal(g["w_hat"], gptq_w4.dequantize(g["q"], g["scale"], g["zero"]))


def test_dead_input_column_is_zero():
    N, K, S = 16, 128, 200
    W = synth.normal(4, synth.KEY_W, 0.02, (N, K))
    X = synth.gptq_calibration(S, K, seed=4)
    X[:, [5, 77]] = 0.0
    g = gptq.pack(W, X)
    assert np.all(g["w_hat"][:, [5, 77]] == 0.0)


@pytest.mark.parametrize("N,K,S", [(64, 256, 256), (100, 512, 128), (33, 384, 200)])
def test_packer_matches_oracle(qlin, N, K, S):
    W = synth.normal(7, synth.KEY_W, 0.02, (N, K))
    X = synth.gptq_calibration(S, K, seed=7)
    X[:, 3] = 0.0  # one dead input
    h = qlin.qlin_pack_w4g128_gptq(W, X)
    ex = qlin.qlin_export(h)
    ref = gptq.pack(W, X)
    assert np.array_equal(ex["codes"], ref["codes"])
    assert np.array_equal(_f16_bits(ex["scale"]), _f16_bits(ref["scale"]))
    assert np.array_equal(_f16_bits(ex["zero"]), _f16_bits(ref["zero"]))
    assert h.info.packed_bytes == gptq_w4.packed_bytes(N, K)


def test_packer_identity_calibration_equals_rtn_packer(qlin):
    K = 256
    W = synth.normal(2, synth.KEY_W, 0.02, (40, K))
    a = qlin.qlin_export(qlin.qlin_pack_w4g128_gptq(W, np.eye(K, dtype=np.float32)))
    b = qlin.qlin_export(qlin.qlin_pack_w4g128(W))
    for key in ("codes", "scale", "zero"):
        assert np.array_equal(np.asarray(a[key]).view(np.uint8), np.asarray(b[key]).view(np.uint8)), key


def test_packer_rejects_bad_arguments(qlin):
    W = synth.normal(1, synth.KEY_W, 0.02, (8, 256))
    X = synth.gptq_calibration(16, 256, seed=1)
    with pytest.raises(qlin.QlinError):
        qlin.qlin_pack_w4g128_gptq(W[:, :200], X[:, :200])  # K % 128 != 0
    with pytest.raises(qlin.QlinError):
        qlin.qlin_pack_w4g128_gptq(W, X, damp=0.0)
    bad = X.copy()
    bad[0, 0] = np.nan
    with pytest.raises(qlin.QlinError):
        qlin.qlin_pack_w4g128_gptq(W, bad)
    with pytest.raises(ValueError):
        qlin.qlin_pack_w4g128_gptq(W, X[:, :128])  # calibration width != K
    big = np.zeros((2, 8320), dtype=np.float32)
    with pytest.raises(qlin.QlinError):
        qlin.qlin_pack_w4g128_gptq(big, big)  # K > 8192


# ----------------------------------------------------------------------------- act-order

def _uneven(X):
    """Channel scales 1/4 .. 4 (powers of two keep X^T X exact)."""
    K = X.shape[1]
    return (X * (2.0 ** (np.arange(K) % 5 - 2))[None, :]).astype(np.float32)


def test_act_order_sorts_by_decreasing_diagonal():
    H = np.diag([3.0, 5.0, 0.0, 5.0, 2.0, 1.0])  # the dead input counts as 1; 5 vs 5 keeps index order
    assert list(gptq.act_order(H)) == [1, 3, 0, 4, 2, 5]


def test_act_order_is_invariant_to_input_order():
    """Relabelling the input channels of W and of the calibration rows relabels W_hat the same
    way: the order comes from diag(H) alone, and the codes follow their channels."""
    N, K, S = 40, 256, 300
    W = synth.normal(12, synth.KEY_W, 0.02, (N, K))
    X = _uneven(synth.gptq_calibration(S, K, seed=12))
    P = np.random.default_rng(12).permutation(K)
    a = gptq.pack(W, X, act=True)
    b = gptq.pack(W[:, P], X[:, P], act=True)
    assert np.array_equal(b["w_hat"].view(np.uint32), a["w_hat"][:, P].view(np.uint32))


def test_act_order_lowers_error_with_uneven_channels():
    N, K, S = 64, 256, 256
    W = synth.normal(7, synth.KEY_W, 0.02, (N, K))
    X = _uneven(synth.gptq_calibration(S, K, seed=7))
    act, plain = gptq.pack(W, X, act=True), gptq.pack(W, X)
    assert gptq.output_error(W, act["w_hat"], X) < 0.8 * gptq.output_error(W, plain["w_hat"], X)


@pytest.mark.parametrize("N,K,S", [(64, 256, 256), (100, 512, 300)])
def test_packer_matches_oracle_act_order(qlin, N, K, S):
    W = synth.normal(7, synth.KEY_W, 0.02, (N, K))
    X = _uneven(synth.gptq_calibration(S, K, seed=7))
    ex = qlin.qlin_export(qlin.qlin_pack_w4g128_gptq(W, X, act_order=True))
    ref = gptq.pack(W, X, act=True)
    for key in ("codes", "scale", "zero", "perm"):
        assert np.array_equal(np.asarray(ex[key]).view(np.uint8), np.asarray(ref[key]).view(np.uint8)), key
