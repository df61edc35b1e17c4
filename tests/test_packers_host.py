"""Host packers of libqlin against the oracle, code for code (CPU only).

The packers and the oracle are separate implementations of the same readings;
every canonical array must agree bit for bit.
"""
import numpy as np
import pytest

import qlin_synth as synth
from oracle import gptq_w4, smoothquant, spqr


@pytest.mark.parametrize("N,K", [(64, 512), (50, 256), (130, 1024)])
def test_w4_packer_matches_oracle(qlin, N, K):
    W = synth.normal(7, synth.KEY_W, 0.02, (N, K))
    W[0, :128] = 0.0           # flat group
    W[1, :128] = np.abs(W[1, :128])  # one-signed group
    h = qlin.qlin_pack_w4g128(W)
    ex = qlin.qlin_export(h)
    ref = gptq_w4.pack(W)
    assert np.array_equal(ex["codes"], ref["codes"])
    assert np.array_equal(ex["scale"].view(np.uint16), ref["scale"].view(np.uint16))
    assert np.array_equal(ex["zero"].view(np.uint16), ref["zero"].view(np.uint16))
    inf = h.info
    assert inf.packed_bytes == gptq_w4.packed_bytes(N, K) and inf.bits_per_param == 4.25


@pytest.mark.parametrize("N,K,frac", [(64, 512, 0.01), (70, 768, 0.02), (33, 256, 0.005), (16, 512, 0.0)])
def test_spqr_packer_matches_oracle(qlin, N, K, frac):
    W = synth.student_t3(3, 0.02, (N, K))
    h = qlin.qlin_pack_spqr(W, frac)
    ex = qlin.qlin_export(h)
    ref = spqr.pack(W, frac)
    for key in ("codes", "qs_bits", "qz_bits", "rowptr", "col"):
        assert np.array_equal(ex[key], ref[key]), key
    assert np.array_equal(ex["stats"].view(np.uint16), ref["stats"].view(np.uint16))
    assert np.array_equal(ex["val"].view(np.uint16), ref["val"].view(np.uint16))
    inf = h.info
    assert inf.nnz == spqr.outlier_count(N, K, frac)
    assert inf.packed_bytes == spqr.packed_bytes(N, K, inf.nnz)


def test_spqr_packer_ties_and_all_outlier_group(qlin):
    W = np.full((2, 256), 0.001, dtype=np.float32)
    W[0, :16] = 10.0
    W[1, 5] = -10.0            # ties in magnitude with the first group
    W[1, 200] = 10.0
    frac = 17.5 / 512          # floor -> 17 outliers, two of the three tied last ones excluded
    h = qlin.qlin_pack_spqr(W, frac)
    ex = qlin.qlin_export(h)
    ref = spqr.pack(W, frac)
    assert np.array_equal(ex["col"], ref["col"]) and np.array_equal(ex["rowptr"], ref["rowptr"])
    assert np.array_equal(ex["stats"].view(np.uint16), ref["stats"].view(np.uint16))
    assert np.array_equal(ex["codes"], ref["codes"])


@pytest.mark.parametrize("N,K,alpha", [(64, 512, 0.85), (40, 256, 0.5), (64, 1024, 0.8)])
def test_w8_packer_matches_oracle(qlin, N, K, alpha):
    W, X, absmax, _ = synth.smoothquant_layer(N, K, 32, seed=4)
    h = qlin.qlin_pack_w8(W, absmax, alpha)
    ex = qlin.qlin_export(h)
    ref = smoothquant.quantize_weights(W, absmax, alpha)
    assert np.array_equal(ex["s"].view(np.uint32), ref["s"].view(np.uint32))
    assert np.array_equal(ex["s_inv"].view(np.uint32), ref["s_inv"].view(np.uint32))
    assert np.array_equal(ex["sw"].view(np.uint32), ref["sw"].view(np.uint32))
    assert np.array_equal(ex["qw"], ref["qw"])
    assert h.info.packed_bytes == smoothquant.packed_bytes(N, K)


def test_packers_reject_bad_input(qlin):
    W = np.zeros((8, 256), dtype=np.float32)
    with pytest.raises(qlin.QlinError) as e:
        qlin.qlin_pack_w4g128(np.zeros((8, 100), dtype=np.float32))
    assert e.value.status == qlin.QLIN_ERR_INVALID_ARG
    bad = W.copy()
    bad[3, 7] = np.nan
    for fn in (lambda: qlin.qlin_pack_w4g128(bad), lambda: qlin.qlin_pack_spqr(bad, 0.01),
               lambda: qlin.qlin_pack_w8(bad, np.ones(256, np.float32), 0.85)):
        with pytest.raises(qlin.QlinError):
            fn()
    with pytest.raises(qlin.QlinError):
        qlin.qlin_pack_spqr(np.zeros((8, 200), dtype=np.float32), 0.01)   # K % 256
    with pytest.raises(qlin.QlinError):
        qlin.qlin_pack_spqr(np.zeros((2, 32768 + 256), dtype=np.float32), 0.01)   # int16 columns
    with pytest.raises(qlin.QlinError):
        qlin.qlin_pack_spqr(W, 1.5)
    with pytest.raises(qlin.QlinError):
        qlin.qlin_pack_w8(W, np.ones(256, np.float32), 1.5)
    with pytest.raises(qlin.QlinError):
        big = W.copy()
        big[0, 0], big[0, 1] = -1e6, 1e6      # scale overflows fp16
        qlin.qlin_pack_w4g128(big)


def test_device_image_and_workspace_sizes(qlin):
    W = synth.normal(0, synth.KEY_W, 0.02, (100, 512))
    h = qlin.qlin_pack_w4g128(W)
    nb = qlin.qlin_device_bytes(h)
    assert nb >= 2 * 4 * 4352 and nb % 256 == 0      # 2 row groups x 4 K groups of units
    assert qlin.qlin_workspace_bytes(h, 16) > 0
    h8 = qlin.qlin_pack_w8(W, np.ones(512, np.float32), 0.85)
    assert qlin.qlin_workspace_bytes(h8, 64) > qlin.qlin_workspace_bytes(h8, 1)
