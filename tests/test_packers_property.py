"""Property tests of the host packers against the oracle on random shapes (CPU only).

Ragged row counts, the smallest and a few larger K for each format, empty and crowded outlier
sets, and weights scaled over several octaves: every canonical array must match the oracle
bit for bit, and export -> import must give the same arrays back.
"""
import numpy as np
import pytest

import qlin_synth as synth
from oracle import gptq_w4, smoothquant, spqr

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

_SETTINGS = dict(max_examples=12, deadline=None, derandomize=True)


def _same(a, b):
    return np.array_equal(np.asarray(a).view(np.uint8), np.asarray(b).view(np.uint8))


@settings(**_SETTINGS)
@given(N=st.integers(1, 90), kg=st.integers(1, 4), seed=st.integers(0, 1000), octave=st.integers(-6, 6))
def test_w4_packer_random(qlin, N, kg, seed, octave):
    W = synth.normal(seed, synth.KEY_W, 0.02 * 2.0 ** octave, (N, 128 * kg))
    ex = qlin.qlin_export(qlin.qlin_pack_w4g128(W))
    ref = gptq_w4.pack(W)
    for k in ("codes", "scale", "zero"):
        assert _same(ex[k], ref[k]), k
    h2 = qlin.qlin_import(qlin.FMT_W4G128, N, 128 * kg, ex)
    assert all(_same(qlin.qlin_export(h2)[k], ex[k]) for k in ex)


@settings(**_SETTINGS)
@given(N=st.integers(1, 80), ks=st.integers(1, 3), seed=st.integers(0, 1000),
       frac=st.sampled_from([0.0, 0.001, 0.01, 0.03]), octave=st.integers(-4, 4))
def test_spqr_packer_random(qlin, N, ks, seed, frac, octave):
    K = 256 * ks
    W = synth.student_t3(seed, 0.02 * 2.0 ** octave, (N, K))
    h = qlin.qlin_pack_spqr(W, frac)
    ex = qlin.qlin_export(h)
    ref = spqr.pack(W, frac)
    for key in ("codes", "qs_bits", "qz_bits", "rowptr", "col"):
        assert np.array_equal(ex[key], ref[key]), key
    assert _same(ex["stats"], ref["stats"]) and _same(ex["val"], ref["val"])
    h2 = qlin.qlin_import(qlin.FMT_SPQR, N, K, ex)
    assert all(_same(qlin.qlin_export(h2)[k], ex[k]) for k in ex)
    assert h2.info.device_bytes == h.info.device_bytes


@settings(**_SETTINGS)
@given(N=st.integers(1, 70), kb=st.integers(1, 4), seed=st.integers(0, 1000),
       alpha=st.sampled_from([0.0, 0.5, 0.85, 1.0]))
def test_w8_packer_random(qlin, N, kb, seed, alpha):
    K = 64 * kb
    W = synth.normal(seed, synth.KEY_W, 0.02, (N, K))
    ch = synth.pick_channels(seed, K, max(1, K // 100))
    absmax = synth.channel_absmax(synth.activations_bf16(seed, 8, K, boosted=ch))
    ex = qlin.qlin_export(qlin.qlin_pack_w8(W, absmax, alpha))
    ref = smoothquant.quantize_weights(W, absmax, alpha)
    assert np.array_equal(ex["qw"], ref["qw"])
    for k in ("sw", "s", "s_inv"):
        assert _same(ex[k], ref[k]), k
    h2 = qlin.qlin_import(qlin.FMT_W8A8, N, K, ex)
    assert all(_same(qlin.qlin_export(h2)[k], ex[k]) for k in ex)
