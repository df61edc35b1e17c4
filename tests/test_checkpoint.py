"""Checkpoint load: a handle rebuilt from canonical arrays (qlin_import, QLinear.save/load).

The arrays are the layouts qlin_export documents; loading must give back the same arrays
bit for bit and the same sizes, without quantizing anything, and must refuse arrays no
packer could have written.  (That the rebuilt device image computes the same outputs is
checked on the GPU in test_gpu_decode.py.)
"""
import numpy as np
import pytest

import qlin_synth as synth


def _layers(qlin):
    W = synth.student_t3(3, 0.02, (70, 768))
    Wg = synth.normal(5, synth.KEY_W, 0.02, (40, 256))
    absmax = np.abs(synth.bf16_to_f32(synth.activations_bf16(1, 8, 768))).max(axis=0)
    return {
        "w4": lambda: qlin.QLinear.from_w4g128(W),
        "w4_gptq": lambda: qlin.QLinear.from_w4g128_gptq(Wg, synth.gptq_calibration(64, 256, seed=5)),
        "w4_act": lambda: qlin.QLinear.from_w4g128_gptq(Wg, synth.gptq_calibration(64, 256, seed=5), act_order=True),
        "spqr_0": lambda: qlin.QLinear.from_spqr(W, 0.0),
        "spqr_1": lambda: qlin.QLinear.from_spqr(W, 0.01),
        "spqr_2": lambda: qlin.QLinear.from_spqr(W, 0.02),
        "w8a8": lambda: qlin.QLinear.from_w8(W, absmax, 0.85),
    }


@pytest.mark.parametrize("kind", ["w4", "w4_gptq", "w4_act", "spqr_0", "spqr_1", "spqr_2", "w8a8"])
def test_round_trip(qlin, kind, tmp_path):
    L = _layers(qlin)[kind]()
    ex = L.export()
    path = tmp_path / "layer.npz"
    L.save(path)
    L2 = qlin.QLinear.load(path)
    ex2 = L2.export()
    assert ex.keys() == ex2.keys()
    for k in ex:
        assert np.array_equal(np.asarray(ex[k]).view(np.uint8), np.asarray(ex2[k]).view(np.uint8)), k
    a, b = L.handle.info, L2.handle.info
    assert (a.format, a.N, a.K, a.nnz, a.packed_bytes, a.device_bytes) == \
           (b.format, b.N, b.K, b.nnz, b.packed_bytes, b.device_bytes)


def _reject(qlin, fmt, N, K, arrays):
    with pytest.raises(qlin.QlinError):
        qlin.qlin_import(fmt, N, K, arrays)


def test_rejects_w4_arrays_no_packer_writes(qlin):
    L = _layers(qlin)["w4"]()
    ex, N, K = L.export(), L.N, L.K
    for field, value in (("zero", 16.0), ("zero", 2.5), ("scale", 0.0), ("scale", -0.5), ("scale", np.inf)):
        bad = {k: v.copy() for k, v in ex.items()}
        bad[field][3, 1] = value
        _reject(qlin, qlin.FMT_W4G128, N, K, bad)
    _reject(qlin, qlin.FMT_W4G128, N, 200, ex)  # K % 128
    act = _layers(qlin)["w4_act"]()
    ea = act.export()
    bad = {k: v.copy() for k, v in ea.items()}
    bad["perm"][1] = bad["perm"][0]  # not a permutation
    _reject(qlin, qlin.FMT_W4G128, act.N, act.K, bad)


def test_rejects_spqr_arrays_no_packer_writes(qlin):
    L = _layers(qlin)["spqr_1"]()
    ex, N, K = L.export(), L.N, L.K
    r = ex["rowptr"]
    row = int(np.argmax(np.diff(r) >= 2))  # a row with two outliers or more
    p = int(r[row])
    cases = []
    b = {k: v.copy() for k, v in ex.items()}; b["rowptr"][row + 1] = b["rowptr"][row] - 1; cases.append(b)
    b = {k: v.copy() for k, v in ex.items()}; b["col"][p] = K; cases.append(b)
    b = {k: v.copy() for k, v in ex.items()}; b["col"][p + 1] = b["col"][p]; cases.append(b)
    b = {k: v.copy() for k, v in ex.items()}; b["val"][p] = np.inf; cases.append(b)
    b = {k: v.copy() for k, v in ex.items()}; b["stats"][0, 0, 1] = 0.5; cases.append(b)  # zs not an integer
    b = {k: v.copy() for k, v in ex.items()}; b["stats"][0, 0, 3] = 8.0; cases.append(b)  # zz > 7
    b = {k: v.copy() for k, v in ex.items()}; b["rowptr"][0] = 1; cases.append(b)
    for bad in cases:
        _reject(qlin, qlin.FMT_SPQR, N, K, bad)


def test_rejects_w8_arrays_no_packer_writes(qlin):
    L = _layers(qlin)["w8a8"]()
    ex, N, K = L.export(), L.N, L.K
    for field, idx, value in (("qw", (0, 0), -128), ("sw", 2, 0.0), ("s", 5, np.nan), ("s_inv", 1, -1.0)):
        bad = {k: v.copy() for k, v in ex.items()}
        bad[field][idx] = value
        _reject(qlin, qlin.FMT_W8A8, N, K, bad)


def test_unknown_format(qlin):
    with pytest.raises(ValueError):
        qlin.qlin_import(9, 4, 128, {})
