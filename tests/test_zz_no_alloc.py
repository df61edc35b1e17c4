"""The allocation-free SpQR decode entry point against the regular forward (GPU).

qlin_forward_spqr_static serves callers that may not allocate device memory (a layer inside
an engine that has reserved the device's memory for its own pools, a service that forbids
allocation while serving): it runs the same kernels as qlin_forward but takes its scratch
from a fixed array inside the library.  The kernels are deterministic, so its outputs must
equal qlin_forward's bit for bit, on two calls in a row (the array keeps the previous call's
contents, so the second call checks that stale counters or tagged words never leak into a
result), and qlin_poll_static_status must report no device-side timeout.  The file is named
to be collected last and must pass alone in a fresh process as well as after the other tests.
"""
import numpy as np
import pytest

import qlin_synth as synth
from oracle import forward, spqr
from oracle.fp import bits_to_f32

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


# M = 1: the single-token kernel; M = 3: tagged words of up to four tokens; M = 5, 16: counted
@pytest.mark.parametrize("N,K,M", [(1000, 2048, 1), (11008, 4096, 1), (1000, 2048, 3), (11008, 4096, 3),
                                   (1000, 2048, 5), (256, 512, 16)])
def test_static_scratch_forward_matches_regular_forward(qlin, N, K, M):
    W, X = synth.spqr_layer(N, K, M, seed=7)
    layer = qlin.QLinear.from_spqr(W, 0.01).to("cuda")
    Xd = torch.from_numpy(X).cuda().view(torch.bfloat16)
    y_gpu = _bits(layer(Xd))
    assert layer.poll_status() == qlin.QLIN_OK
    # the regular path itself is within the parity tolerance of the oracle
    y_ref, bound = forward.reference(bits_to_f32(X), spqr.pack(W, 0.01)["w_hat"])
    ok, worst = forward.within_tolerance(bits_to_f32(y_gpu), y_ref, bound)
    assert ok, worst
    for call in range(2):
        Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        qlin.qlin_forward_spqr_static(layer.handle, Xd, Y, M)
        assert qlin.qlin_poll_static_status() == qlin.QLIN_OK, call
        assert np.array_equal(_bits(Y), y_gpu), call


def test_static_scratch_rejects_what_it_cannot_serve(qlin):
    W, X = synth.spqr_layer(128, 512, 1, seed=1)
    layer = qlin.QLinear.from_spqr(W, 0.01).to("cuda")
    Xd = torch.from_numpy(X).cuda().view(torch.bfloat16)
    Y = torch.empty((1, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(qlin.QlinError) as e:
        qlin.qlin_forward_spqr_static(layer.handle, torch.zeros((17, 512), dtype=torch.bfloat16, device="cuda"),
                                      torch.empty((17, 128), dtype=torch.bfloat16, device="cuda"), 17)
    assert e.value.status == qlin.QLIN_ERR_INVALID_ARG
    w4 = qlin.QLinear.from_w4g128(synth.normal(0, synth.KEY_W, 0.02, (128, 512))).to("cuda")
    with pytest.raises(qlin.QlinError):
        qlin.qlin_forward_spqr_static(w4.handle, Xd, Y, 1)
    unbound = qlin.QLinear.from_spqr(W, 0.01)
    with pytest.raises(qlin.QlinError) as e:
        qlin.qlin_forward_spqr_static(unbound.handle, Xd, Y, 1)
    assert e.value.status == qlin.QLIN_ERR_NOT_BOUND


def _zero_spqr_layer(qlin, N, K):
    """An all-zero SpQR layer of the given shape, loaded from canonical arrays (no packing)."""
    arrays = {"codes": np.zeros((N, 3 * K // 8), np.uint8), "qs_bits": np.zeros((N, 3 * (K // 16) // 8), np.uint8),
              "qz_bits": np.zeros((N, 3 * (K // 16) // 8), np.uint8),
              "stats": np.zeros((N, K // 256, 4), np.float16), "rowptr": np.zeros(N + 1, np.int32),
              "col": np.zeros(0, np.int16), "val": np.zeros(0, np.float16)}
    return qlin.QLinear(qlin.qlin_import(qlin.FMT_SPQR, N, K, arrays))


# past the array's limits: 8193 row groups of 64 rows; 1278 row groups x 128 supergroups
# = 163,584 units of 64 x 256 (the stated limit is 162,560; one token alone fits up to 163,520)
@pytest.mark.parametrize("N,K", [(8193 * 64, 256), (1278 * 64, 32768)])
def test_static_scratch_rejects_layers_beyond_its_limits(qlin, N, K):
    layer = _zero_spqr_layer(qlin, N, K).to("cuda", max_M=2)
    for M in (1, 2):
        X = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
        Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        with pytest.raises(qlin.QlinError) as e:
            qlin.qlin_forward_spqr_static(layer.handle, X, Y, M)
        assert e.value.status == qlin.QLIN_ERR_WORKSPACE, M
    assert qlin.qlin_poll_static_status() == qlin.QLIN_OK
