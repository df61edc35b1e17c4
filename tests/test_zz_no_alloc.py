"""The allocation-free SpQR decode entry point against the regular forward (GPU).

qlin_forward_spqr_static serves callers that may not allocate device memory: it runs the
same decode kernel as qlin_forward but takes its scratch from a fixed array inside the
library.  Its output must match qlin_forward's within the parity tolerance of the other
tests, on two calls in a row (the array keeps the previous call's contents, so the second
call checks that stale counters and slots do not leak into a result).  The file is named to
be collected last and must pass alone in a fresh process as well as after the other tests.
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


def _f32(t):
    return bits_to_f32(t.view(torch.int16).cpu().numpy().view(np.uint16))


@pytest.mark.parametrize("N,K,M", [(1000, 2048, 1), (11008, 4096, 1), (1000, 2048, 5), (256, 512, 16)])
def test_static_scratch_forward_matches_regular_forward(qlin, N, K, M):
    W, X = synth.spqr_layer(N, K, M, seed=7)
    layer = qlin.QLinear.from_spqr(W, 0.01).to("cuda")
    Xd = torch.from_numpy(X).cuda().view(torch.bfloat16)
    y_ref_gpu = _f32(layer(Xd))
    x = bits_to_f32(X)
    y_ref, bound = forward.reference(x, spqr.pack(W, 0.01)["w_hat"])
    for call in range(2):
        Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        qlin.qlin_forward_spqr_static(layer.handle, Xd, Y, M)
        torch.cuda.synchronize()
        y = _f32(Y)
        # same kernel: within the tolerance of the regular path, and of the oracle
        ok, worst = forward.within_tolerance(y, y_ref_gpu.astype(np.float64), bound)
        assert ok, (call, worst)
        ok, worst = forward.within_tolerance(y, y_ref, bound)
        assert ok, (call, worst)


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
