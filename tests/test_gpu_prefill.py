"""GPU parity of the tensor-core prefill path (M > 16) against the oracle, through the C ABI.

W4 / SpQR: bf16 outputs within 1e-2 * sum |x w| + 1 ulp of the fp64 oracle.
W8A8: int32 accumulators and bf16 outputs bit-exact (the fp16 MMA is exact on int8 codes,
and K is cut into chunks whose sums stay below 2^24, drained into int32).
"""
import numpy as np
import pytest

import qlin_synth as synth
from oracle import forward, gptq_w4, smoothquant, spqr
from oracle.fp import bits_to_f32

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


def _y(layer, X):
    Y = layer(torch.from_numpy(np.ascontiguousarray(X)).cuda().view(torch.bfloat16))
    torch.cuda.synchronize()
    assert layer.poll_status() == 0
    return bits_to_f32(Y.view(torch.int16).cpu().numpy().view(np.uint16))


@pytest.mark.parametrize("N,K,M", [(128, 512, 17), (256, 1024, 128), (384, 512, 200), (192, 1024, 129)])
def test_w4_prefill_tolerance(qlin, N, K, M):
    W, X = synth.gptq_layer(N, K, M, seed=M)
    layer = qlin.QLinear.from_w4g128(W).to("cuda")
    y = _y(layer, X)
    ok, worst = forward.within_tolerance(y, *forward.reference(bits_to_f32(X), gptq_w4.pack(W)["w_hat"]))
    assert ok, worst


# M = 300, 1024: an even number of 256-token tiles, so CTA pairs share the weight tiles (N = 320:
# a last weight tile of one 64-row group)
@pytest.mark.parametrize("N,K,M,frac", [(128, 512, 17, 0.01), (256, 1024, 160, 0.02), (192, 768, 64, 0.01),
                                        (256, 1024, 300, 0.01), (320, 512, 1024, 0.02)])
def test_spqr_prefill_tolerance(qlin, N, K, M, frac):
    W, X = synth.spqr_layer(N, K, M, seed=M)
    layer = qlin.QLinear.from_spqr(W, frac).to("cuda")
    y = _y(layer, X)
    ok, worst = forward.within_tolerance(y, *forward.reference(bits_to_f32(X), spqr.pack(W, frac)["w_hat"]))
    assert ok, worst


@pytest.mark.parametrize("N,K,M", [(128, 512, 17), (256, 2048, 130), (192, 3072, 64)])
def test_w8a8_prefill_bit_exact(qlin, N, K, M):
    W, X, absmax, _ = synth.smoothquant_layer(N, K, M, seed=M)
    layer = qlin.QLinear.from_w8(W, absmax, 0.85).to("cuda", max_M=M)
    pk = smoothquant.quantize_weights(W, absmax, 0.85)
    y_ref, acc_ref, _, _ = smoothquant.forward(bits_to_f32(X), pk)
    acc = layer.forward_acc(torch.from_numpy(X).cuda().view(torch.bfloat16)).cpu().numpy()
    assert np.array_equal(acc.astype(np.int64), acc_ref)
    y = _y(layer, X)
    assert np.array_equal(y.view(np.uint32), y_ref.view(np.uint32))


@pytest.mark.parametrize("K,M,sign", [(3072, 40, 1.0), (2048, 300, -1.0)])
def test_w8a8_prefill_exact_at_largest_codes(qlin, K, M, sign):
    """Every activation and weight code at +-127, so each 1024-wide chunk sums to 127^2 * 1024
    (just under 2^24) and the whole row far above it: the chunking and the int32 drain must
    still give the exact accumulator.  A few tokens of small codes ride along in the tile, and
    M = 300 leaves a partial 256-token tile."""
    N = 128
    W = np.full((N, K), 0.02, dtype=np.float32)
    W[1::2] *= sign
    x = np.ones((M, K), dtype=np.float32)
    x[::7] = 0.01 * synth.normal(5, synth.KEY_X, 1.0, (len(range(0, M, 7)), K))
    X = synth.f32_to_bf16(x)
    absmax = synth.channel_absmax(X)
    layer = qlin.QLinear.from_w8(W, absmax, 0.85).to("cuda", max_M=M)
    pk = smoothquant.quantize_weights(W, absmax, 0.85)
    y_ref, acc_ref, _, _ = smoothquant.forward(bits_to_f32(X), pk)
    assert np.abs(acc_ref).max() > 2 ** 24  # the exactness limit of one fp32 accumulation
    acc = layer.forward_acc(torch.from_numpy(X).cuda().view(torch.bfloat16)).cpu().numpy()
    assert np.array_equal(acc.astype(np.int64), acc_ref)
    y = _y(layer, X)
    assert np.array_equal(y.view(np.uint32), y_ref.view(np.uint32))
