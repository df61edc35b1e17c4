"""GPU parity at the workloads' full sizes (configurations of the GPTQ, SpQR and SmoothQuant
layers), in the launch configuration the benchmark times.  Where the fp64 oracle cannot cover
the whole output in seconds, a seeded sample of output rows and tokens is checked.
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


def _run(layer, X):
    Y = layer(torch.from_numpy(np.ascontiguousarray(X)).cuda().view(torch.bfloat16))
    torch.cuda.synchronize()
    assert layer.poll_status() == 0
    return Y


def _rows(Y, rows_m, rows_n):
    y = Y.view(torch.int16)[torch.as_tensor(rows_m, device="cuda")][:, torch.as_tensor(rows_n, device="cuda")]
    return bits_to_f32(y.cpu().numpy().view(np.uint16))


def _tile_sample(n, tile, seed):
    """One index in every tile of `tile` consecutive indices, at an offset that moves from tile
    to tile (so every tile of the kernel's grid, and every position class inside a tile, is
    reached), plus the first and the last index."""
    rng = np.random.default_rng(seed)
    starts = np.arange(0, n, tile)
    offs = (rng.integers(0, tile, size=len(starts)) + 37 * np.arange(len(starts))) % tile
    s = np.minimum(starts + offs, n - 1)
    return np.unique(np.concatenate([s, [0, n - 1]]))


def _sample(n, count, seed):
    rng = np.random.default_rng(seed)
    s = np.sort(rng.choice(n, size=min(count, n), replace=False))
    s[0], s[-1] = 0, n - 1
    return np.unique(s)


# ---------------------------------------------------------------- configs 0 and 1 (full oracle)

def test_gptq_w4g128_4096x4096_m1(qlin):
    W, X = synth.gptq_layer(4096, 4096, 16, seed=0)
    layer = qlin.QLinear.from_w4g128(W).to("cuda")
    assert layer.handle.info.packed_bytes == 8912896
    w_hat = gptq_w4.pack(W)["w_hat"]
    for M in (1, 16):
        y = bits_to_f32(_run(layer, X[:M]).view(torch.int16).cpu().numpy().view(np.uint16))
        ok, worst = forward.within_tolerance(y, *forward.reference(bits_to_f32(X[:M]), w_hat))
        assert ok, (M, worst)


def test_spqr_11008x4096_m1_1pct(qlin):
    W, X = synth.spqr_layer(11008, 4096, 1, seed=0)
    layer = qlin.QLinear.from_spqr(W, 0.01).to("cuda")
    inf = layer.handle.info
    assert inf.nnz == 450887 and inf.packed_bytes == 22278432
    assert 3.36 <= inf.bits_per_param <= 4.75
    y = bits_to_f32(_run(layer, X).view(torch.int16).cpu().numpy().view(np.uint16))
    ok, worst = forward.within_tolerance(y, *forward.reference(bits_to_f32(X), spqr.pack(W, 0.01)["w_hat"]))
    assert ok, worst


def test_smoothquant_w8a8_4096x4096(qlin):
    W, X, absmax, _ = synth.smoothquant_layer(4096, 4096, 2048, seed=0)
    layer = qlin.QLinear.from_w8(W, absmax, 0.85).to("cuda", max_M=2048)
    pk = smoothquant.quantize_weights(W, absmax, 0.85)
    x = bits_to_f32(X)
    # decode, M = 16: whole output, bit-exact
    y = bits_to_f32(_run(layer, X[:16]).view(torch.int16).cpu().numpy().view(np.uint16))
    y_ref = smoothquant.forward(x[:16], pk)[0]
    assert np.array_equal(y.view(np.uint32), y_ref.view(np.uint32))
    # prefill, M = 2048: sampled tokens, all rows, accumulators and outputs bit-exact
    Y = _run(layer, X)
    acc = layer.forward_acc(torch.from_numpy(X).cuda().view(torch.bfloat16))
    ms = _sample(2048, 48, 1)
    qx, sx = smoothquant.quantize_activations(x, pk["s_inv"])
    acc_ref = smoothquant.accumulate(qx[ms], pk["qw"])
    assert np.array_equal(acc[torch.as_tensor(ms, device="cuda")].cpu().numpy().astype(np.int64), acc_ref)
    y_ref = smoothquant.epilogue(acc_ref, sx[ms], pk["sw"])
    assert np.array_equal(_rows(Y, ms, np.arange(4096)).view(np.uint32), y_ref.view(np.uint32))


# ---------------------------------------------------------------- config 3: decode sweep (sampled rows)

SHAPES = [(8192, 8192), (8192, 28672), (28672, 8192)]  # (K, N)


@pytest.mark.parametrize("K,N", SHAPES)
def test_decode_sweep_w4(qlin, K, N):
    W, X = synth.gptq_layer(N, K, 16, seed=0)
    layer = qlin.QLinear.from_w4g128(W).to("cuda")
    ns = _sample(N, 192, 2)
    w_hat = gptq_w4.pack(W[ns])["w_hat"]
    for M in (1, 4, 16):
        Y = _run(layer, X[:M])
        ok, worst = forward.within_tolerance(_rows(Y, np.arange(M), ns), *forward.reference(bits_to_f32(X[:M]), w_hat))
        assert ok, (M, worst)


def test_decode_w8a8_8192x8192_sampled(qlin):
    """A 67 MB W8A8 layer at 1, 4 and 16 tokens (up to eight tokens layers of 24 MB and more run
    four CTAs per SM, smaller ones three): sampled rows, outputs bit-exact."""
    N = K = 8192
    W, X, absmax, _ = synth.smoothquant_layer(N, K, 16, seed=2)
    layer = qlin.QLinear.from_w8(W, absmax, 0.85).to("cuda")
    ns = _sample(N, 160, 4)
    s, s_inv = smoothquant.smoothing_factors(absmax, W, 0.85)
    qw, sw = smoothquant.quantize_rows_int8(smoothquant.fold_weights(W[ns], s))
    for M in (1, 4, 16):
        Y = _run(layer, X[:M])
        qx, sx = smoothquant.quantize_activations(bits_to_f32(X[:M]), s_inv)
        y_ref = smoothquant.epilogue(smoothquant.accumulate(qx, qw), sx, sw)
        assert np.array_equal(_rows(Y, np.arange(M), ns).view(np.uint32), y_ref.view(np.uint32)), M


@pytest.mark.parametrize("K,N", SHAPES)
@pytest.mark.parametrize("frac", [0.005, 0.01, 0.02])
def test_decode_sweep_spqr(qlin, K, N, frac):
    W, X = synth.spqr_layer(N, K, 16, seed=0)
    layer = qlin.QLinear.from_spqr(W, frac).to("cuda")
    assert 3.36 <= layer.handle.info.bits_per_param <= 4.75
    ns = _sample(N, 128, 3)
    w_hat = spqr.dequantize(spqr.quantize_rows(W, frac, ns))
    for M in (1, 4, 16):
        Y = _run(layer, X[:M])
        ok, worst = forward.within_tolerance(_rows(Y, np.arange(M), ns), *forward.reference(bits_to_f32(X[:M]), w_hat))
        assert ok, (M, worst)


# ---------------------------------------------------------------- config 4: prefill M = 4096 (sampled)

@pytest.mark.parametrize("K,N", [(8192, 28672), (28672, 8192)])
@pytest.mark.parametrize("fmt", ["w4", "spqr", "w8a8"])
def test_prefill_4096(qlin, K, N, fmt):
    """Every 128-row weight tile and every 256-token tile of the M = 4096 grid is sampled at
    least once (one row / token per tile at a moving offset, plus extra tokens)."""
    M = 4096
    ms = np.union1d(_tile_sample(M, 256, 4), _sample(M, 12, 6))
    ns = _tile_sample(N, 128, 5)
    if fmt == "w8a8":
        W, X, absmax, _ = synth.smoothquant_layer(N, K, M, seed=0)
        layer = qlin.QLinear.from_w8(W, absmax, 0.85).to("cuda", max_M=M)
        Y = _run(layer, X)
        s, s_inv = smoothquant.smoothing_factors(absmax, W, 0.85)
        qw, sw = smoothquant.quantize_rows_int8(smoothquant.fold_weights(W[ns], s))
        qx, sx = smoothquant.quantize_activations(bits_to_f32(X[ms]), s_inv)
        y_ref = smoothquant.epilogue(smoothquant.accumulate(qx, qw), sx, sw)
        assert np.array_equal(_rows(Y, ms, ns).view(np.uint32), y_ref.view(np.uint32))
        return
    if fmt == "w4":
        W, X = synth.gptq_layer(N, K, M, seed=0)
        layer = qlin.QLinear.from_w4g128(W).to("cuda")
        w_hat = gptq_w4.pack(W[ns])["w_hat"]
    else:
        W, X = synth.spqr_layer(N, K, M, seed=0)
        layer = qlin.QLinear.from_spqr(W, 0.01).to("cuda")
        w_hat = spqr.dequantize(spqr.quantize_rows(W, 0.01, ns))
    Y = _run(layer, X)
    ok, worst = forward.within_tolerance(_rows(Y, ms, ns), *forward.reference(bits_to_f32(X[ms]), w_hat))
    assert ok, worst
