"""GPU parity of the decode (M <= 16) path against the oracle, through the C ABI.

Bars (stated target): dequantized weights, int8 codes and int32 accumulators bit-exact;
bf16 outputs within 1e-2 * sum_k |x_k w_k| + 1 bf16 ulp of the fp64 oracle.
"""
import numpy as np
import pytest

import qlin_synth as synth
from oracle import forward, gptq_w4, smoothquant, spqr
from oracle.fp import bits_to_f32, bf16_round

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _y(layer, X, M):
    Xd = _dev(X).view(torch.bfloat16)
    Y = layer(Xd)
    torch.cuda.synchronize()
    assert layer.poll_status() == 0
    return bits_to_f32(Y.view(torch.int16).cpu().numpy().view(np.uint16))


def _check(y, x_bits, w_hat):
    y_ref, bound = forward.reference(bits_to_f32(x_bits), w_hat)
    ok, worst = forward.within_tolerance(y, y_ref, bound)
    assert ok, f"worst |err|/tol = {worst}"
    return worst


# ----------------------------------------------------------------------------- W4 g128

@pytest.mark.parametrize("N,K", [(256, 1024), (100, 512), (64, 128)])
def test_w4_device_dequant_bit_exact(qlin, N, K):
    W = synth.normal(11, synth.KEY_W, 0.02, (N, K))
    layer = qlin.QLinear.from_w4g128(W).to("cuda")
    wd = layer.dequant_device().cpu().numpy()
    ref = gptq_w4.pack(W)["w_hat"]
    assert np.array_equal(wd.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("N,K", [(256, 1024), (100, 512), (1000, 2048)])
@pytest.mark.parametrize("M", [1, 3, 8, 9, 16])
def test_w4_forward_tolerance(qlin, N, K, M):
    W, X = synth.gptq_layer(N, K, M, seed=M)
    layer = qlin.QLinear.from_w4g128(W).to("cuda")
    _check(_y(layer, X, M), X, gptq_w4.pack(W)["w_hat"])


def test_w4_one_hot_rows_bit_exact(qlin):
    N, K = 192, 512
    W = synth.normal(5, synth.KEY_W, 0.02, (N, K))
    layer = qlin.QLinear.from_w4g128(W).to("cuda")
    w_hat = gptq_w4.pack(W)["w_hat"]
    ks = [0, 1, 7, 8, 9, 127, 128, 300, 511]
    X = np.zeros((len(ks), K), dtype=np.float32)
    for i, k in enumerate(ks):
        X[i, k] = 1.0
    y = _y(layer, synth.f32_to_bf16(X), len(ks))
    for i, k in enumerate(ks):
        assert np.array_equal(y[i], bf16_round(w_hat[:, k]))


@pytest.mark.parametrize("act", [False, True])
@pytest.mark.parametrize("M", [1, 16, 40])
def test_w4_gptq_layer(qlin, M, act):
    """GPTQ-packed codes (error-compensated, same W4 g128 format): the same kernels read
    them; dequantized weights bit-exact, outputs within tolerance (M = 40: prefill).  With
    act-order the codes are in the permuted column order and the forward gathers X[:, perm]
    first."""
    from oracle import gptq
    N, K = 192, 1024
    W = synth.normal(21, synth.KEY_W, 0.02, (N, K))
    Xcal = synth.gptq_calibration(256, K, seed=21)
    Xcal = (Xcal * (2.0 ** (np.arange(K) % 5 - 2))[None, :]).astype(np.float32)
    layer = qlin.QLinear.from_w4g128_gptq(W, Xcal, act_order=act).to("cuda", max_M=40)
    ref = gptq.pack(W, Xcal, act=act)
    wd = layer.dequant_device().cpu().numpy()
    assert np.array_equal(wd.view(np.uint32), ref["w_hat_perm" if act else "w_hat"].view(np.uint32))
    X = synth.activations_bf16(21, M, K)
    _check(_y(layer, X, M), X, ref["w_hat"])


# K = 8192: the largest K whose single-token forward gathers x inside the kernel; 8320: past
# it (a gather launch first); 1152: nine K groups, so the CTAs' staged ranges wrap around K
@pytest.mark.parametrize("N,K", [(2048, 8192), (1000, 8320), (4096, 1152)])
def test_w4_act_order_single_token(qlin, N, K):
    """One token through an act-order layer (codes in permuted column order, imported with a
    permutation) equals, bit for bit, the same codes without the permutation fed x[perm] (the
    staged activations are the same values), and the oracle within the tolerance."""
    W = synth.normal(23, synth.KEY_W, 0.02, (N, K))
    c = qlin.QLinear.from_w4g128(W).export()
    perm = np.random.default_rng(23).permutation(K).astype(np.int32)
    plain = qlin.QLinear(qlin.qlin_import(qlin.FMT_W4G128, N, K, c)).to("cuda")
    act = qlin.QLinear(qlin.qlin_import(qlin.FMT_W4G128, N, K, dict(c, perm=perm))).to("cuda")
    X = synth.activations_bf16(23, 1, K)
    y_act = _y(act, X, 1)
    assert np.array_equal(y_act.view(np.uint32), _y(plain, np.ascontiguousarray(X[:, perm]), 1).view(np.uint32))
    w_hat = gptq_w4.dequantize(gptq_w4.unpack_codes(c["codes"]), c["scale"], c["zero"])
    y_ref, bound = forward.reference(bits_to_f32(X)[:, perm], w_hat)
    ok, worst = forward.within_tolerance(y_act, y_ref, bound)
    assert ok, worst


@pytest.mark.parametrize("kind", ["w4", "w4_act", "spqr", "w8a8"])
def test_checkpoint_reload_computes_the_same(qlin, kind, tmp_path):
    """A layer saved and loaded back (qlin_import, no requantization) gives the same outputs
    bit for bit as the layer that was saved, decode and prefill, and matches the oracle run on
    the loaded canonical arrays (W8A8 bit for bit, the others within the tolerance)."""
    N, K = 160, 1024
    if kind == "w4":
        W, X = synth.gptq_layer(N, K, 40, seed=41)
        L = qlin.QLinear.from_w4g128(W)
    elif kind == "w4_act":
        W, X = synth.gptq_layer(N, K, 40, seed=41)
        Xcal = synth.gptq_calibration(128, K, seed=41)
        L = qlin.QLinear.from_w4g128_gptq(W, (Xcal * (2.0 ** (np.arange(K) % 5 - 2))[None, :]).astype(np.float32),
                                          act_order=True)
    elif kind == "spqr":
        W, X = synth.spqr_layer(N, K, 40, seed=41)
        L = qlin.QLinear.from_spqr(W, 0.02)
    else:
        W, X, absmax, _ = synth.smoothquant_layer(N, K, 40, seed=41)
        L = qlin.QLinear.from_w8(W, absmax, 0.85)
    L.save(tmp_path / "layer.npz")
    L2 = qlin.QLinear.load(tmp_path / "layer.npz")
    a, b = L.to("cuda", max_M=40), L2.to("cuda", max_M=40)
    # the oracle on the loaded canonical arrays alone (no packer involved)
    c = L2.export()
    x = bits_to_f32(X)
    if kind == "w8a8":
        qx, sx = smoothquant.quantize_activations(x, c["s_inv"])
        y_ora = smoothquant.epilogue(smoothquant.accumulate(qx, c["qw"]), sx, c["sw"])
    elif kind == "spqr":
        w_hat = spqr.dequantize_canonical(N, K, c["codes"], c["qs_bits"], c["qz_bits"], c["stats"], c["rowptr"],
                                          c["col"], c["val"])
    else:
        w_hat = gptq_w4.dequantize(gptq_w4.unpack_codes(c["codes"]), c["scale"], c["zero"])
        if kind == "w4_act":  # codes of W[:, perm]: the forward multiplies by X[:, perm]
            x = x[:, c["perm"]]
    for M in (1, 40):
        yb = _y(b, X[:M], M)
        assert np.array_equal(_y(a, X[:M], M).view(np.uint32), yb.view(np.uint32))
        if kind == "w8a8":
            assert np.array_equal(yb.view(np.uint32), y_ora[:M].view(np.uint32))
        else:
            ok, worst = forward.within_tolerance(yb, *forward.reference(x[:M], w_hat))
            assert ok, (M, worst)


def test_forward_host_graph_replays(qlin):
    """qlin_forward_host captures its copies and kernels into a graph per argument set and
    replays it: new input contents, another output buffer, another M and re-attached weights
    must all give qlin_forward's outputs bit for bit."""
    N, K = 256, 1024
    W, X = synth.spqr_layer(N, K, 8, seed=51)
    layer = qlin.QLinear.from_spqr(W, 0.01).to("cuda", max_M=8)
    stream = torch.cuda.Stream()
    Xd = torch.empty((8, K), dtype=torch.bfloat16, device="cuda")
    Yd = torch.empty((8, N), dtype=torch.bfloat16, device="cuda")
    Xh = torch.empty((8, K), dtype=torch.bfloat16).pin_memory()
    Yh = [torch.empty((8, N), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    X2 = synth.activations_bf16(52, 8, K)

    def expect(xbits, M):
        return _y(layer, xbits[:M], M).view(np.uint32)

    def host(xbits, M, yh):
        Xh[:M].copy_(torch.from_numpy(np.ascontiguousarray(xbits[:M])).view(torch.bfloat16))
        qlin.qlin_forward_host(layer.handle, Xh, yh, Xd, Yd, M, stream)
        return bits_to_f32(yh[:M].view(torch.int16).numpy().view(np.uint16)).view(np.uint32)

    for M in (1, 1, 5):
        assert np.array_equal(host(X, M, Yh[0]), expect(X, M))
    assert np.array_equal(host(X2, 1, Yh[0]), expect(X2, 1))  # replay reads the new input
    assert np.array_equal(host(X2, 1, Yh[1]), expect(X2, 1))  # another output buffer
    nb = qlin.qlin_device_bytes(layer.handle)
    image = layer.weights[(-layer.weights.data_ptr()) % 256:][:nb]
    copy = torch.empty_like(image)  # a fresh allocation: 256-byte aligned
    copy.copy_(image)
    torch.cuda.synchronize()
    qlin.qlin_attach(layer.handle, copy.data_ptr(), nb)
    assert np.array_equal(host(X2, 5, Yh[1]), expect(X2, 5))  # other weights, same values


# ----------------------------------------------------------------------------- SpQR

@pytest.mark.parametrize("N,K,frac", [(128, 512, 0.01), (100, 768, 0.02), (64, 256, 0.0)])
def test_spqr_device_dequant_bit_exact(qlin, N, K, frac):
    W = synth.student_t3(13, 0.02, (N, K))
    layer = qlin.QLinear.from_spqr(W, frac).to("cuda")
    wd = layer.dequant_device().cpu().numpy()
    ref = spqr.pack(W, frac)["w_hat"]
    assert np.array_equal(wd.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("N,K,frac", [(128, 512, 0.01), (100, 768, 0.02), (1000, 2048, 0.01), (192, 1024, 0.001)])
@pytest.mark.parametrize("M", [1, 2, 5, 8, 16])
def test_spqr_forward_tolerance(qlin, N, K, frac, M):
    """frac = 0.001 leaves most (unit, row tile) outlier buckets nearly empty; 0.02 fills them."""
    W, X = synth.spqr_layer(N, K, M, seed=M)
    layer = qlin.QLinear.from_spqr(W, frac).to("cuda")
    _check(_y(layer, X, M), X, spqr.pack(W, frac)["w_hat"])


@pytest.mark.parametrize("M", [1, 5, 16, 40, 512])
def test_spqr_outliers_crowded_into_few_rows(qlin, M):
    """Four rows carry weights 100x larger, so most outliers sit in them: row runs of
    hundreds of entries inside one bucket, and units whose outliers overflow the staged copy
    (read from global memory instead).  M = 40 runs the same layer through the prefill path,
    M = 512 through its CTA pairs (two token tiles share each weight tile)."""
    N, K, frac = 128, 1024, 0.04
    W = synth.student_t3(23, 0.02, (N, K))
    W[[5, 6, 7, 70]] *= 100.0
    X = synth.activations_bf16(23, M, K)
    layer = qlin.QLinear.from_spqr(W, frac).to("cuda")
    _check(_y(layer, X, M), X, spqr.pack(W, frac)["w_hat"])


@pytest.mark.parametrize("M", [1, 5, 40, 512])
def test_spqr_widest_rows(qlin, M):
    """K = 32768, the widest row the int16 outlier columns allow (128 supergroups per row
    group, a long staged range of bucket offsets per CTA), decode and prefill (M = 512: CTA
    pairs over 512 k-blocks)."""
    N, K = 96, 32768
    W, X = synth.spqr_layer(N, K, M, seed=31)
    layer = qlin.QLinear.from_spqr(W, 0.01).to("cuda")
    _check(_y(layer, X, M), X, spqr.pack(W, 0.01)["w_hat"])


@pytest.mark.parametrize("M", [1, 16, 40])
def test_w4_widest_rows(qlin, M):
    N, K = 96, 32768
    W, X = synth.gptq_layer(N, K, M, seed=32)
    layer = qlin.QLinear.from_w4g128(W).to("cuda")
    _check(_y(layer, X, M), X, gptq_w4.pack(W)["w_hat"])


def test_spqr_one_hot_rows(qlin):
    """M == 1 accumulates exact integer products per (row, group): one-hot rows are bit-exact.
    M >= 2 dequantizes to bf16 in registers (one bf16 FMA of s^ and -s^ z^ per pair), so there
    the bar is the stated tolerance -- here at most 2^-7 relative plus the bf16 rounding of the
    s^ z^ term."""
    N, K = 128, 512
    W = synth.student_t3(17, 0.02, (N, K))
    layer = qlin.QLinear.from_spqr(W, 0.02).to("cuda")
    p = spqr.pack(W, 0.02)
    w_hat = p["w_hat"]
    for k in (0, 3, 100, 255, 256, 511):
        X = np.zeros((1, K), dtype=np.float32)
        X[0, k] = 1.0
        y = _y(layer, synth.f32_to_bf16(X), 1)
        assert np.array_equal(y[0], bf16_round(w_hat[:, k])), k
    ks = [3, 100, 255, 256, 511]
    X = np.zeros((len(ks), K), dtype=np.float32)
    for i, k in enumerate(ks):
        X[i, k] = 1.0
    y = _y(layer, synth.f32_to_bf16(X), len(ks))
    sh = np.repeat(np.abs(p["s_hat"]).astype(np.float64), 16, axis=1)
    zh = np.repeat(np.abs(p["z_hat"]).astype(np.float64), 16, axis=1)
    for i, k in enumerate(ks):
        ref = w_hat[:, k].astype(np.float64)
        bound = 2.0 ** -7 * (np.abs(ref) + sh[:, k] * (7 + zh[:, k])) + 1e-9
        assert np.all(np.abs(y[i] - ref) <= bound), k


def test_spqr_zero_dequantized_scale_groups(qlin):
    """Groups whose 3-bit scale code is 0 (dequantized scale exactly 0, codes 0, the group's
    outlier kept as fp16(w)): device dequantization bit-exact, decode (M = 1, 5) and prefill
    (M = 40; 512 in CTA pairs) within tolerance, and the one-hot columns of the outliers
    bit-exact at M = 1."""
    N, K = 128, 512
    W = synth.spqr_quiet_group_layer(N, K, seed=4)
    frac = (N + 0.5) / (N * K)
    p = spqr.pack(W, frac)
    layer = qlin.QLinear.from_spqr(W, frac).to("cuda", max_M=512)
    assert layer.handle.info.nnz == N
    wd = layer.dequant_device().cpu().numpy()
    assert np.array_equal(wd.view(np.uint32), p["w_hat"].view(np.uint32))
    for M in (1, 5, 40, 512):
        X = synth.activations_bf16(4, M, K)
        _check(_y(layer, X, M), X, p["w_hat"])
    for k in sorted({int(np.flatnonzero(p["mask"][r])[0]) for r in range(0, N, 9)}):
        X = np.zeros((1, K), dtype=np.float32)
        X[0, k] = 1.0
        y = _y(layer, synth.f32_to_bf16(X), 1)
        assert np.array_equal(y[0], bf16_round(p["w_hat"][:, k])), k


@pytest.mark.parametrize("fmt,N,K", [("w4", 64, 128), ("w4", 64, 256), ("w4", 128, 384), ("w4", 192, 640),
                                     ("spqr", 64, 256), ("spqr", 64, 512), ("spqr", 128, 768), ("spqr", 200, 1024)])
def test_single_token_tiny_layers(qlin, fmt, N, K):
    """Layers with fewer units than the single-token kernel has workers: some workers get no
    units (and must still complete the row groups they sit in), twice in a row."""
    if fmt == "w4":
        W, X = synth.gptq_layer(N, K, 1, seed=61)
        layer, w_hat = qlin.QLinear.from_w4g128(W).to("cuda"), gptq_w4.pack(W)["w_hat"]
    else:
        W, X = synth.spqr_layer(N, K, 1, seed=61)
        layer, w_hat = qlin.QLinear.from_spqr(W, 0.01).to("cuda"), spqr.pack(W, 0.01)["w_hat"]
    y0 = _y(layer, X, 1)
    _check(y0, X, w_hat)
    assert np.array_equal(_y(layer, X, 1).view(np.uint32), y0.view(np.uint32))


# ----------------------------------------------------------------------------- W8A8

@pytest.mark.parametrize("N,K", [(128, 512), (100, 256), (256, 2048)])
@pytest.mark.parametrize("M", [1, 7, 16])
def test_w8a8_codes_accumulators_and_output(qlin, N, K, M):
    W, X, absmax, _ = synth.smoothquant_layer(N, K, M, seed=M + 1)
    layer = qlin.QLinear.from_w8(W, absmax, 0.85).to("cuda", max_M=16)
    pk = smoothquant.quantize_weights(W, absmax, 0.85)
    assert np.array_equal(layer.dequant_device().cpu().numpy(), pk["qw"])
    x = bits_to_f32(X)
    qx_ref, sx_ref = smoothquant.quantize_activations(x, pk["s_inv"])
    Xd = _dev(X).view(torch.bfloat16)
    qx, sx = layer.act_quant(Xd)
    assert np.array_equal(qx.cpu().numpy(), qx_ref)
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), sx_ref.view(np.uint32))
    acc = layer.forward_acc(Xd).cpu().numpy()
    acc_ref = smoothquant.accumulate(qx_ref, pk["qw"])
    assert np.array_equal(acc.astype(np.int64), acc_ref)
    y = _y(layer, X, M)
    y_ref = smoothquant.epilogue(acc_ref, sx_ref, pk["sw"])
    assert np.array_equal(y.view(np.uint32), y_ref.view(np.uint32))


# ----------------------------------------------------------------------------- edge cases

def test_m_zero_is_noop_and_bad_args(qlin):
    W = synth.normal(0, synth.KEY_W, 0.02, (64, 256))
    layer = qlin.QLinear.from_w4g128(W).to("cuda")
    X = torch.zeros((1, 256), dtype=torch.bfloat16, device="cuda")
    Y = torch.zeros((1, 64), dtype=torch.bfloat16, device="cuda")
    qlin.qlin_forward(layer.handle, X, Y, 0)
    with pytest.raises(qlin.QlinError) as e:
        qlin.qlin_forward(layer.handle, X.data_ptr() + 2, Y, 1)   # misaligned X
    assert e.value.status == qlin.QLIN_ERR_INVALID_ARG
    unbound = qlin.QLinear.from_w4g128(W)
    with pytest.raises(qlin.QlinError) as e:
        qlin.qlin_forward(unbound.handle, X, Y, 1)
    assert e.value.status == qlin.QLIN_ERR_NOT_BOUND


def test_zero_weights_and_zero_activations(qlin):
    N, K = 64, 512
    layer = qlin.QLinear.from_spqr(np.zeros((N, K), np.float32), 0.01).to("cuda")
    X = synth.activations_bf16(0, 2, K)
    assert np.all(_y(layer, X, 2) == 0)
    W = synth.normal(0, synth.KEY_W, 0.02, (N, K))
    layer = qlin.QLinear.from_w4g128(W).to("cuda")
    assert np.all(_y(layer, np.zeros((3, K), np.uint16), 3) == 0)


def test_device_wait_limit_reports_timeout(qlin):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    qlin.qlin_debug_wait_timeout(status, 20000)  # 20 ms
    torch.cuda.synchronize()
    assert int(status.item()) == qlin.QLIN_ERR_TIMEOUT
    # the context is still usable afterwards
    W = synth.normal(0, synth.KEY_W, 0.02, (64, 256))
    layer = qlin.QLinear.from_w4g128(W).to("cuda")
    assert np.all(np.isfinite(_y(layer, synth.activations_bf16(0, 1, 256), 1)))


def test_repeated_forwards_are_deterministic(qlin):
    # many row groups split across CTAs: counters must return to zero between calls
    W, X = synth.spqr_layer(2000, 1024, 1, seed=3)
    layer = qlin.QLinear.from_spqr(W, 0.01).to("cuda")
    Xd = _dev(X).view(torch.bfloat16)
    ys = [layer(Xd).clone() for _ in range(5)]
    torch.cuda.synchronize()
    for y in ys[1:]:
        assert torch.equal(y, ys[0])
    assert layer.poll_status() == 0
