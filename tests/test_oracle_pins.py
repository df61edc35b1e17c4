"""Pins of the oracle against what the pages and the mathematics fix (CPU only).

Each test is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign or index, a transposed operand, round-half-up instead of
half-even, a wrong group or bit order) fails at least one of them:

* grid-exact idempotence: weights built from known codes and statistics must
  come back bit for bit (RTN, W4 g128, the whole SpQR bi-level chain);
* closed forms: hand-worked RTN groups, bitstream bytes, the smoothing
  factors at alpha = 0 and alpha = 1;
* invariants: outlier count and ordering, residual rounding, int8 code error,
  the SmoothQuant identity with quantization off;
* the pages' figures (``tests/golden/page_figures.json``): group sizes,
  bits per parameter range, alpha range, memory reductions;
* brute force: pure-Python dot products on 8x16 tiles.
"""
import json
import math
import os

import numpy as np
import pytest

import qlin_synth as synth
from oracle import forward, gptq_w4, rtn, smoothquant, spqr
from oracle.fp import bf16_round, bf16_ulp, to_fp16

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


@pytest.fixture(scope="module")
def figures(golden_dir):
    with open(os.path.join(golden_dir, "page_figures.json")) as f:
        return {k: v["value"] for k, v in json.load(f).items() if not k.startswith("_")}


# ----------------------------------------------------------------------------- RTN core

def _grid_groups(rng, G, n, bits):
    """Groups whose values sit exactly on an RTN grid containing 0 and the top code."""
    qmax = 2 ** bits - 1
    q0 = rng.integers(0, qmax + 1, size=(G, n))
    q0[:, 0] = 0
    q0[:, 1] = qmax
    z0 = rng.integers(0, qmax + 1, size=G)
    mant = rng.integers(1024, 2048, size=G)  # 11-bit significands
    expo = rng.integers(-18, -6, size=G)
    s0 = to_fp16(np.ldexp(mant.astype(np.float64), expo - 10).astype(np.float32))
    v = ((q0 - z0[:, None]).astype(np.float32) * s0.astype(np.float32)[:, None]).astype(np.float32)
    return v, q0, z0, s0


@pytest.mark.parametrize("bits", [3, 4])
def test_rtn_grid_exact_idempotent(bits):
    rng = np.random.default_rng(1)
    v, q0, z0, s0 = _grid_groups(rng, 500, 16 if bits == 3 else 128, bits)
    q, s, z = rtn.quantize_groups(v, bits)
    assert np.array_equal(q, q0)
    assert np.array_equal(s.view(np.uint16), s0.view(np.uint16))
    assert np.array_equal(z.astype(np.int64), z0)
    w = rtn.dequantize_groups(q, s, z)
    assert np.array_equal(w.view(np.uint32), v.view(np.uint32))


def test_rtn_hand_worked_groups():
    # b = 2, v = [-1, 0, 0.5, 2]: lo = -1, hi = 2, scale = fp16(3/3) = 1, z = rint(1) = 1,
    # q = rint(v) + 1 = [0, 1, 1, 3] (rint(0.5) = 0: ties to even), w_hat = [-1, 0, 0, 2].
    q, s, z = rtn.quantize_groups(np.array([[-1.0, 0.0, 0.5, 2.0]], dtype=np.float32), 2)
    assert q.tolist() == [[0, 1, 1, 3]]
    assert float(s[0]) == 1.0 and float(z[0]) == 1.0
    assert rtn.dequantize_groups(q, s, z).tolist() == [[-1.0, 0.0, 0.0, 2.0]]
    # b = 3, v = [0.7, 1.4]: lo = 0, hi = 1.4, scale = fp16(0.2) = 0.199951171875, z = 0,
    # q = [rint(3.5009), rint(7.0017)] = [4, 7], w_hat = [4 s, 7 s].
    q, s, z = rtn.quantize_groups(np.array([[0.7, 1.4]], dtype=np.float32), 3)
    assert float(s[0]) == 0.199951171875 and float(z[0]) == 0.0
    assert q.tolist() == [[4, 7]]
    assert rtn.dequantize_groups(q, s, z).tolist() == [[0.7998046875, 1.399658203125]]
    # one-signed negative group, b = 4: v = [-3, -1.5]: lo = -3, hi = 0, scale = 0.2, z = 15
    q, s, z = rtn.quantize_groups(np.array([[-3.0, -1.5]], dtype=np.float32), 4)
    assert float(z[0]) == 15.0 and float(s[0]) == 0.199951171875
    assert q.tolist() == [[0, 7]]


def test_rtn_flat_and_degenerate_groups():
    q, s, z = rtn.quantize_groups(np.zeros((2, 16), dtype=np.float32), 3)
    assert np.all(q == 0) and np.all(s == 1) and np.all(z == 0)
    assert not np.signbit(z.astype(np.float32)).any()
    # a group whose only valid entries are masked out behaves like an all-zero group
    v = np.full((1, 16), 5.0, dtype=np.float32)
    _, s, z = rtn.quantize_groups(v, 3, valid=np.zeros((1, 16), dtype=bool))
    assert float(s[0]) == 1.0 and float(z[0]) == 0.0
    # tiny range: the scale would round to 0 in fp16 and becomes 2^-24
    _, s, _ = rtn.quantize_groups(np.array([[0.0, 1e-9]], dtype=np.float32), 4)
    assert float(s[0]) == 2.0 ** -24


def test_rtn_error_bound_on_random_groups():
    rng = np.random.default_rng(2)
    v = rng.standard_normal((2000, 128)).astype(np.float32) * 0.02
    q, s, z = rtn.quantize_groups(v, 4)
    w = rtn.dequantize_groups(q, s, z)
    sc = s.astype(np.float64)[:, None]
    bound = 0.5 * sc + 2.0 ** -10 * np.abs(v).max(axis=1, keepdims=True)
    assert np.all(np.abs(w.astype(np.float64) - v) <= bound)
    assert q.min() >= 0 and q.max() <= 15


def test_rtn_rejects_fp16_overflow():
    with pytest.raises(ValueError):
        rtn.quantize_groups(np.array([[-1e6, 1e6]], dtype=np.float32), 4)


# ----------------------------------------------------------------------------- W4 g128

def test_w4_nibble_order():
    q = (np.arange(128) % 16).reshape(1, 128)
    words = gptq_w4.pack_codes(q)
    assert int(words[0, 0]) == 0x76543210 and int(words[0, 1]) == 0xFEDCBA98
    assert np.array_equal(gptq_w4.unpack_codes(words), q)


def test_w4_grid_exact_roundtrip():
    rng = np.random.default_rng(3)
    N, K = 8, 512
    v, q0, z0, s0 = _grid_groups(rng, N * K // 128, 128, 4)
    W = v.reshape(N, K)
    p = gptq_w4.pack(W)
    assert np.array_equal(p["q"], q0.reshape(N, K))
    assert np.array_equal(p["w_hat"].view(np.uint32), W.view(np.uint32))
    assert np.array_equal(p["zero"].reshape(-1).astype(np.int64), z0)


def test_w4_bits_per_param_and_page_figures(figures):
    N, K = 64, 1024
    W = synth.normal(0, synth.KEY_W, 0.02, (N, K))
    p = gptq_w4.pack(W)
    nbytes = p["codes"].nbytes + p["scale"].nbytes + p["zero"].nbytes
    assert nbytes == gptq_w4.packed_bytes(N, K)
    bpp = forward.bits_per_param(nbytes, N, K)
    assert bpp == 4 + 32 / figures["gptq_group_size"] == 4.25
    # the GPTQ page's "75% smaller than FP16" is 4-bit codes alone; with g128 fp16 stats it is 73.4%
    assert abs((1 - bpp / 16) - figures["gptq_memory_reduction"]) < 0.02
    assert gptq_w4.GROUP == figures["gptq_group_size"]


def test_w4_one_hot_column():
    N, K = 16, 256
    W = synth.normal(0, synth.KEY_W, 0.02, (N, K))
    p = gptq_w4.pack(W)
    for k in (0, 1, 127, 128, 255):
        x = np.zeros((1, K), dtype=np.float32)
        x[0, k] = 1.0
        y, _ = forward.reference(x, p["w_hat"])
        assert np.array_equal(y[0], p["w_hat"][:, k].astype(np.float64))


def test_w4_rtn_error_small():
    W = synth.normal(0, synth.KEY_W, 0.02, (32, 1024))
    p = gptq_w4.pack(W)
    s = np.repeat(p["scale"].astype(np.float64), 128, axis=1)
    # half a step, stretched at the grid ends by the fp16 rounding of the scale (15 codes x 2^-11)
    assert np.all(np.abs(p["w_hat"].astype(np.float64) - W) <= 0.5 * s * (1 + 15 * 2.0 ** -11))


# ----------------------------------------------------------------------------- SpQR

def test_spqr_bitstream_bytes():
    # stream = sum_i c_i << 3i = 1 + 2*8 + 3*64 + 4*512 + 5*4096 + 6*32768 + 7*262144 = 0x1F58D1
    out = spqr.pack_bits3(np.array([[1, 2, 3, 4, 5, 6, 7, 0]]))
    assert out.tolist() == [[0xD1, 0x58, 0x1F]]
    rng = np.random.default_rng(4)
    c = rng.integers(0, 8, size=(5, 64))
    assert np.array_equal(spqr.unpack_bits3(spqr.pack_bits3(c), 64), c)


def test_spqr_outlier_count_order_and_ties():
    W = synth.student_t3(0, 0.02, (64, 512))
    for f in (0.005, 0.01, 0.02):
        m = spqr.select_outliers(W, f)
        assert m.sum() == math.floor(float(np.float32(f)) * 64 * 512)
        a = np.abs(W)
        assert a[m].min() >= a[~m].max()
    # ties: 10 equal magnitudes, 4 picked -> the 4 smallest linear indices
    W = np.zeros((2, 256), dtype=np.float32)
    idx = [3, 17, 200, 256 + 1, 256 + 9, 256 + 100, 256 + 255, 40, 41, 42]
    W.ravel()[idx] = np.where(np.arange(10) % 2 == 0, 1.0, -1.0)
    frac = 4.5 / 512  # floor(f * 512) = 4 in float64 of the fp32 value
    m = spqr.select_outliers(W, frac)
    assert sorted(np.flatnonzero(m).tolist()) == [3, 17, 40, 41]


def _bilevel_grid_weights(rng, N, K):
    """Weights whose first- and second-level statistics sit exactly on their grids (no outliers)."""
    G = K // 16
    S = K // 256
    c = to_fp16(np.ldexp(rng.integers(1, 8, size=(N, S)).astype(np.float64), -9).astype(np.float32))
    j = rng.integers(1, 8, size=(N, G))
    j[:, ::16] = 7  # max of every supergroup is 7 -> ss = c exactly
    z = rng.integers(0, 8, size=(N, G))
    z[:, 1::16] = 7  # max zero 7 -> sz = 1, zz = 0
    s_g = (np.repeat(c.astype(np.float32), 16, axis=1) * j).astype(np.float32)
    q0 = rng.integers(0, 8, size=(N, K))
    q0[:, ::16] = 0
    q0[:, 1::16] = 7
    W = ((q0 - np.repeat(z, 16, axis=1)).astype(np.float32) * np.repeat(s_g, 16, axis=1)).astype(np.float32)
    return W, q0, j, z, s_g


def test_spqr_bilevel_grid_exact():
    rng = np.random.default_rng(5)
    N, K = 6, 768
    W, q0, j, z, s_g = _bilevel_grid_weights(rng, N, K)
    p = spqr.pack(W, 0.0)
    assert p["mask"].sum() == 0
    assert np.array_equal(p["s_g"].astype(np.float32), s_g)
    assert np.array_equal(p["z_g"].astype(np.int64), z)
    assert np.array_equal(p["qs"], j)
    assert np.array_equal(p["qz"], z)
    assert np.array_equal(p["q"], q0)
    assert np.array_equal(p["w_hat"].view(np.uint32), W.view(np.uint32))
    st = p["stats"].astype(np.float32)
    assert np.all(st[:, :, 1] == 0) and np.all(st[:, :, 2] == 1) and np.all(st[:, :, 3] == 0)


def test_spqr_outlier_residual_and_canonical_dequant():
    W = synth.student_t3(0, 0.02, (48, 512))
    p = spqr.pack(W, 0.01)
    m = p["mask"]
    res = np.abs(W[m].astype(np.float64) - p["D"][m])
    err = np.abs(p["w_hat"][m].astype(np.float64) - W[m])
    # fp16 rounding of the residual (half an ulp, 2^-11 relative) plus the fp32 add
    assert np.all(err <= 2.0 ** -11 * res + 2.0 ** -24 * np.abs(W[m]) + 2.0 ** -25)
    # outliers reproduce far better than the dense part around them
    assert err.max() < np.abs(p["D"][~m] - W[~m]).max()
    wc = spqr.dequantize_canonical(48, 512, p["codes"], p["qs_bits"], p["qz_bits"], p["stats"],
                                   p["rowptr"], p["col"], p["val"])
    assert np.array_equal(wc.view(np.uint32), p["w_hat"].view(np.uint32))
    # CSR invariants
    assert p["rowptr"][0] == 0 and p["rowptr"][-1] == m.sum()
    for n in range(48):
        c = p["col"][p["rowptr"][n]:p["rowptr"][n + 1]]
        assert np.all(np.diff(c.astype(np.int64)) > 0)


def test_spqr_all_outlier_group():
    W = np.full((1, 256), 0.001, dtype=np.float32)
    W[0, :16] = 10.0  # the 16 largest -> the whole first group is outliers
    p = spqr.pack(W, 16 / 256)
    assert p["mask"][0, :16].all() and p["mask"].sum() == 16
    assert float(p["s_g"][0, 0]) == 1.0 and float(p["z_g"][0, 0]) == 0.0


def test_spqr_zero_dequantized_scale_group():
    """SpQR page, "İddia ve Gerçeklik: SpQR" (bi-level statistics), reading 3: the 16 group
    scales of a supergroup are themselves 3-bit RTN codes; scales are non-negative, so the
    second-level zero zs is 0 and a group whose scale is below ss / 2 gets qs = 0, a
    dequantized scale of exactly 0, every dense code 0 (reading 5) and D = 0 -- so an outlier
    in that group keeps fp16(w) itself (reading 7: the residual w - D with D = 0)."""
    N, K = 8, 512
    W = synth.spqr_quiet_group_layer(N, K, seed=3)
    frac = (N + 0.5) / (N * K)
    p = spqr.pack(W, frac)
    G = K // 16
    assert int(p["mask"].sum()) == N == spqr.outlier_count(N, K, frac)
    assert np.all(p["stats"][:, :, 1].astype(np.float32) == 0)  # zs = 0: scales are >= 0
    for r in range(N):
        g = (5 * r) % G
        sl = slice(16 * g, 16 * g + 16)
        ss = float(p["stats"][r, g // 16, 0])
        assert float(p["s_g"][r, g]) < ss / 2  # the first-level scale rounds to code 0
        assert p["qs"][r, g] == 0 and p["s_hat"][r, g] == 0
        assert np.all(p["q"][r, sl] == 0) and np.all(p["D"][r, sl] == 0)
        k = int(np.flatnonzero(p["mask"][r])[0])
        assert k == 16 * g + r % 16
        v = p["val"][p["rowptr"][r]]
        assert v == np.float16(W[r, k]) and p["w_hat"][r, k] == np.float32(np.float16(W[r, k]))
        others = np.delete(p["w_hat"][r, sl], r % 16)
        assert np.all(others == 0)
    # the quiet groups are the only zero scales; everything else dequantizes normally
    assert int((p["s_hat"] != 0).sum()) == N * G - N
    wc = spqr.dequantize_canonical(N, K, p["codes"], p["qs_bits"], p["qz_bits"], p["stats"], p["rowptr"],
                                   p["col"], p["val"])
    assert np.array_equal(wc.view(np.uint32), p["w_hat"].view(np.uint32))


def test_spqr_bits_per_param_in_page_range(figures):
    lo, hi = figures["spqr_bits_per_param_range"]
    N, K = 32, 4096
    W = synth.student_t3(0, 0.02, (N, K))
    expect = {}
    for f in (0.005, 0.01, 0.02):
        p = spqr.quantize(W, f)
        nbytes = sum(p[k].nbytes for k in ("codes", "qs_bits", "qz_bits", "stats", "rowptr", "col", "val"))
        nnz = int(p["mask"].sum())
        assert nbytes == spqr.packed_bytes(N, K, nnz)
        # the full-size layer (11008 x 4096) at the same fraction
        nnz_full = spqr.outlier_count(11008, 4096, f)
        expect[f] = forward.bits_per_param(spqr.packed_bytes(11008, 4096, nnz_full), 11008, 4096)
        assert lo <= expect[f] <= hi
    assert abs(expect[0.005] - 3.79) < 0.01 and abs(expect[0.01] - 3.95) < 0.01 and abs(expect[0.02] - 4.27) < 0.01
    assert spqr.GROUP == figures["spqr_group_size"]


def test_spqr_tolerance_on_student_t_layer():
    # the dense part is a real approximation: its error is bounded by its own dequantized grid
    W = synth.student_t3(0, 0.02, (32, 1024))
    p = spqr.pack(W, 0.01)
    m = p["mask"]
    sh = np.repeat(np.abs(p["s_hat"]).astype(np.float64), 16, axis=1)
    zh = np.repeat(p["z_hat"].astype(np.float64), 16, axis=1)
    ok = (~m) & (sh > 0) & (W / np.where(sh > 0, sh, 1) + zh >= -0.5) & (W / np.where(sh > 0, sh, 1) + zh <= 7.5)
    assert np.all(np.abs(p["D"][ok] - W[ok]) <= 0.5 * sh[ok] * (1 + 1e-6) + 1e-7)


# ----------------------------------------------------------------------------- SmoothQuant

def test_smoothquant_identity_with_quantization_off():
    N, K, M = 256, 512, 16
    W, X, absmax, _ = synth.smoothquant_layer(N, K, M, seed=0)
    x = synth.bf16_to_f32(X)
    s, s_inv = smoothquant.smoothing_factors(absmax, W, 0.85)
    xs = smoothquant.scale_activations(x, s_inv).astype(np.float64)
    ws = smoothquant.fold_weights(W, s).astype(np.float64)
    lhs = xs @ ws.T
    rhs = x.astype(np.float64) @ W.astype(np.float64).T
    denom = np.abs(x.astype(np.float64)) @ np.abs(W.astype(np.float64)).T
    assert np.max(np.abs(lhs - rhs) / denom) <= 1e-6
    # smoothing really moves range: outlier channels shrink on the activation side
    assert np.abs(xs).max() < np.abs(x).max()


def test_smoothing_closed_forms():
    N, K = 64, 256
    W, X, absmax, _ = synth.smoothquant_layer(N, K, 8, seed=1)
    aw = np.abs(W).max(axis=0).astype(np.float64)
    s0, _ = smoothquant.smoothing_factors(absmax, W, 0.0)
    assert np.array_equal(s0, (1.0 / aw).astype(np.float32))
    s1, s1_inv = smoothquant.smoothing_factors(absmax, W, 1.0)
    assert np.array_equal(s1, absmax.astype(np.float32))
    assert np.array_equal(s1_inv, (np.float32(1) / absmax).astype(np.float32))


def test_int8_code_error_and_range():
    N, K, M = 128, 1024, 32
    W, X, absmax, _ = synth.smoothquant_layer(N, K, M, seed=2)
    pk = smoothquant.quantize_weights(W, absmax, 0.85)
    x = synth.bf16_to_f32(X)
    qx, sx = smoothquant.quantize_activations(x, pk["s_inv"])
    xs = smoothquant.scale_activations(x, pk["s_inv"])
    assert np.all(np.abs(xs - sx[:, None] * qx.astype(np.float32)) <= sx[:, None] * (0.5 + 1e-6))
    assert np.all(np.abs(qx.astype(np.int64)).max(axis=1) == 127)
    ws = smoothquant.fold_weights(W, pk["s"])
    assert np.all(np.abs(ws - pk["sw"][:, None] * pk["qw"].astype(np.float32)) <= pk["sw"][:, None] * (0.5 + 1e-6))
    assert np.all(np.abs(pk["qw"].astype(np.int64)).max(axis=1) == 127)
    # a zero row gets scale 1 and all-zero codes
    q, sc = smoothquant.quantize_rows_int8(np.zeros((1, 8), dtype=np.float32))
    assert float(sc[0]) == 1.0 and np.all(q == 0)


def test_int8_rounding_is_half_even():
    # row max 127 -> scale 1, so codes are rint of the values themselves
    a = np.array([[127.0, 0.5, 1.5, 2.5, -0.5, -1.5]], dtype=np.float32)
    q, sc = smoothquant.quantize_rows_int8(a)
    assert float(sc[0]) == 1.0
    assert q.tolist() == [[127, 0, 2, 2, 0, -2]]


def test_w8a8_bruteforce_tile_and_alpha(figures):
    lo, hi = figures["smoothquant_alpha_range"]
    assert lo <= 0.85 <= hi
    N, K, M = 16, 256, 8
    W, X, absmax, ch = synth.smoothquant_layer(N, K, M, seed=3)
    assert len(ch) == K // 100
    pk = smoothquant.quantize_weights(W, absmax, 0.85)
    y, acc, qx, sx = smoothquant.forward(synth.bf16_to_f32(X), pk)
    for m in range(M):
        for n in range(N):
            a = 0
            for k in range(K):
                a += int(qx[m, k]) * int(pk["qw"][n, k])
            assert a == int(acc[m, n])
            yy = np.float32(np.float32(np.float32(a) * sx[m]) * pk["sw"][n])
            assert bf16_round(np.array([yy]))[0] == y[m, n]
    # accumulators of the largest layer fit int32
    assert 127 * 127 * 28672 < 2 ** 31
    # W8 storage vs FP16: the page's 50% memory figure
    bpp = forward.bits_per_param(smoothquant.packed_bytes(4096, 4096), 4096, 4096)
    assert abs((1 - bpp / 16) - figures["smoothquant_memory_reduction"]) < 0.01


# ----------------------------------------------------------------------------- forward, bf16

def test_forward_bruteforce_tiles():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((8, 40)).astype(np.float32)
    w = rng.standard_normal((16, 40)).astype(np.float32)
    y, b = forward.reference(x, w)
    for m in range(8):
        for n in range(16):
            acc = 0.0
            bb = 0.0
            for k in range(40):
                acc += float(x[m, k]) * float(w[n, k])
                bb += abs(float(x[m, k]) * float(w[n, k]))
            assert abs(acc - y[m, n]) <= 1e-12 * bb
            assert abs(bb - b[m, n]) <= 1e-12 * bb


def test_bf16_rounding_and_ulp():
    v = np.array([1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, -1 - 2 ** -8, 3.0], dtype=np.float32)
    assert bf16_round(v).tolist() == [1.0, 1.0, 1 + 2 ** -6, -1.0, 3.0]
    assert bf16_ulp(np.array([1.0, 1.5, 2.0, -0.75])).tolist() == [2 ** -7, 2 ** -7, 2 ** -6, 2 ** -8]
    ok, _ = forward.within_tolerance(np.array([1.0]), np.array([1.0 + 2 ** -8]), np.array([0.0]))
    assert ok
    ok, _ = forward.within_tolerance(np.array([1.0]), np.array([1.0 + 2 ** -6]), np.array([0.0]))
    assert not ok


def test_spqr_threshold_selection_equals_sorted_selection():
    W = synth.student_t3(9, 0.02, (96, 512))
    W.ravel()[::97] = 0.05  # many exact ties
    for f in (0.0, 0.003, 0.01, 0.02, 0.3):
        assert np.array_equal(spqr.select_outliers(W, f), spqr.select_outliers_by_threshold(W, f))
    # row subsets reproduce the full pack row for row
    p = spqr.pack(W, 0.01)
    rows = np.array([5, 0, 77])
    sub = spqr.quantize_rows(W, 0.01, rows)
    assert np.array_equal(sub["q"], p["q"][rows]) and np.array_equal(sub["D"], p["D"][rows])
    assert np.array_equal(spqr.dequantize(sub), p["w_hat"][rows])
