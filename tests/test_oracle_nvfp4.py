"""Pins of the oracle's NVFP4 codec and block-scaled linear (the prefill chain's FP4 band: the
fp8_chain page's precision bands put the FFN pair and the output projection in NVFP4 with block
scales computed from the data; element and scale formats from NVIDIA's published NVFP4 definition):

- E2M1 from the format's definition: the 16 codes decode to m/2 (exponent field 0) or
  (1 + m/2) 2^(e-1); finite codes re-encode to themselves; midpoints go to the even mantissa;
  magnitudes beyond 6 saturate; every encoding is a nearest grid value (brute force);
- block quantization: each element decodes to a nearest point of its block's grid
  g * scale * {E2M1 values} (brute force over the grid); the block's largest magnitude lands at the
  top of the grid within the E4M3 rounding of the scale, and exactly when the ideal scale is an
  E4M3 value; an all-zero block has scale 0 and zero codes; the global scale is max|x| / (6 * 448);
- the linear: within the fp32 accumulation bound of a float64 dot product of the dequantized
  operands, and bit-equal to the pinned bf16 linear when every scale is 1 (all values then exact);
  a transposed block-scale index or a dropped scale fails the brute force."""
import numpy as np
import pytest

import oracle
import workloads as W

GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


@pytest.fixture(scope="module")
def orc():
    oracle.build()
    return oracle


def test_e2m1_codes_from_the_definition(orc):
    for c in range(16):
        s, e, m = c >> 3, (c >> 1) & 3, c & 1
        ref = m / 2.0 if e == 0 else (1 + m / 2.0) * 2.0 ** (e - 1)
        v = float(orc.e2m1_decode(np.uint8(c)))
        assert v == (-ref if s else ref)
        assert int(orc.e2m1_encode(np.float32(v))) == c or (ref == 0.0 and int(orc.e2m1_encode(np.float32(v))) in (0, 8))
    assert sorted({abs(float(orc.e2m1_decode(np.uint8(c)))) for c in range(16)}) == GRID.tolist()


def test_e2m1_rounding_and_saturation(orc):
    for a, b in zip(GRID[:-1], GRID[1:]):
        mid = (a + b) / 2
        got = float(orc.e2m1_decode(orc.e2m1_encode(np.float32(mid))))
        even = a if int(orc.e2m1_encode(np.float32(a))) % 2 == 0 else b
        assert got == even, (a, b, got)
        assert float(orc.e2m1_decode(orc.e2m1_encode(np.nextafter(np.float32(mid), np.float32(0))))) == a
        assert float(orc.e2m1_decode(orc.e2m1_encode(np.nextafter(np.float32(mid), np.float32(99))))) == b
    for x in (6.0, 6.5, 1e9, np.inf):
        assert float(orc.e2m1_decode(orc.e2m1_encode(np.float32(x)))) == 6.0
        assert float(orc.e2m1_decode(orc.e2m1_encode(np.float32(-x)))) == -6.0
    x = np.random.default_rng(0).uniform(-7, 7, 4000).astype(np.float32)
    dec = orc.e2m1_decode(orc.e2m1_encode(x)).astype(np.float64)
    full = np.concatenate([-GRID[::-1], GRID])
    nearest = np.min(np.abs(x[:, None].astype(np.float64) - full[None, :]), axis=1)
    assert np.all(np.abs(dec - x) == nearest)


def _bf16(a):
    return oracle.bf16_bits(np.asarray(a, np.float32))


def test_global_scale(orc):
    x = _bf16(np.random.default_rng(1).standard_normal((7, 64)) * 3)
    amax = np.float32(np.abs(oracle.bf16_value(x)).max())
    assert orc.nvfp4_global(x) == float(amax / np.float32(6 * 448))
    assert orc.nvfp4_global(_bf16(np.zeros((2, 32)))) == 1.0


def test_block_quantization(orc):
    g_rng = np.random.default_rng(2)
    rows, K = 12, 128
    x = _bf16(g_rng.standard_normal((rows, K)) * np.exp(g_rng.uniform(-4, 4, (rows, 1))))
    x[3, 16:32] = 0                                   # an all-zero block
    g = orc.nvfp4_global(x)
    codes, scales = orc.quantize_nvfp4(x, g)
    xv = oracle.bf16_value(x).astype(np.float64)
    sc = oracle.e4m3_decode(scales).astype(np.float64)
    dec = oracle.e2m1_decode(codes).astype(np.float64)
    full = np.concatenate([-GRID[::-1], GRID])
    for r in range(rows):
        for b in range(K // 16):
            step = np.float64(np.float32(g) * np.float32(sc[r, b]))
            blk = xv[r, 16 * b:16 * b + 16]
            if step == 0.0:
                assert np.all(codes[r, 16 * b:16 * b + 16] == 0)
                assert np.all(blk == 0)
                continue
            got = step * dec[r, 16 * b:16 * b + 16]
            # each element: a nearest point of the block's grid (x / step rounded in fp32 first)
            q = (blk.astype(np.float32) / np.float32(step)).astype(np.float64)
            nearest = np.min(np.abs(q[:, None] - full[None, :]), axis=1)
            assert np.all(np.abs(dec[r, 16 * b:16 * b + 16] - q) == nearest)
            # the block's largest magnitude sits at the top of the grid, within the scale's rounding
            amax = np.abs(blk).max()
            assert abs(6 * step / amax - 1) <= 2.0 ** -4 + 1e-6, (r, b)
            assert np.max(np.abs(got)) == pytest.approx(6 * step)


def test_block_scale_exact_when_representable(orc):
    # g = 1 and a block amax of 6 * 2^e (e4m3 value 2^e): the largest element decodes exactly
    x = np.zeros((4, 32), np.float32)
    for r, e in enumerate((-3, 0, 2, 5)):
        x[r, :] = np.random.default_rng(r).uniform(-1, 1, 32) * 6 * 2.0 ** e
        x[r, 5] = 6 * 2.0 ** e
        x[r, 21] = -6 * 2.0 ** e
    xb = _bf16(x)
    codes, scales = orc.quantize_nvfp4(xb, 1.0)
    dec = oracle.e2m1_decode(codes) * oracle.e4m3_decode(np.repeat(scales, 16, axis=1))
    for r, e in enumerate((-3, 0, 2, 5)):
        assert dec[r, 5] == 6 * 2.0 ** e and dec[r, 21] == -6 * 2.0 ** e


def _dequant(codes, scales, g):
    return (oracle.e2m1_decode(codes).astype(np.float64) * np.repeat(oracle.e4m3_decode(scales).astype(np.float64), 16, axis=1)
            * np.float64(g))


@pytest.mark.parametrize("T,N,K", [(5, 7, 64), (9, 33, 256), (1, 16, 512)])
def test_linear_nvfp4_brute_force(orc, T, N, K):
    g_rng = np.random.default_rng(T + N + K)
    a = _bf16(g_rng.standard_normal((T, K)) * 2)
    w = _bf16(g_rng.standard_normal((N, K)) * 0.05)
    ga, gw = orc.nvfp4_global(a), orc.nvfp4_global(w)
    ca, sa = orc.quantize_nvfp4(a, ga)
    cw, sw = orc.quantize_nvfp4(w, gw)
    y = orc.linear_nvfp4(ca, sa, cw, sw, ga, gw).astype(np.float64)
    ad = _dequant(ca, sa, 1.0)
    wd = _dequant(cw, sw, 1.0)
    g = np.float64(np.float32(ga) * np.float32(gw))
    ref = (ad @ wd.T) * g
    # fp32: the sum over K/16 exact block terms, then one scaling
    terms = (np.abs(ad) @ np.abs(wd).T) * g
    bound = (K // 16 + 2) * 2.0 ** -24 * terms + 2.0 ** -24 * np.abs(ref) + 1e-30
    assert np.all(np.abs(y - ref) <= bound)
    # a transposed block-scale index (t <-> block) or a dropped weight scale is far outside it
    if T > 1 and K // 16 > 1:
        bad = (ad / np.repeat(oracle.e4m3_decode(sa).astype(np.float64), 16, axis=1)) @ wd.T * g
        assert np.any(np.abs(bad - ref) > 10 * bound)


def test_linear_nvfp4_equals_bf16_linear_when_scales_are_one(orc):
    g_rng = np.random.default_rng(5)
    T, N, K = 6, 11, 96
    ca = g_rng.integers(0, 16, (T, K), dtype=np.uint8)
    cw = g_rng.integers(0, 16, (N, K), dtype=np.uint8)
    one = np.uint8(orc.e4m3_encode(np.float32(1.0)))
    sa = np.full((T, K // 16), one, np.uint8)
    sw = np.full((N, K // 16), one, np.uint8)
    y = orc.linear_nvfp4(ca, sa, cw, sw, 1.0, 1.0)
    ab = oracle.bf16_bits(oracle.e2m1_decode(ca))
    wb = oracle.bf16_bits(oracle.e2m1_decode(cw))
    np.testing.assert_array_equal(y, orc.linear(ab, wb))


def _nvfp4_setup(orc, d, w, tok, lens):
    hw = orc.host_weights_from(d, w)
    amax = orc.calibrate(d, hw, tok, lens, 32)
    return hw, amax


def test_nvfp4_band_scales(orc):
    """The band's static input scales: amax / 448 for the QKV input (its FP8 scale), amax / (6 * 448)
    for the NVFP4 inputs, 1 where amax is 0."""
    amax = np.array([[448.0, 2688.0, 0.0, 5.0]], np.float32)
    np.testing.assert_array_equal(orc.nvfp4_a_scales(amax), np.array([[1.0, 1.0, 1.0, np.float32(5.0) / np.float32(2688.0)]],
                                                                      np.float32))


def test_nvfp4_prefill_pins(orc):
    """The NVFP4-band prefill: batch/pad invariant bit for bit; its layer-0 K/V (QKV in the band's
    static FP8) equal the FP8 prefill's with the same QKV weights and scale; it stays close to the
    bf16 prefill but farther from it than the FP8 variant (the NVFP4 band does quantize, more
    coarsely); and each NVFP4 projection's inputs are quantized (the band's activation codes), so
    moving one NVFP4 input scale moves the result while moving an unused one does not."""
    d = W.tiny_dims()
    w = W.make_backbone(d, 0, "cpu")
    g = np.random.default_rng(14)
    lens = [13, 6, 9]
    tok = np.zeros((3, 13), np.int32)
    for b, n in enumerate(lens):
        tok[b, :n] = g.integers(0, d.vocab, n)
    hw, amax = _nvfp4_setup(orc, d, w, tok, lens)
    a_sc = orc.nvfp4_a_scales(amax)
    nv = orc.Nvfp4Weights(hw, a_sc)
    kv4, last4 = orc.prefill_nvfp4(d, hw, nv, tok, lens, 32)
    for b in range(3):
        t1 = np.full((1, 20), d.vocab + 3, np.int32)
        t1[0, :lens[b]] = tok[b, :lens[b]]
        kv1, last1 = orc.prefill_nvfp4(d, hw, nv, t1, [lens[b]], 32)
        np.testing.assert_array_equal(last1[0], last4[b])
        np.testing.assert_array_equal(kv1[:, 0], kv4[:, b])
    # layer 0's K/V depend only on the embedding, the first norm and the band's FP8 QKV
    f8 = orc.Fp8Weights(hw, amax / np.float32(448.0))
    kv8, last8 = orc.prefill_fp8(d, hw, f8, tok, lens, 32)
    np.testing.assert_array_equal(kv4[0], kv8[0])
    assert np.any(kv4[1] != kv8[1])
    _, last16 = orc.prefill(d, hw, tok, lens, 32)
    a4, a8, c = (orc.bf16_value(x).astype(np.float64) for x in (last4, last8, last16))
    cos = lambda u, v: np.sum(u * v, axis=1) / np.linalg.norm(u, axis=1) / np.linalg.norm(v, axis=1)
    assert np.all(cos(a4, c) > 0.95), cos(a4, c)
    assert np.all(1 - cos(a4, c) > 1 - cos(a8, c)), (cos(a4, c), cos(a8, c))
    # the gate/up input's global scale matters; halving it changes the result
    a2 = a_sc.copy()
    a2[:, 2] = a2[:, 2] * np.float32(0.5)
    _, last_h = orc.prefill_nvfp4(d, hw, orc.Nvfp4Weights(hw, a2), tok, lens, 32)
    assert np.any(last_h != last4)
