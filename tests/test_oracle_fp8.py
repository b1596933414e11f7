"""Pins of the oracle's static-FP8 variant (the "flashrt-structures 0.2.0, prefill_tower/fp8_chain.py"
page, its description: E4M3 weights with
per-tensor scales, inputs quantized with calibrated static scales; "Stabilize Higgs Audio
termination and prefill", Summary: calibration on a fixed prompt):

- the E4M3 codec from the format's definition: every code decodes to (1 + M/8) 2^(E-7) or
  M/8 2^-6, every finite code encodes back to itself, midpoints round to the even mantissa,
  overflow saturates to +-448, and inside +-448 the encoder agrees with torch's float8_e4m3fn cast;
- the FP8 linear is bit-equal to the bf16 linear on the decoded values (every E4M3 value is exact
  in bf16) and within the fp32 summation bound of a float64 brute force; weight scaling maps the
  largest magnitude to +-448;
- calibration records exactly the max |input| of each projection (layer 0 recomputed directly);
- the FP8 prefill is batch/pad invariant bit for bit and stays close to the bf16 prefill."""
import numpy as np
import pytest
import torch

import workloads as W


def test_e4m3_codes_from_the_definition(orc):
    for c in range(256):
        s, E, M = c >> 7, (c >> 3) & 15, c & 7
        v = orc.e4m3_decode(np.uint8(c))
        if E == 15 and M == 7:
            assert np.isnan(v)
            continue
        ref = (M / 8.0) * 2.0 ** -6 if E == 0 else (1 + M / 8.0) * 2.0 ** (E - 7)
        assert float(v) == (-ref if s else ref)
        assert int(orc.e4m3_encode(v)) == c or (ref == 0.0 and int(orc.e4m3_encode(v)) in (0, 128))
    assert float(orc.e4m3_decode(np.uint8(0x7E))) == 448.0


def test_e4m3_rounding_and_saturation(orc):
    finite = sorted({float(orc.e4m3_decode(np.uint8(c))) for c in range(128) if c != 0x7F})
    for a, b in zip(finite[:-1], finite[1:]):
        mid = np.float32((a + b) / 2)
        if float(mid) != (a + b) / 2:
            continue
        got = float(orc.e4m3_decode(orc.e4m3_encode(mid)))
        even = a if (int(orc.e4m3_encode(np.float32(a))) & 1) == 0 else b
        assert got == even, (a, b, got)
        assert float(orc.e4m3_decode(orc.e4m3_encode(np.nextafter(mid, np.float32(0))))) == a
        assert float(orc.e4m3_decode(orc.e4m3_encode(np.nextafter(mid, np.float32(1e9))))) == b
    for x, y in ((449.0, 448.0), (464.0, 448.0), (1e9, 448.0), (-3e5, -448.0), (2.0 ** -10, 0.0),
                 (3 * 2.0 ** -10, 2.0 ** -8)):
        assert float(orc.e4m3_decode(orc.e4m3_encode(np.float32(x)))) == y


def test_e4m3_matches_torch_inside_the_range(orc):
    g = np.random.default_rng(0)
    x = np.concatenate([g.standard_normal(20000) * s for s in (1e-3, 0.05, 1.0, 30.0)]).astype(np.float32)
    x = x[np.abs(x) <= 448.0]
    ours = orc.e4m3_decode(orc.e4m3_encode(x))
    theirs = torch.from_numpy(x).to(torch.float8_e4m3fn).float().numpy()
    np.testing.assert_array_equal(ours, theirs)


def test_fp8_linear_equals_bf16_linear_on_the_decoded_values(orc):
    g = np.random.default_rng(1)
    T, N, K = 7, 33, 192
    x8 = g.integers(0, 256, (T, K), dtype=np.uint8)
    w8 = g.integers(0, 256, (N, K), dtype=np.uint8)
    x8[(x8 & 0x7F) == 0x7F] = 0x10          # no NaN codes
    w8[(w8 & 0x7F) == 0x7F] = 0x21
    y = orc.linear_fp8(x8, w8, 1.0)
    xb = orc.bf16_bits(orc.e4m3_decode(x8))
    wb = orc.bf16_bits(orc.e4m3_decode(w8))
    np.testing.assert_array_equal(y, orc.linear(xb, wb))
    xd, wd = orc.e4m3_decode(x8).astype(np.float64), orc.e4m3_decode(w8).astype(np.float64)
    ref = xd @ wd.T
    bound = K * 2.0 ** -24 * (np.abs(xd) @ np.abs(wd).T)
    assert np.all(np.abs(y - ref) <= bound + 1e-30)
    # the scale multiplies the fp32 sum once
    np.testing.assert_array_equal(orc.linear_fp8(x8, w8, 0.375), (y * np.float32(0.375)).astype(np.float32))


def test_weight_quantization(orc):
    g = np.random.default_rng(2)
    w = orc.bf16_bits((g.standard_normal((64, 96)) * 0.02).astype(np.float32))
    sc, q = orc.quantize_weight_e4m3(w)
    wv = orc.bf16_value(w).astype(np.float32)
    assert sc == np.float32(np.abs(wv).max()) / np.float32(448.0)
    i = np.unravel_index(np.argmax(np.abs(wv)), wv.shape)
    assert float(orc.e4m3_decode(q[i])) == (448.0 if wv[i] > 0 else -448.0)
    np.testing.assert_array_equal(q, orc.e4m3_encode((wv / np.float32(sc)).astype(np.float32)))


def test_calibration_records_projection_inputs(orc):
    d = W.Dims(**{**W.tiny_dims().__dict__, "n_layers": 2})
    w = W.make_backbone(d, 0, "cpu")
    hw = orc.host_weights_from(d, w)
    g = np.random.default_rng(3)
    lens = [9, 5]
    tok = np.zeros((2, 9), np.int32)
    for b, n in enumerate(lens):
        tok[b, :n] = g.integers(0, d.vocab, n)
    amax = orc.calibrate(d, hw, tok, lens, 16)
    assert amax.shape == (2, 4) and np.all(amax > 0)
    rows = np.concatenate([hw.embed[tok[b, :n]] for b, n in enumerate(lens)])
    y = orc.rmsnorm(rows, hw.layers[0]["attn_norm"], d.rms_eps)
    assert amax[0, 0] == np.abs(orc.bf16_value(y)).max()


def _fp8_setup(orc, d, w, tok, lens):
    hw = orc.host_weights_from(d, w)
    amax = orc.calibrate(d, hw, tok, lens, 32)
    return hw, orc.Fp8Weights(hw, amax / np.float32(448.0))


def test_fp8_prefill_invariance_and_closeness(orc):
    d = W.tiny_dims()
    w = W.make_backbone(d, 0, "cpu")
    g = np.random.default_rng(4)
    lens = [13, 6, 9]
    tok = np.zeros((3, 13), np.int32)
    for b, n in enumerate(lens):
        tok[b, :n] = g.integers(0, d.vocab, n)
    hw, f8 = _fp8_setup(orc, d, w, tok, lens)
    kv8, last8 = orc.prefill_fp8(d, hw, f8, tok, lens, 32)
    for b in range(3):
        t1 = np.full((1, 20), d.vocab + 3, np.int32)
        t1[0, :lens[b]] = tok[b, :lens[b]]
        kv1, last1 = orc.prefill_fp8(d, hw, f8, t1, [lens[b]], 32)
        np.testing.assert_array_equal(last1[0], last8[b])
        np.testing.assert_array_equal(kv1[:, 0], kv8[:, b])
    _, last16 = orc.prefill(d, hw, tok, lens, 32)
    a, c = orc.bf16_value(last8).astype(np.float64), orc.bf16_value(last16).astype(np.float64)
    cos = np.sum(a * c, axis=1) / np.linalg.norm(a, axis=1) / np.linalg.norm(c, axis=1)
    assert np.all(cos > 0.99), cos
    assert np.any(last8 != last16)            # the variant does quantize
