"""GPU parity of the NVFP4 band (the chain's FP4 band, the fp8_chain page's precision bands)
against the pinned oracle:

- the quantizer (hra_nvfp4_quantize, hra_nvfp4_quantize_weight): codes, block scales and global
  scales bit for bit, over magnitudes that put block scales in the E4M3 normal and subnormal
  ranges, an all-zero block and saturating elements;
- the NVFP4 GEMM (hra_linear_nvfp4) against oracle_linear_nvfp4 on the same operands, within the
  fp32 summation bound, for every epilogue and ragged M / N;
- the NVFP4-band prefill (hra_prefill_nvfp4) against oracle_prefill_nvfp4 on the tiny model and
  one full-width layer."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from parity import assert_parity, assert_parity_nvfp4, bf16_ulp, ref_np, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def hra():
    import qwen3_prefill_delayed_gb300 as h
    h.lib()
    return h


@pytest.mark.parametrize("rows,K,gmode", [(40, 256, "tensor"), (7, 64, "tensor"), (33, 512, "one"), (5, 4096, "small")])
def test_nvfp4_quantize_bit_exact(hra, rows, K, gmode):
    g_rng = np.random.default_rng(rows + K)
    x = g_rng.standard_normal((rows, K)) * np.exp(g_rng.uniform(-6, 4, (rows, 1)))
    x[0, 16:32] = 0.0                        # an all-zero block
    x[1, 40] = 1e4                           # a block whose other elements round to 0
    xb = oracle.bf16_bits(x.astype(np.float32))
    g = {"tensor": oracle.nvfp4_global(xb), "one": 1.0, "small": 1e-3}[gmode]
    codes_o, scales_o = oracle.quantize_nvfp4(xb, g)
    xt = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).to(DEV)
    gt = torch.tensor([g], dtype=torch.float32, device=DEV)
    codes, scales = hra.nvfp4_quantize(xt, gt)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(scales.cpu().numpy(), scales_o)
    np.testing.assert_array_equal(codes.cpu().numpy(), codes_o)


def _quantized(rows, K, seed, std):
    g = np.random.default_rng(seed)
    x = (g.standard_normal((rows, K)) * std).astype(np.float32)
    xb = oracle.bf16_bits(x)
    gs = oracle.nvfp4_global(xb)
    c, s = oracle.quantize_nvfp4(xb, gs)
    return c, s, gs


def _dequant(codes, scales, g):
    v = oracle.e2m1_decode(codes).astype(np.float64)
    sc = np.repeat(oracle.e4m3_decode(scales).astype(np.float64), 16, axis=1)
    return v * sc * g


@pytest.mark.parametrize("M,N,K,epi", [(1, 256, 64, 3), (37, 264, 256, 3), (300, 512, 2560, 3), (129, 2560, 512, 0),
                                       (64, 2560, 1024, 1), (200, 384, 2560, 2)])
def test_nvfp4_linear(hra, M, N, K, epi):
    """hra_linear_nvfp4 against the oracle's NVFP4 linear on the same codes and scales: fp32 output
    within the fp32 summation bound of the float64 product sum (the tensor core adds in its own
    order); bf16 epilogues within one bf16 step of the oracle's value plus that bound."""
    n_w = 2 * N if epi == 2 else N
    ac, asc, ga = _quantized(M, K, M + K, 1.0)
    wc, wsc, gw = _quantized(n_w, K, N + K + 1, 0.02)
    y_o = oracle.linear_nvfp4(ac, asc, wc, wsc, ga, gw)                    # fp32 [M, n_w]
    exact = _dequant(ac, asc, ga) @ _dequant(wc, wsc, gw).T
    bound = 2.0 * K * 2.0 ** -24 * (np.abs(_dequant(ac, asc, ga)) @ np.abs(_dequant(wc, wsc, gw)).T) + 1e-30
    assert np.all(np.abs(y_o - exact) <= bound)                           # the oracle itself
    t = lambda a: torch.from_numpy(a).to(DEV)
    g_a = torch.tensor([ga], dtype=torch.float32, device=DEV)
    g_w = torch.tensor([gw], dtype=torch.float32, device=DEV)
    out = None
    if epi == 1:
        r0 = oracle.bf16_bits((np.random.default_rng(3).standard_normal((M, N))).astype(np.float32))
        out = torch.from_numpy(r0.view(np.int16)).view(torch.bfloat16).to(DEV)
    got = hra.hra_linear_nvfp4(t(ac), t(asc), t(wc), t(wsc), g_a, g_w, epi, out=out)
    torch.cuda.synchronize()
    g_np = got.float().cpu().numpy().astype(np.float64)
    if epi == 3:
        assert np.all(np.abs(g_np - exact) <= bound), np.max(np.abs(g_np - exact) - bound)
        return
    if epi == 0:
        ref = oracle.bf16_value(oracle.bf16_bits(y_o)).astype(np.float64)
        tol = bf16_ulp(ref) + bound
    elif epi == 1:
        ref = oracle.bf16_value(oracle.bf16_bits(oracle.bf16_value(r0) + y_o)).astype(np.float64)
        tol = bf16_ulp(ref) + bound
    else:
        gate = oracle.bf16_value(oracle.bf16_bits(y_o[:, :N])).astype(np.float64)
        up = oracle.bf16_value(oracle.bf16_bits(y_o[:, N:])).astype(np.float64)
        ref = gate / (1.0 + np.exp(-gate)) * up
        # one bf16 step of g or u (their fp32 sums differ in order) moves h by about that much
        tol = 2 * bf16_ulp(ref) + (np.abs(gate) + np.abs(up)) * 2.0 ** -7
    assert np.all(np.abs(g_np - ref) <= tol), f"worst excess {np.max(np.abs(g_np - ref) - tol)}"


def test_nvfp4_weight_quantization_bit_exact(hra):
    g = np.random.default_rng(21)
    w = (g.standard_normal((300, 256)) * 0.02).astype(np.float32)
    wb = oracle.bf16_bits(w)
    c_o, s_o = oracle.quantize_nvfp4(wb, oracle.nvfp4_global(wb))
    wt = torch.from_numpy(wb.view(np.int16)).view(torch.bfloat16).to(DEV)
    c, s, gg = hra.nvfp4_quantize_weight(wt)
    torch.cuda.synchronize()
    assert float(gg.item()) == oracle.nvfp4_global(wb)
    np.testing.assert_array_equal(s.cpu().numpy(), s_o)
    np.testing.assert_array_equal(c.cpu().numpy(), c_o)


def _dev_w(w):
    return {"embed": w["embed"].to(DEV), "final_norm": w["final_norm"].to(DEV),
            "layers": [{k: v.to(DEV) for k, v in l.items()} for l in w["layers"]]}


def _tokens(seed, lens, vocab):
    g = np.random.default_rng(seed)
    t = np.zeros((len(lens), max(lens)), np.int32)
    for b, n in enumerate(lens):
        t[b, :n] = g.integers(0, vocab, n)
    return t


@pytest.mark.parametrize("which", ["tiny", "full_layer"])
def test_nvfp4_prefill(hra, which):
    """The NVFP4-band prefill (hra_prefill_nvfp4) against the oracle's, on the same calibrated
    static scales; the weight codes, block scales and global scales bit for bit."""
    if which == "tiny":
        d = W.tiny_dims()
        lens_cal, lens, n_slots = [13, 7], [13, 5, 9, 1], 32
    else:
        d = W.full_dims(1)
        lens_cal, lens, n_slots = [40, 24], [96, 13, 200], 256
    w = W.make_backbone(d, 6, "cpu")
    hw = oracle.host_weights_from(d, w)
    bb = hra.Backbone(d, _dev_w(w))
    nv = hra.Nvfp4Backbone(bb)
    tok_cal = _tokens(60, lens_cal, d.vocab)
    cache = hra.new_kv_cache(d, len(lens_cal), n_slots, DEV)
    nv.calibrate(torch.from_numpy(tok_cal).to(DEV), lens_cal, cache)
    amax_o = oracle.calibrate(d, hw, tok_cal, lens_cal, n_slots)
    a_o = oracle.nvfp4_a_scales(amax_o)
    nv.a_scale.copy_(torch.from_numpy(a_o).to(DEV))                  # the oracle's scales on both sides
    nvo = oracle.Nvfp4Weights(hw, a_o)
    np.testing.assert_array_equal(nv.w_scale.cpu().numpy(), np.array(nvo.w_scale, np.float32))
    for l in range(d.n_layers):
        for p in range(1, 4):
            np.testing.assert_array_equal(nv.keep[l]["codes"][p].cpu().numpy(), nvo.keep[l]["codes"][p])
            np.testing.assert_array_equal(nv.keep[l]["scales"][p].cpu().numpy(), nvo.keep[l]["scales"][p])
    tok = _tokens(61, lens, d.vocab)
    cache = hra.new_kv_cache(d, len(lens), n_slots, DEV, fill=float("nan"))
    hid = nv.prefill(torch.from_numpy(tok).to(DEV), lens, cache)
    assert hra.hra_device_error(nv.last_ws) == 0
    kv_o, hid_o = oracle.prefill_nvfp4(d, hw, nvo, tok, lens, n_slots)
    with oracle.sum_order(True):
        kv_a, hid_a = oracle.prefill_nvfp4(d, hw, nvo, tok, lens, n_slots)
    nvu = oracle.Nvfp4Weights(hw, np.nextafter(a_o, np.float32(np.inf)))
    kv_u, hid_u = oracle.prefill_nvfp4(d, hw, nvu, tok, lens, n_slots)
    kv_b, hid_b = oracle.prefill(d, hw, tok, lens, n_slots)
    assert_parity_nvfp4(to_np(hid), ref_np(hid_o), (ref_np(hid_a), ref_np(hid_u)), ref_np(hid_b),
                        what=f"nvfp4 last hidden ({which})")
    g = cache.float().cpu().numpy()
    for b, n in enumerate(lens):
        # layer 0's K/V: embedding, norm and the band's FP8 QKV only
        assert_parity(g[:1, b, :, :, :n].astype(np.float64), ref_np(kv_o[:1, b, :, :, :n]),
                      ref_np(kv_a[:1, b, :, :, :n]), what=f"nvfp4 layer-0 kv seq {b}",
                      extra_alts=(ref_np(kv_u[:1, b, :, :, :n]),))
        if d.n_layers > 1:
            assert_parity_nvfp4(g[1:, b, :, :, :n].astype(np.float64), ref_np(kv_o[1:, b, :, :, :n]),
                                (ref_np(kv_a[1:, b, :, :, :n]), ref_np(kv_u[1:, b, :, :, :n])),
                                ref_np(kv_b[1:, b, :, :, :n]), what=f"nvfp4 kv seq {b}")
        assert np.all(np.isnan(g[:, b, :, :, n:]))
