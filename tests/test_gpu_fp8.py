"""GPU parity of the static-FP8 variant against the oracle (the "flashrt-structures 0.2.0,
prefill_tower/fp8_chain.py" page, its description;
"Stabilize Higgs Audio termination and prefill", Summary):

- E4M3 weight and activation quantization: codes and scales bit-exact;
- the FP8 tcgen05 GEMM (kind::f8f6f4) against the oracle's FP8 linear on the same codes and scales,
  for every epilogue and the plan shapes of the tile kernel (M below one tile, split K, several
  rounds with last-round K pieces, SwiGLU with a ragged tile), from 512 rows in both GEMM forms
  (2-CTA clusters and single CTAs);
- calibration: max |input| of every projection within one bf16 step of the oracle's;
- the FP8 prefill against the oracle's FP8 prefill (both given the oracle's calibrated activation
  scales, so no oracle input comes from the GPU), tiny model and one full-width layer; its noise
  floor also takes the oracle re-run with every static scale one fp32 ulp higher, and past the
  first quantization the bar is widened by the E4M3 amplification (tests/parity.py) while the
  result must stay well inside the gap between the oracle's FP8 and bf16 prefills."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from parity import assert_parity, assert_parity_fp8, bf16_ulp, ref_np, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def hra():
    import qwen3_prefill_delayed_gb300 as h
    h.lib()
    return h


def _rand(shape, std, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * std).to(torch.bfloat16)


def test_quantization_bit_exact(hra):
    for shape, std, seed in (((6144, 2560), 0.02, 1), ((512, 256), 3.0, 2), ((8, 64), 1e-3, 3)):
        w = _rand(shape, std, seed)
        w8, sc = hra.fp8_quantize_weight(w.to(DEV))
        sc_o, q_o = oracle.quantize_weight_e4m3(W.to_u16(w))
        assert float(sc.item()) == sc_o
        np.testing.assert_array_equal(w8.cpu().numpy(), q_o)
        x = _rand(shape, 5.0, seed + 10)
        s = torch.tensor([0.0371], dtype=torch.float32)
        x8 = hra.fp8_quantize(x.to(DEV), s.to(DEV))
        np.testing.assert_array_equal(x8.cpu().numpy(), oracle.quantize_e4m3(W.to_u16(x), float(s.item())))


CASES = [
    # M, N, K, epilogue
    (13, 512, 256, "store"),                # one partly filled M tile
    (64, 1024, 1024, "f32"),                # one M tile, split K
    (300, 768, 256, "swiglu"),
    (130, 1000, 512, "swiglu"),             # ragged SwiGLU tile
    (1000, 2560, 1024, "residual"),
    (4255, 2560, 640, "store"),             # several rounds; the last one in K pieces
    (1000, 1536, 1024, "swiglu"),           # 2-CTA form: gate rows in one CTA, up rows in the other
]
PAIR_MIN_M = 512   # the library's threshold for the 2-CTA form
CASES_BOTH = [c + (True,) for c in CASES] + [c + (False,) for c in CASES if c[0] >= PAIR_MIN_M]


@pytest.fixture()
def gemm_form(hra, request):
    prev = hra.hra_set_gemm_pairs(request.param)
    yield request.param
    hra.hra_set_gemm_pairs(prev)


@pytest.mark.parametrize("M,N,K,epi,gemm_form", CASES_BOTH, indirect=["gemm_form"])
def test_fp8_linear(hra, M, N, K, epi, gemm_form):
    code = {"store": hra.EPI_STORE, "residual": hra.EPI_RESIDUAL, "swiglu": hra.EPI_SWIGLU, "f32": hra.EPI_F32}[epi]
    rows = 2 * N if epi == "swiglu" else N
    w = _rand((rows, K), 0.02, N + K)
    x = _rand((M, K), 1.0, M + 3 * K)
    w8, w_sc = hra.fp8_quantize_weight(w.to(DEV))
    a_sc = torch.tensor([float(np.abs(x.float().numpy()).max()) / 448.0], dtype=torch.float32, device=DEV)
    x8 = hra.fp8_quantize(x.to(DEV), a_sc)
    scale = np.float32(a_sc.item()) * np.float32(w_sc.item())
    acc = oracle.linear_fp8(x8.cpu().numpy(), w8.cpu().numpy(), float(scale)).astype(np.float64)
    xd = oracle.e4m3_decode(x8.cpu().numpy()).astype(np.float64)
    wd = oracle.e4m3_decode(w8.cpu().numpy()).astype(np.float64)
    bound = 2 * K * 2.0 ** -24 * (np.abs(xd) @ np.abs(wd).T) * float(scale) + 1e-30
    out = None
    if epi == "residual":
        r0 = _rand((M, N), 1.0, 99)
        out = r0.to(DEV).clone()
    got = to_np(hra.hra_linear_fp8(x8, w8, a_sc, w_sc, code, out=out))
    torch.cuda.synchronize()
    if epi == "f32":
        assert np.all(np.abs(got - acc) <= bound)
        return
    if epi == "store":
        ref, tol = acc, bf16_ulp(acc) + bound
    elif epi == "residual":
        ref = r0.double().numpy() + acc
        tol = bf16_ulp(ref) + bound
    else:
        g = np.float32(acc[:, :N]); u = np.float32(acc[:, N:])
        gb = oracle.bf16_value(oracle.bf16_bits(g)).astype(np.float32)
        ub = oracle.bf16_value(oracle.bf16_bits(u)).astype(np.float32)
        ref = (gb / (np.float32(1) + np.exp(-gb)) * ub).astype(np.float64)
        dg = np.abs(ub.astype(np.float64)) * 1.1 * (bound[:, :N] + bf16_ulp(g))
        du = np.abs(gb.astype(np.float64)) * (bound[:, N:] + bf16_ulp(u))
        tol = 2 * bf16_ulp(ref) + dg + du
    refb = oracle.bf16_value(oracle.bf16_bits(np.float32(ref))).astype(np.float64)
    bad = np.abs(got - refb) > tol + 1e-7
    assert not bad.any(), f"{bad.sum()} of {bad.size} outside tolerance; worst {np.max(np.abs(got - refb))}"


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
def test_fp8_prefill_and_calibration(hra, which):
    if which == "tiny":
        d = W.tiny_dims()
        lens_cal, lens = [13, 7], [13, 5, 9, 1]
        n_slots = 32
    else:
        d = W.full_dims(1)
        lens_cal, lens = [40, 24], [96, 13, 200]
        n_slots = 256
    w = W.make_backbone(d, 5, "cpu")
    hw = oracle.host_weights_from(d, w)
    bb = hra.Backbone(d, _dev_w(w))
    f8 = hra.Fp8Backbone(bb)
    # calibration on its own prompts (GPU) against the oracle's
    tok_cal = _tokens(50, lens_cal, d.vocab)
    cache = hra.new_kv_cache(d, len(lens_cal), n_slots, DEV)
    amax, a_scale = f8.calibrate(torch.from_numpy(tok_cal).to(DEV), lens_cal, cache)
    amax_o = oracle.calibrate(d, hw, tok_cal, lens_cal, n_slots)
    got = amax.cpu().numpy()
    assert np.all(np.abs(got - amax_o) <= bf16_ulp(amax_o)), (got, amax_o)
    np.testing.assert_array_equal(a_scale.cpu().numpy(), np.where(got > 0, got / np.float32(448.0), 1.0).astype(np.float32))
    # FP8 prefill with the oracle's scales on both sides
    a_o = (amax_o / np.float32(448.0)).astype(np.float32)
    f8.a_scale.copy_(torch.from_numpy(a_o).to(DEV))
    f8o = oracle.Fp8Weights(hw, a_o)
    np.testing.assert_array_equal(f8.w_scale.cpu().numpy(), np.array(f8o.w_scale, np.float32))
    tok = _tokens(51, lens, d.vocab)
    cache = hra.new_kv_cache(d, len(lens), n_slots, DEV, fill=float("nan"))
    hid = f8.prefill(torch.from_numpy(tok).to(DEV), lens, cache)
    assert hra.hra_device_error(f8.last_ws) == 0
    kv_o, hid_o = oracle.prefill_fp8(d, hw, f8o, tok, lens, n_slots)
    with oracle.sum_order(True):
        kv_a, hid_a = oracle.prefill_fp8(d, hw, f8o, tok, lens, n_slots)
    # a second equally valid oracle run: every static scale one fp32 ulp up (the calibration fixes
    # a scale only up to its rounding; E4M3 turns such last-bit changes into whole-step code flips)
    f8u = oracle.Fp8Weights(hw, np.nextafter(a_o, np.float32(np.inf)))
    kv_u, hid_u = oracle.prefill_fp8(d, hw, f8u, tok, lens, n_slots)
    kv_b, hid_b = oracle.prefill(d, hw, tok, lens, n_slots)          # the bf16 prefill, for the gap check
    assert_parity_fp8(to_np(hid), ref_np(hid_o), (ref_np(hid_a), ref_np(hid_u)), ref_np(hid_b), what="fp8 last hidden")
    g = cache.float().cpu().numpy()
    for b, n in enumerate(lens):
        # the first layer's K/V pass one quantization (of a bit-exact RMSNorm output): the plain bar
        first = slice(0, 1)
        assert_parity(g[first, b, :, :, :n].astype(np.float64), ref_np(kv_o[first, b, :, :, :n]),
                      ref_np(kv_a[first, b, :, :, :n]), what=f"fp8 layer-0 kv seq {b}",
                      extra_alts=(ref_np(kv_u[first, b, :, :, :n]),))
        if d.n_layers > 1:
            assert_parity_fp8(g[1:, b, :, :, :n].astype(np.float64), ref_np(kv_o[1:, b, :, :, :n]),
                              (ref_np(kv_a[1:, b, :, :, :n]), ref_np(kv_u[1:, b, :, :, :n])),
                              ref_np(kv_b[1:, b, :, :, :n]), what=f"fp8 kv seq {b}")
        assert np.all(np.isnan(g[:, b, :, :, n:]))
