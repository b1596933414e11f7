"""Pins of the oracle's element kernels against what mathematics fixes: bf16 rounding against torch,
RMSNorm closed forms and invariances, linear against float64 brute force within the fp32
summation bound, RoPE against the complex-rotation form, attention against a float64 masked
softmax with explicit GQA head repetition, plus the invariants named for the path (per-pair norm
preservation, probability rows summing to 1, pad keys with zero weight, query 0 returning v0)."""
import numpy as np
import pytest
import torch
from scipy.special import softmax

U = 2.0 ** -8      # bf16 unit roundoff (8-bit significand incl. the implicit bit -> half-ulp 2^-8)


def _bits(orc, x):
    return orc.bf16_bits(np.asarray(x, np.float32))


def _val(orc, u):
    return orc.bf16_value(u).astype(np.float64)


# ------------------------------------------------------------------ bf16 rounding

def test_bf16_rounding_matches_torch(orc):
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.normal(0, 1, 100000).astype(np.float32),
        rng.normal(0, 1e-30, 1000).astype(np.float32),
        (rng.normal(0, 1, 1000) * 1e38).astype(np.float32),
        # exact ties: low 16 bits == 0x8000 with both even and odd kept bit
        (np.arange(1000, dtype=np.uint32) << 16 | 0x3f800000 | 0x8000).view(np.float32),
        np.array([0.0, -0.0, np.inf, -np.inf, 3.3895314e38], np.float32),
    ])
    ours = orc.bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)


# ------------------------------------------------------------------ RMSNorm

def test_rmsnorm_constant_vector_closed_form(orc):
    n, eps = 256, 1e-6
    for c in (0.5, -3.0, 0.0078125, 7.0):
        x = _bits(orc, np.full((1, n), c))
        g = _bits(orc, np.ones(n))
        y = _val(orc, orc.rmsnorm(x, g, eps))
        want = c / np.sqrt(c * c + eps)          # mean(x^2) = c^2
        assert np.all(np.abs(y - want) <= U * abs(want) * 1.01)


def test_rmsnorm_against_float64_and_gain(orc):
    rng = np.random.default_rng(1)
    n, eps = 2560, 1e-6
    x = _bits(orc, rng.normal(0, 1, (7, n)))
    g = _bits(orc, 1 + rng.normal(0, 0.02, n))
    y = _val(orc, orc.rmsnorm(x, g, eps))
    x64, g64 = _val(orc, x), _val(orc, g)
    ref = x64 / np.sqrt(np.mean(x64 ** 2, axis=1, keepdims=True) + eps) * g64
    assert np.all(np.abs(y - ref) <= U * np.abs(ref) + 1e-6 * np.abs(ref) + 1e-30)
    # doubling the gain doubles the output exactly (power-of-two scaling commutes with rounding)
    g2 = _bits(orc, 2 * _val(orc, g))
    np.testing.assert_array_equal(_val(orc, orc.rmsnorm(x, g2, eps)), 2 * y)
    # scale invariance up to eps: RMSNorm(2x) == RMSNorm(x) within one bf16 ulp
    x2 = _bits(orc, 2 * _val(orc, x))
    y2 = _val(orc, orc.rmsnorm(x2, g, eps))
    assert np.all(np.abs(y2 - y) <= 2 * U * np.abs(y) + 1e-30)


# ------------------------------------------------------------------ linear

@pytest.mark.parametrize("T,N,K", [(1, 300, 256), (13, 77, 640), (5, 1026, 96)])
def test_linear_brute_force_bound(orc, T, N, K):
    rng = np.random.default_rng(T * 1000 + N)
    x = _bits(orc, rng.normal(0, 1, (T, K)))
    w = _bits(orc, rng.normal(0, 0.02, (N, K)))
    y = orc.linear(x, w).astype(np.float64)
    x64, w64 = _val(orc, x), _val(orc, w)
    ref = x64 @ w64.T
    bound = K * 2.0 ** -24 * (np.abs(x64) @ np.abs(w64).T)
    assert y.shape == (T, N)
    assert np.all(np.abs(y - ref) <= bound)


def test_linear_selection_matrix_is_exact(orc):
    """W with one 1.0 per row selects input columns exactly: catches transposed operands."""
    rng = np.random.default_rng(2)
    T, K, N = 4, 48, 20
    x = _bits(orc, rng.normal(0, 1, (T, K)))
    sel = rng.permutation(K)[:N]
    w = np.zeros((N, K), np.float32)
    w[np.arange(N), sel] = 1.0
    y = orc.linear(x, _bits(orc, w))
    np.testing.assert_array_equal(y, _val(orc, x)[:, sel].astype(np.float32))


# ------------------------------------------------------------------ RoPE

def _norm64(orc, x, g, eps):
    x64, g64 = _val(orc, x), _val(orc, g)
    return x64 / np.sqrt(np.mean(x64 ** 2, axis=-1, keepdims=True) + eps) * g64


@pytest.mark.parametrize("hd", [64, 128])
def test_rope_matches_complex_rotation(orc, hd):
    rng = np.random.default_rng(hd)
    rows, eps, theta = 50, 1e-6, 1e6
    x = _bits(orc, rng.normal(0, 1, (rows, hd)))
    g = _bits(orc, 1 + rng.normal(0, 0.02, hd))
    pos = rng.integers(0, 4096, rows).astype(np.int32)
    out = _val(orc, orc.qk_norm_rope(x, g, pos, eps, theta))
    xn = _norm64(orc, x, g, eps)
    half = hd // 2
    freq = theta ** (-(2.0 * np.arange(half)) / hd)
    z = (xn[:, :half] + 1j * xn[:, half:]) * np.exp(1j * pos[:, None] * freq[None, :])
    ref = np.concatenate([z.real, z.imag], axis=1)
    scale = np.abs(xn).max()
    assert np.all(np.abs(out - ref) <= U * np.abs(ref) + 1e-5 * scale)
    # per-pair norm preserved
    pn_out = np.hypot(out[:, :half], out[:, half:])
    pn_in = np.hypot(xn[:, :half], xn[:, half:])
    assert np.all(np.abs(pn_out - pn_in) <= 2 * U * pn_in + 1e-5 * scale)


def test_rope_position_zero_is_identity(orc):
    rng = np.random.default_rng(3)
    hd, eps = 128, 1e-6
    x = _bits(orc, rng.normal(0, 1, (9, hd)))
    g = _bits(orc, 1 + rng.normal(0, 0.02, hd))
    out = orc.qk_norm_rope(x, g, np.zeros(9, np.int32), eps, 1e6)
    np.testing.assert_array_equal(out, orc.rmsnorm(x, g, eps))


def test_rope_relative_position(orc):
    """<R_m q, R_n k> depends only on m - n."""
    rng = np.random.default_rng(4)
    hd, eps = 128, 1e-6
    q = _bits(orc, rng.normal(0, 1, (1, hd)))
    k = _bits(orc, rng.normal(0, 1, (1, hd)))
    g = _bits(orc, np.ones(hd))
    vals = []
    for shift in (0, 17, 900, 3000):
        qr = _val(orc, orc.qk_norm_rope(q, g, np.array([40 + shift], np.int32), eps, 1e6))
        kr = _val(orc, orc.qk_norm_rope(k, g, np.array([25 + shift], np.int32), eps, 1e6))
        vals.append(float((qr @ kr.T)[0, 0]))
    assert max(vals) - min(vals) <= 4 * U * hd ** 0.5 * 2


def test_rope_table_values(orc):
    c, s = orc.rope_table(4096, 128, 1e6)
    assert np.all(c[0] == 1.0) and np.all(s[0] == 0.0)
    i = np.arange(64)
    ang = np.arange(4096)[:, None] * (1e6 ** (-(2.0 * i) / 128))[None, :]
    np.testing.assert_allclose(c, np.cos(ang), rtol=0, atol=2 ** -24)
    np.testing.assert_allclose(s, np.sin(ang), rtol=0, atol=2 ** -24)


# ------------------------------------------------------------------ attention

def _attn_inputs(orc, rng, n, nq, nkv, hd, n_slots, pos0=0):
    q = _bits(orc, rng.normal(0, 1, (n, nq, hd)))
    kc = _bits(orc, rng.normal(0, 1, (nkv, n_slots, hd)))
    vc = _bits(orc, rng.normal(0, 1, (nkv, n_slots, hd)))
    return q, kc, vc


def _brute(orc, q, kc, vc, pos0):
    n, nq, hd = q.shape
    nkv = kc.shape[0]
    kk = np.repeat(_val(orc, kc), nq // nkv, axis=0)      # [nq, S, hd]: head h -> kv h // group
    vv = np.repeat(_val(orc, vc), nq // nkv, axis=0)
    q64 = _val(orc, q)
    nk = pos0 + n
    s = np.einsum("ihd,hjd->hij", q64, kk[:, :nk]) / np.sqrt(hd)
    mask = np.arange(nk)[None, :] <= (pos0 + np.arange(n))[:, None]
    s = np.where(mask[None], s, -np.inf)
    p = softmax(s, axis=-1)
    o = np.einsum("hij,hjd->ihd", p, vv[:, :nk])
    return o.reshape(n, nq * hd), p


@pytest.mark.parametrize("n,nq,nkv,hd,pos0", [(13, 4, 2, 64, 0), (7, 8, 2, 128, 30), (1, 32, 8, 128, 200)])
def test_attention_brute_force(orc, n, nq, nkv, hd, pos0):
    rng = np.random.default_rng(n + nq + pos0)
    S = pos0 + n + 5
    q, kc, vc = _attn_inputs(orc, rng, n, nq, nkv, hd, S)
    out, probs = orc.attend(q, kc, vc, pos0, want_probs=True)
    ref, p_ref = _brute(orc, q, kc, vc, pos0)
    assert np.all(np.abs(_val(orc, out) - ref) <= U * np.abs(ref) + 1e-5)
    np.testing.assert_allclose(probs.transpose(1, 0, 2), p_ref, rtol=1e-5, atol=1e-7)
    # rows sum to 1; keys past the query position have weight exactly 0
    np.testing.assert_allclose(probs.sum(-1), 1.0, rtol=0, atol=1e-5)
    for i in range(n):
        assert np.all(probs[i, :, pos0 + i + 1:] == 0.0)


def test_attention_pad_keys_unread(orc):
    """NaN in every slot past the used run changes nothing: pads carry zero weight and are unread."""
    rng = np.random.default_rng(7)
    n, nq, nkv, hd, S = 9, 4, 2, 64, 32
    q, kc, vc = _attn_inputs(orc, rng, n, nq, nkv, hd, S)
    clean = orc.attend(q, kc, vc, 0)
    nan = np.uint16(0x7fc0)
    kc2, vc2 = kc.copy(), vc.copy()
    kc2[:, n:] = nan
    vc2[:, n:] = nan
    np.testing.assert_array_equal(orc.attend(q, kc2, vc2, 0), clean)
    # causality: perturbing key/value j changes only rows i >= j
    kc3, vc3 = kc.copy(), vc.copy()
    kc3[:, 5] = _bits(orc, rng.normal(0, 1, (nkv, hd)))
    vc3[:, 5] = _bits(orc, rng.normal(0, 1, (nkv, hd)))
    pert = orc.attend(q, kc3, vc3, 0)
    np.testing.assert_array_equal(pert[:5], clean[:5])
    assert np.any(pert[5:] != clean[5:])


def test_attention_query0_and_equal_keys(orc):
    rng = np.random.default_rng(8)
    n, nq, nkv, hd, S = 6, 4, 2, 64, 8
    q, kc, vc = _attn_inputs(orc, rng, n, nq, nkv, hd, S)
    out = orc.attend(q, kc, vc, 0).reshape(n, nq, hd)
    for h in range(nq):
        np.testing.assert_array_equal(out[0, h], vc[h // (nq // nkv), 0])   # query 0 sees only key 0
    kc_eq = np.repeat(kc[:, :1], S, axis=1)                                   # all keys equal
    out_eq = _val(orc, orc.attend(q, kc_eq, vc, 0)).reshape(n, nq, hd)
    v64 = _val(orc, vc)
    for i in range(n):
        for h in range(nq):
            mean = v64[h // (nq // nkv), :i + 1].mean(0)
            assert np.all(np.abs(out_eq[i, h] - mean) <= U * np.abs(mean) + 1e-6)
