"""Pins of the oracle's sampled codebook step (temperature, top-k, top-p, exponential race on
per-row seeded Philox4x32-10 noise; vLLM-Omni PR #8226, Purpose and Test Plan):

- the generator against its published known-answer vectors (tests/golden/philox4x32_10_kat.txt);
- the noise is Exp(1): mean, and uniforms inside (0, 1];
- special cases that reduce to the pinned greedy step: top-k 1, and a top-p below every
  probability, give the argmax codes (forced BOS/EOC slots and the EOC rule included);
- the race draws from the right distribution: with fixed logits and independent seeds, the sample
  frequencies match softmax(z / T) restricted to the top-k / top-p set (a reversed race, a missing
  temperature or an off-by-one in either cut fails these)."""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")


def test_philox_known_answers():
    rows = [l.split() for l in open(GOLDEN) if l.strip() and not l.startswith("#")]
    assert len(rows) == 3
    for r in rows:
        w = [int(x, 16) for x in r]
        assert oracle.philox4x32_10(w[0:4], w[4:6]).tolist() == w[6:10]


def test_exponential_noise_is_exp1():
    e = np.array([oracle.exponential(1234, t, k, v) for t in range(4) for k in range(4) for v in range(1026)])
    assert np.all(e >= 0.0) and np.all(np.isfinite(e))
    n = e.size
    assert abs(e.mean() - 1.0) < 4.0 / np.sqrt(n)
    assert abs(np.mean(np.exp(-e)) - 0.5) < 4.0 * 0.29 / np.sqrt(n)     # exp(-E) = u is U(0, 1]
    # distinct frames, codebooks and seeds give distinct noise
    assert oracle.exponential(1, 0, 0, 5) != oracle.exponential(1, 1, 0, 5)
    assert oracle.exponential(1, 0, 0, 5) != oracle.exponential(1, 0, 1, 5)
    assert oracle.exponential(1, 0, 0, 5) != oracle.exponential(2, 0, 0, 5)
    assert oracle.exponential(1 << 40, 0, 0, 5) != oracle.exponential(0, 0, 0, 5)


def _states(rng, B, K):
    st = np.zeros((B, 4), np.int32)
    st[:, 0] = rng.integers(0, 2 * K, B)
    st[:, 1] = -1
    ended = rng.random(B) < 0.3
    st[ended, 1] = np.maximum(st[ended, 0] - rng.integers(0, K, ended.sum()), 0)
    return st


@pytest.mark.parametrize("top_k,top_p", [(1, 1.0), (0, 1e-7), (1, 0.5)])
def test_degenerate_cuts_are_greedy(top_k, top_p):
    rng = np.random.default_rng(3)
    K, Vc, B = 8, 1026, 16
    for step in range(6):
        lg = rng.standard_normal((B, K, Vc)).astype(np.float32)
        bias = np.zeros((B, K), np.float32)
        bias[rng.random((B, K)) < 0.1] = 10.0
        st = _states(rng, B, K)
        st2 = st.copy()
        c_g, d_g = oracle.delay_step(K, Vc, 1024, 1025, lg, bias, st)
        c_s, d_s, _, _ = oracle.sample_step(K, Vc, 1024, 1025, lg, bias, 0.7, top_k, top_p,
                                            rng.integers(0, 2**63, B, dtype=np.uint64), st2)
        assert c_s.tolist() == c_g.tolist() and d_s.tolist() == d_g.tolist() and st2.tolist() == st.tolist()


def _frequencies(z, T, top_k, top_p, n):
    """n independent samples (one seed each) of one codebook with logits z (frame 0, no EOC)."""
    Vc = z.size
    lg = np.tile(z.astype(np.float32), (n, 1, 1))
    seeds = np.arange(n, dtype=np.uint64) * np.uint64(0x9E3779B97F4A7C15 & 0x7FFFFFFFFFFFFFFF) + np.uint64(7)
    st = np.zeros((n, 4), np.int32)
    st[:, 1] = -1
    codes, _, _, _ = oracle.sample_step(1, Vc, Vc, Vc + 1, lg, None, T, top_k, top_p, seeds, st)
    return np.bincount(codes[:, 0], minlength=Vc) / n


def _expected(z, T, keep):
    w = np.exp((z - z.max()) / T) * keep
    return w / w.sum()


def _chi2_ok(f, p, n):
    m = p > 0
    assert np.all(f[~m] == 0), "a sample outside the kept set"
    chi2 = n * np.sum((f[m] - p[m]) ** 2 / p[m])
    dof = max(int(m.sum()) - 1, 1)
    assert chi2 < dof + 6 * np.sqrt(2 * dof) + 10, f"chi2 {chi2:.1f} with {dof} degrees of freedom"


def test_race_matches_softmax():
    z = np.array([1.2, 0.3, -0.5, 0.9, 2.0, -1.0, 0.0, 0.4], np.float64)
    n = 40000
    for T in (1.0, 0.5, 2.0):
        _chi2_ok(_frequencies(z, T, 0, 1.0, n), _expected(z, T, np.ones_like(z)), n)


def test_top_k_and_top_p_sets():
    n = 30000
    z = np.array([1.2, 0.3, -0.5, 0.9, 2.0, -1.0, 0.0, 0.4], np.float64)
    keep3 = np.isin(np.arange(8), [4, 0, 3]).astype(float)            # the three largest
    _chi2_ok(_frequencies(z, 1.0, 3, 1.0, n), _expected(z, 1.0, keep3), n)
    # ties at the top-k threshold are kept: 2nd-4th largest tie
    zt = np.array([0.0, 1.0, 1.0, 3.0, 1.0, -2.0], np.float64)
    _chi2_ok(_frequencies(zt, 1.0, 2, 1.0, n), _expected(zt, 1.0, (zt >= 1.0).astype(float)), n)
    # top-p: probabilities 0.5, 0.3, 0.15, 0.05 -> 0.79 keeps the first two, 0.81 the first three
    zp = np.log(np.array([0.15, 0.5, 0.05, 0.3]))
    _chi2_ok(_frequencies(zp, 1.0, 0, 0.79, n), _expected(zp, 1.0, np.array([0, 1, 0, 1.0])), n)
    _chi2_ok(_frequencies(zp, 1.0, 0, 0.81, n), _expected(zp, 1.0, np.array([1, 1, 0, 1.0])), n)
    # top-k then top-p: k = 3 keeps {0.5, 0.3, 0.15}; renormalised 0.526, 0.316, 0.158 -> p 0.6 keeps two
    _chi2_ok(_frequencies(zp, 1.0, 3, 0.6, n), _expected(zp, 1.0, np.array([0, 1, 0, 1.0])), n)


def test_sampling_is_seeded():
    rng = np.random.default_rng(9)
    K, Vc, B = 8, 1026, 6
    lg = rng.standard_normal((B, K, Vc)).astype(np.float32)
    seeds = rng.integers(0, 2**63, B, dtype=np.uint64)
    st = np.zeros((B, 4), np.int32)
    st[:, 0] = 9
    st[:, 1] = -1
    a = oracle.sample_step(K, Vc, 1024, 1025, lg, None, 1.0, 50, 0.95, seeds, st.copy())[0]
    b = oracle.sample_step(K, Vc, 1024, 1025, lg, None, 1.0, 50, 0.95, seeds, st.copy())[0]
    c = oracle.sample_step(K, Vc, 1024, 1025, lg, None, 1.0, 50, 0.95, seeds + np.uint64(1), st.copy())[0]
    assert a.tolist() == b.tolist()
    assert a.tolist() != c.tolist()
