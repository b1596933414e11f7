"""Pins of the oracle's delayed-codebook step: hand-enumerated schedules, exhaustive properties of
the delay pattern, argmax tie rule, and the codebook embedding sum.

Source of the rule: "Stabilize Higgs Audio termination and prefill" (FlashRT PR #141), Summary
(per-frame argmax, delay handling, codebook embedding accumulation) and Root cause (the old
delayed-EOC check only handled the first codebook reliably)."""
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
VC, BOS, EOC = 1026, 1024, 1025


def _argmax_code(k, t):
    return (37 * k + 11 * t) % 1000


def _parse(name):
    rows, meta = [], {"BIAS": [], "EOCLOGIT": []}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            tok = line.split()
            if tok[0] in ("K", "START"):
                meta[tok[0]] = int(tok[1])
            elif tok[0] in ("BIAS", "EOCLOGIT"):
                meta[tok[0]].append((int(tok[1]), int(tok[2])))
            else:
                rows.append(tok)
    return meta, rows


def _frame_logits(rng, K, t, meta):
    lg = rng.normal(0.0, 0.1, size=(1, K, VC)).astype(np.float32)
    for k in range(K):
        lg[0, k, _argmax_code(k, t)] = 5.0
    for (ft, k) in meta["EOCLOGIT"]:
        if ft == t:
            lg[0, k, EOC] = 20.0
    bias = np.zeros((1, K), np.float32)
    for (ft, k) in meta["BIAS"]:
        if ft == t:
            bias[0, k] = 10.0
    return lg, bias


@pytest.mark.parametrize("name", ["delay_k4_tiny.txt", "delay_k8_injected.txt", "delay_k8_two_eoc.txt"])
def test_hand_schedule(orc, name):
    meta, rows = _parse(name)
    K = meta["K"]
    rng = np.random.default_rng(5)
    state = np.array([[meta["START"], -1, 0, 0]], np.int32)
    for tok in rows:
        t = int(tok[0])
        assert state[0, 0] == t
        lg, bias = _frame_logits(rng, K, t, meta)
        codes, done = orc.delay_step(K, VC, BOS, EOC, lg, bias, state)
        want = []
        for k, c in enumerate(tok[1:1 + K]):
            want.append({"a": _argmax_code(k, t), "B": BOS, "E": EOC}[c])
        assert codes[0].tolist() == want, f"frame {t}"
        assert state[0, 1] == int(tok[1 + K]), f"eoc frame at {t}"
        assert done[0] == int(tok[2 + K]) == state[0, 2], f"done at {t}"
        assert state[0, 0] == t + 1


def _run(orc, K, t0, inject, frames):
    """inject: dict frame -> list of codebooks whose EOC logit wins at that frame."""
    rng = np.random.default_rng(t0 * 131 + len(inject))
    state = np.array([[t0, -1, 0, 0]], np.int32)
    hist = []
    for t in range(t0, t0 + frames):
        lg = rng.normal(0.0, 0.1, size=(1, K, VC)).astype(np.float32)
        for k in range(K):
            lg[0, k, _argmax_code(k, t)] = 5.0
        for k in inject.get(t, []):
            lg[0, k, EOC] = 20.0
        codes, done = orc.delay_step(K, VC, BOS, EOC, lg, None, state)
        hist.append((t, codes[0].copy(), int(state[0, 1]), int(done[0])))
    return hist


def test_exhaustive_k4(orc):
    """Every start frame t0 <= 12 and every single injection (frame, codebook) for K = 4."""
    K = 4
    for t0 in range(0, 13):
        for f in range(t0, t0 + 8):
            for kin in range(K):
                hist = _run(orc, K, t0, {f: [kin]}, 14)
                # expected end frame: only if codebook kin is active and not forced at frame f
                e_exp = f - kin if f >= kin else -1
                for (t, codes, e, done) in hist:
                    for k in range(K):
                        if t < k:
                            assert codes[k] == BOS
                        elif e_exp >= 0 and t >= f and t - k >= e_exp:
                            assert codes[k] == EOC
                        else:
                            assert codes[k] == _argmax_code(k, t)
                    assert e == (e_exp if (e_exp >= 0 and t >= f) else -1)
                    assert done == int(e_exp >= 0 and t >= f and t >= e_exp + K - 1)


def test_argmax_ties_and_bos(orc):
    K = 2
    lg = np.zeros((1, K, VC), np.float32)
    lg[0, 0, [7, 9, 700]] = 3.0          # tie: lowest index wins
    lg[0, 1, BOS] = 4.0                  # BOS may be chosen in an active slot (no masking)
    state = np.array([[5, -1, 0, 0]], np.int32)
    codes, _ = orc.delay_step(K, VC, BOS, EOC, lg, None, state)
    assert codes[0].tolist() == [7, BOS]


def test_eoc_bias_is_added_to_eoc_logit_only(orc):
    K = 2
    lg = np.zeros((2, K, VC), np.float32)
    lg[:, :, 3] = 1.0
    lg[:, :, EOC] = 0.5
    bias = np.array([[0.6, 0.4], [0.0, 0.0]], np.float32)   # row 0 cb0: 1.1 > 1.0 -> EOC
    state = np.array([[4, -1, 0, 0], [4, -1, 0, 0]], np.int32)
    codes, _ = orc.delay_step(K, VC, BOS, EOC, lg, bias, state)
    assert codes.tolist() == [[EOC, 3], [3, 3]]            # row 0: e = 4; cb1 has 4 - 1 < 4
    assert state[0, 1] == 4 and state[1, 1] == -1


def test_code_embed_sum_closed_form(orc):
    """One-hot tables: the sum picks exactly the coded rows; fp32 sum of K values, ascending k."""
    K, H = 4, 64
    tab = np.zeros((K, VC, H), np.float32)
    for k in range(K):
        for v in range(VC):
            tab[k, v, (v + k) % H] = 2.0 ** (k - 2)        # exact in bf16
    codes = np.array([[5, 5, 1023, EOC], [0, BOS, 3, 3]], np.int32)
    out = orc.bf16_value(orc.code_embed_sum(orc.bf16_bits(tab), codes))
    want = np.zeros((2, H), np.float32)
    for b in range(2):
        for k in range(K):
            want[b, (codes[b, k] + k) % H] += 2.0 ** (k - 2)
    np.testing.assert_array_equal(out, want)


def test_code_embed_sum_rounding_once(orc):
    """Sum of values that are not representable together in bf16 rounds once at the end."""
    K, H = 3, 8
    vals = np.array([1.0, 2.0 ** -8, 2.0 ** -8], np.float32)   # 1 + 2^-7: exact in bf16
    tab = np.zeros((K, VC, H), np.float32)
    for k in range(K):
        tab[k, 0, :] = vals[k]
    out = orc.bf16_value(orc.code_embed_sum(orc.bf16_bits(tab), np.zeros((1, K), np.int32)))
    # rounding after each add would give 1.0 (1 + 2^-8 is a tie to even -> 1.0, twice)
    assert np.all(out == np.float32(1.0 + 2.0 ** -7))


def test_codebook_step_logits_brute_force(orc):
    from workloads import tiny_dims
    d = tiny_dims()
    rng = np.random.default_rng(1)
    B, K, H = 3, d.n_codebooks, d.hidden
    hid = orc.bf16_bits(rng.normal(0, 1, (B, H)).astype(np.float32))
    head = orc.bf16_bits(rng.normal(0, 0.02, (K * VC, H)).astype(np.float32))
    tab = orc.bf16_bits(rng.normal(0, 0.02, (K, VC, H)).astype(np.float32))
    state = np.array([[0, -1, 0, 0], [2, -1, 0, 0], [9, 4, 0, 0]], np.int32)
    codes, nxt, done, logits = orc.codebook_step(d, hid, head, tab, state)
    x64 = orc.bf16_value(hid).astype(np.float64)
    w64 = orc.bf16_value(head).astype(np.float64)
    ref = (x64 @ w64.T).reshape(B, K, VC)
    bound = H * 2.0 ** -24 * (np.abs(x64) @ np.abs(w64).T).reshape(B, K, VC)
    assert np.all(np.abs(logits - ref) <= bound + 1e-30)
    # row 2 has e = 4 at t = 9 >= 4 + K - 1: done, all EOC
    assert codes[2].tolist() == [EOC] * K and done[2] == 1
    # row 0 at t = 0: only codebook 0 active
    assert codes[0, 1:].tolist() == [BOS] * (K - 1)
    assert codes[0, 0] == int(np.argmax(logits[0, 0]))
