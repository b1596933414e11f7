"""Model-level pins of the oracle on the tiny 2-layer shape: structural invariants (batch and
ragged invariance, pad independence, causality, untouched cache slots), decode == prefill of one
more token, and closed forms reached by zeroing or selecting weight blocks (residual stream,
uniform attention, SwiGLU MLP) checked against float64 brute force."""
import numpy as np
import pytest
import torch

import workloads as W

U = 2.0 ** -8


@pytest.fixture(scope="module")
def tiny(orc):
    d = W.tiny_dims()
    w = W.make_backbone(d, 0, "cpu")
    hw = orc.host_weights_from(d, w)
    return d, w, hw


def _tokens(rng, lens, vocab, pmax=None, pad=0):
    pmax = pmax or max(lens)
    t = np.full((len(lens), pmax), pad, np.int32)
    for b, n in enumerate(lens):
        t[b, :n] = rng.integers(0, vocab, n)
    return t


def _val(orc, u):
    return orc.bf16_value(u).astype(np.float64)


def test_batch_and_pad_invariance(orc, tiny):
    d, _, hw = tiny
    rng = np.random.default_rng(0)
    lens = [13, 5, 9]
    tok = _tokens(rng, lens, d.vocab)
    kv, last = orc.prefill(d, hw, tok, lens, 32)
    for b in range(3):
        # alone, with extra trailing pads holding out-of-range ids (never read)
        t1 = np.full((1, 20), d.vocab + 99, np.int32)
        t1[0, :lens[b]] = tok[b, :lens[b]]
        kv1, last1 = orc.prefill(d, hw, t1, [lens[b]], 32)
        np.testing.assert_array_equal(last1[0], last[b])
        np.testing.assert_array_equal(kv1[:, 0], kv[:, b])


def test_unused_slots_untouched_and_causality(orc, tiny):
    d, _, hw = tiny
    rng = np.random.default_rng(1)
    lens = [11]
    tok = _tokens(rng, lens, d.vocab)
    poison = np.full(orc.kv_shape(d, 1, 32), 0x7fc1, np.uint16)
    kv, _ = orc.prefill(d, hw, tok, lens, 32, kv=poison.copy())
    assert np.all(kv[..., 11:, :] == 0x7fc1)
    assert not np.any(kv[..., :11, :] == 0x7fc1)
    tok2 = tok.copy()
    tok2[0, 7:] = (tok2[0, 7:] + 1) % d.vocab
    kv2, _ = orc.prefill(d, hw, tok2, lens, 32)
    np.testing.assert_array_equal(kv2[..., :7, :], kv[..., :7, :])
    assert np.any(kv2[..., 7:11, :] != kv[..., 7:11, :])


def test_decode_extends_prefill(orc, tiny):
    """Prefill of n tokens, then a decode pass fed E[tok_n] at position n, equals prefill of n+1."""
    d, w, hw = tiny
    rng = np.random.default_rng(2)
    tok = _tokens(rng, [9], d.vocab)
    kv_a, _ = orc.prefill(d, hw, tok[:, :8], [8], 32)
    emb = hw.embed[tok[0, 8]][None, :]
    hid = orc.decode(d, hw, emb, [8], kv_a, 32)
    kv_b, last_b = orc.prefill(d, hw, tok, [9], 32)
    np.testing.assert_array_equal(hid, last_b)
    np.testing.assert_array_equal(kv_a, kv_b)


def test_chunked_prefill_equals_whole(orc, tiny):
    """A batch mixing a first chunk (start 0), a single-token step and a multi-token chunk after
    cached positions reproduces, bit for bit, the prefill of each whole sequence."""
    d, _, hw = tiny
    rng = np.random.default_rng(5)
    lens = [13, 10, 12]
    tok = _tokens(rng, lens, d.vocab)
    kv_w, last_w = orc.prefill(d, hw, tok, lens, 32)
    cut = [0, 9, 5]                      # positions already in the cache before the chunk
    kv = np.full(orc.kv_shape(d, 3, 32), 0x7fc1, np.uint16)
    first = list(cut)
    pre = [b for b in range(3) if first[b] > 0]
    t_pre = np.zeros((len(pre), max(first)), np.int32)
    for j, b in enumerate(pre):
        t_pre[j, :first[b]] = tok[b, :first[b]]
    kv_pre, _ = orc.prefill(d, hw, t_pre, [first[b] for b in pre], 32)
    for j, b in enumerate(pre):
        kv[:, b, :, :, :first[b]] = kv_pre[:, j, :, :, :first[b]]
    before = kv.copy()
    n_new = [lens[b] - cut[b] for b in range(3)]
    n_new[1] = 1                          # sequence 1 takes one token (a decode-like step)
    t_new = np.full((3, max(n_new)), d.vocab + 5, np.int32)   # trailing pads: out-of-range ids, never read
    for b in range(3):
        t_new[b, :n_new[b]] = tok[b, cut[b]:cut[b] + n_new[b]]
    last = orc.prefill_chunk(d, hw, t_new, n_new, cut, kv, 32)
    for b in (0, 2):
        np.testing.assert_array_equal(last[b], last_w[b])
        np.testing.assert_array_equal(kv[:, b, :, :, :lens[b]], kv_w[:, b, :, :, :lens[b]])
    # sequence 1 stopped after cut + 1 positions: equal to the whole prefill of that prefix
    kv_1, last_1 = orc.prefill(d, hw, tok[1:2, :cut[1] + 1], [cut[1] + 1], 32)
    np.testing.assert_array_equal(last[1], last_1[0])
    np.testing.assert_array_equal(kv[:, 1, :, :, :cut[1] + 1], kv_1[:, 0, :, :, :cut[1] + 1])
    # cached slots are read only; slots past each chunk stay untouched
    for b in range(3):
        np.testing.assert_array_equal(kv[:, b, :, :, :cut[b]], before[:, b, :, :, :cut[b]])
        assert np.all(kv[:, b, :, :, cut[b] + n_new[b]:] == 0x7fc1)


def test_chunk_reads_the_cached_prefix(orc, tiny):
    """The chunk attends the cached keys: perturbing one cached key changes its output, perturbing
    a slot past the chunk does not; a start that runs past the cache is rejected."""
    d, _, hw = tiny
    rng = np.random.default_rng(6)
    tok = _tokens(rng, [10], d.vocab)
    kv0, _ = orc.prefill(d, hw, tok[:, :6], [6], 32)
    base = orc.prefill_chunk(d, hw, tok[:, 6:], [4], [6], kv0.copy(), 32)
    kv1 = kv0.copy()
    kv1[0, 0, 0, 0, 3, :] ^= 0x0040              # key of position 3, layer 0, kv head 0
    moved = orc.prefill_chunk(d, hw, tok[:, 6:], [4], [6], kv1, 32)
    assert np.any(moved != base)
    kv2 = kv0.copy()
    kv2[..., 20, :] = 0x7fc1                     # a slot no position of the chunk reaches
    same = orc.prefill_chunk(d, hw, tok[:, 6:], [4], [6], kv2, 32)
    np.testing.assert_array_equal(same, base)
    with pytest.raises(ValueError):
        orc.prefill_chunk(d, hw, tok[:, 6:], [4], [29], kv0.copy(), 32)


def _one_layer(d, w, **override):
    d1 = W.Dims(**{**d.__dict__, "n_layers": 1})
    lay = {k: v.clone() for k, v in w["layers"][0].items()}
    lay.update(override)
    return d1, {"embed": w["embed"], "layers": [lay], "final_norm": w["final_norm"]}


def test_zero_branches_leave_residual(orc, tiny):
    d, w, _ = tiny
    H = d.hidden
    wz = {"embed": w["embed"], "final_norm": w["final_norm"],
          "layers": [{**l, "w_o": torch.zeros_like(l["w_o"]), "w_down": torch.zeros_like(l["w_down"])}
                     for l in w["layers"]]}
    hw = orc.host_weights_from(d, wz)
    rng = np.random.default_rng(3)
    tok = _tokens(rng, [6, 4], d.vocab)
    _, last = orc.prefill(d, hw, tok, [6, 4], 16)
    for b, n in enumerate([6, 4]):
        e = hw.embed[tok[b, n - 1]][None, :]
        np.testing.assert_array_equal(last[b], orc.rmsnorm(e, hw.final_norm, d.rms_eps)[0])


def _rms64(x, g, eps):
    return x / np.sqrt(np.mean(x ** 2, axis=-1, keepdims=True) + eps) * g


def test_uniform_attention_closed_form(orc, tiny):
    """W_q = 0 makes every score 0, so attention returns the running mean of V; W_o selects it back
    into the residual; W_down = 0.  Checked against float64 brute force."""
    d, w, _ = tiny
    H, hd, nq, nkv = d.hidden, d.head_dim, d.n_q_heads, d.n_kv_heads
    assert nq * hd == H
    wqkv = w["layers"][0]["w_qkv"].clone()
    wqkv[:nq * hd] = 0
    d1, w1 = _one_layer(d, w, w_qkv=wqkv, w_o=torch.eye(H, dtype=torch.bfloat16),
                        w_down=torch.zeros(H, d.ffn, dtype=torch.bfloat16))
    hw = orc.host_weights_from(d1, w1)
    rng = np.random.default_rng(4)
    n = 10
    tok = _tokens(rng, [n], d.vocab)
    _, last = orc.prefill(d1, hw, tok, [n], 16)
    E = _val(orc, hw.embed[tok[0]])
    y = _rms64(E, _val(orc, hw.layers[0]["attn_norm"]), d.rms_eps)
    wv = _val(orc, hw.layers[0]["w_qkv"])[(nq + nkv) * hd:]
    V = (y @ wv.T).reshape(n, nkv, hd)
    att = np.concatenate([V[:, h // (nq // nkv)].mean(0) for h in range(nq)])   # last query sees all n
    r = E[-1] + att
    ref = _rms64(r, _val(orc, hw.final_norm), d.rms_eps)
    got = _val(orc, last[0])
    assert np.max(np.abs(got - ref)) <= 6 * U * np.max(np.abs(ref))


def test_swiglu_closed_form(orc, tiny):
    """W_o = 0 and W_down selecting the first H of the F gated units: r = E + silu(g) * u."""
    d, w, _ = tiny
    H, F = d.hidden, d.ffn
    sel = torch.zeros(H, F, dtype=torch.bfloat16)
    sel[torch.arange(H), torch.arange(H)] = 1
    d1, w1 = _one_layer(d, w, w_o=torch.zeros(H, d.n_q_heads * d.head_dim, dtype=torch.bfloat16),
                        w_down=sel)
    hw = orc.host_weights_from(d1, w1)
    rng = np.random.default_rng(5)
    tok = _tokens(rng, [3], d.vocab)
    _, last = orc.prefill(d1, hw, tok, [3], 8)
    E = _val(orc, hw.embed[tok[0, 2]])
    y = _rms64(E, _val(orc, hw.layers[0]["mlp_norm"]), d.rms_eps)
    wgu = _val(orc, hw.layers[0]["w_gate_up"])
    g, u = y @ wgu[:F].T, y @ wgu[F:].T
    h = g / (1 + np.exp(-g)) * u
    ref = _rms64(E + h[:H], _val(orc, hw.final_norm), d.rms_eps)
    got = _val(orc, last[0])
    assert np.max(np.abs(got - ref)) <= 6 * U * np.max(np.abs(ref))
    # swapping gate and up (a plausible mistake) is far outside that bound
    h_sw = u / (1 + np.exp(-u)) * g
    bad = _rms64(E + h_sw[:H], _val(orc, hw.final_norm), d.rms_eps)
    assert np.max(np.abs(bad - ref)) > 20 * U * np.max(np.abs(ref))


def test_tiny_reference_ar_schedule(orc):
    """Tiny workload end to end: prefill, then 6 frames of codebook step + decode pass.  The EOC bias
    on codebook 0 at frame 2 stops the stream at frame 2 + K - 1 = 5 (no chance EOC earlier)."""
    wl = W.tiny_reference("cpu")
    d, p = wl["dims"], wl["prompts"]
    hw = orc.host_weights_from(d, wl["weights"])
    kv, hid = orc.prefill(d, hw, p.tokens.numpy(), p.lengths, wl["n_slots"])
    head, tab = W.to_u16(wl["audio"]["head_w"]), W.to_u16(wl["audio"]["code_emb"])
    state = np.array([[0, -1, 0, 0]], np.int32)
    K, BOS, EOC = d.n_codebooks, d.bos_id, d.eoc_id
    for t in range(wl["frames"]):
        codes, nxt, done, logits = orc.codebook_step(d, hid, head, tab, state, wl["eoc_bias"][t].numpy())
        for k in range(K):
            if t < k:
                assert codes[0, k] == BOS
            elif t - k >= 2:
                assert codes[0, k] == EOC
            else:
                assert codes[0, k] == int(np.argmax(logits[0, k])) != EOC
        assert done[0] == int(t == 5)
        assert state[0, 1] == (2 if t >= 2 else -1)
        hid = orc.decode(d, hw, nxt, [p.lengths[0] + t], kv, wl["n_slots"])
