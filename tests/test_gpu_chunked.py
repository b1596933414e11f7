"""GPU parity of hra_prefill_chunk (one chunk per sequence after the positions already in the
cache) against the oracle's whole-sequence prefill.

- tiny 2-layer model: a batch mixing a first chunk (start 0), a single-token step and a chunk after
  cached positions, on a cache that hra_prefill filled; last hidden and every written slot;
- full-width 2 layers: chunks starting at 300 and 77 (not multiples of the 64-key tile), so the
  causal diagonal of the chunk straddles key tiles of cached and new positions;
- a full-width mixed batch of single-token steps and chunks in one launch;
- a chunk that ends in the last cache slot, and starts that run past the cache (refused before any
  launch);
- every GQA group size the attention kernel takes at both head dims (G = 1: 128 positions per query
  tile; G = 8: 16 positions), with prompts spanning several query tiles and a chunk after cached
  positions."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from parity import assert_parity, ref_np, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def hra():
    import qwen3_prefill_delayed_gb300 as h
    h.lib()
    return h


def _dev(w):
    return {"embed": w["embed"].to(DEV), "final_norm": w["final_norm"].to(DEV),
            "layers": [{k: v.to(DEV) for k, v in l.items()} for l in w["layers"]]}


def _tokens(seed, lens, vocab):
    g = np.random.default_rng(seed)
    t = np.zeros((len(lens), max(lens)), np.int32)
    for b, n in enumerate(lens):
        t[b, :n] = g.integers(0, vocab, n)
    return t


def _pack(rows, vocab, width=None):
    width = width or max(len(r) for r in rows)
    t = np.full((len(rows), width), vocab + 3, np.int32)   # trailing pads: out-of-range ids, never read
    for b, r in enumerate(rows):
        t[b, :len(r)] = r
    return torch.from_numpy(t)


def _run_chunks(hra, d, w, tok, lens, cut, n_new, n_slots, full_last=False):
    """GPU: hra_prefill of each sequence's first cut[b] tokens (where cut[b] > 0), then one
    hra_prefill_chunk call with n_new[b] tokens at positions cut[b].. for every sequence."""
    bb = hra.Backbone(d, _dev(w))
    B = len(lens)
    cache = hra.new_kv_cache(d, B, n_slots, DEV, fill=float("nan"))
    pre = [b for b in range(B) if cut[b] > 0]
    if pre:
        sub = hra.new_kv_cache(d, len(pre), n_slots, DEV, fill=float("nan"))
        bb.prefill(_pack([tok[b, :cut[b]] for b in pre], d.vocab).to(DEV), [cut[b] for b in pre], sub)
        for j, b in enumerate(pre):
            cache[:, b] = sub[:, j]
    chunk = _pack([tok[b, cut[b]:cut[b] + n_new[b]] for b in range(B)], d.vocab).to(DEV)
    hid = bb.prefill(chunk, n_new, cache, start_pos=cut, full_last_layer=full_last)
    assert hra.hra_device_error(bb.last_ws) == 0
    return hid, cache


def _check(d, w, tok, cut, n_new, hid, cache, n_slots, tier="deep"):
    hw = oracle.host_weights_from(d, w)
    ends = [c + n for c, n in zip(cut, n_new)]
    t_o = tok[:, :max(ends)].copy()
    kv_o, hid_o = oracle.prefill(d, hw, t_o, ends, n_slots)
    with oracle.sum_order(True):
        kv_a, hid_a = oracle.prefill(d, hw, t_o, ends, n_slots)
    got = cache.float().cpu().numpy()
    assert_parity(to_np(hid), ref_np(hid_o), ref_np(hid_a), what="last hidden", tier=tier)
    for b, e in enumerate(ends):
        assert_parity(got[:, b, :, :, :e].astype(np.float64), ref_np(kv_o[:, b, :, :, :e]),
                      ref_np(kv_a[:, b, :, :, :e]), what=f"kv seq {b}", tier=tier)
        assert np.all(np.isnan(got[:, b, :, :, e:])), f"seq {b}: slots past position {e - 1} were written"


@pytest.mark.parametrize("full_last", [False, True])
def test_tiny_mixed_chunks(hra, full_last):
    d = W.tiny_dims()
    w = W.make_backbone(d, 0, "cpu")
    lens = [13, 10, 12, 7]
    tok = _tokens(5, lens, d.vocab)
    cut = [0, 9, 5, 6]
    n_new = [13, 1, 7, 1]
    hid, cache = _run_chunks(hra, d, w, tok, lens, cut, n_new, 32, full_last)
    _check(d, w, tok, cut, n_new, hid, cache, 32, tier="layer")


def test_full_width_chunks_straddle_tiles(hra):
    d = W.full_dims(2)
    w = W.make_backbone(d, 11, "cpu")
    lens = [500, 227]
    tok = _tokens(6, lens, d.vocab)
    cut = [300, 77]
    n_new = [200, 150]
    hid, cache = _run_chunks(hra, d, w, tok, lens, cut, n_new, 512)
    _check(d, w, tok, cut, n_new, hid, cache, 512)


def test_full_width_mixed_steps_and_chunks(hra):
    d = W.full_dims(2)
    w = W.make_backbone(d, 12, "cpu")
    lens = [40, 131, 64, 90, 5]
    tok = _tokens(7, lens, d.vocab)
    cut = [39, 60, 0, 89, 4]
    n_new = [1, 71, 64, 1, 1]
    hid, cache = _run_chunks(hra, d, w, tok, lens, cut, n_new, 256)
    _check(d, w, tok, cut, n_new, hid, cache, 256)


def test_chunk_to_the_last_slot_and_range_errors(hra):
    d = W.tiny_dims()
    w = W.make_backbone(d, 0, "cpu")
    lens = [32, 20]
    tok = _tokens(8, lens, d.vocab)
    cut = [25, 0]
    n_new = [7, 20]                      # sequence 0 ends in slot 31 of 32
    hid, cache = _run_chunks(hra, d, w, tok, lens, cut, n_new, 32)
    _check(d, w, tok, cut, n_new, hid, cache, 32, tier="layer")
    bb = hra.Backbone(d, _dev(w))
    chunk = _pack([tok[0, :7], tok[1, :7]], d.vocab).to(DEV)
    with pytest.raises(hra.HraError, match="outside the cache"):
        bb.prefill(chunk, [7, 7], cache, start_pos=[26, 0])
    with pytest.raises(hra.HraError, match="outside the cache"):
        bb.prefill(chunk, [7, 7], cache, start_pos=[0, -1])


@pytest.mark.parametrize("nq,nkv,hd", [(8, 8, 64), (4, 4, 128), (16, 2, 64), (8, 1, 128)])
def test_gqa_group_sizes(hra, nq, nkv, hd):
    d = W.Dims(n_layers=2, hidden=256, n_q_heads=nq, n_kv_heads=nkv, head_dim=hd, ffn=256, vocab=512,
               n_codebooks=4)
    w = W.make_backbone(d, 13, "cpu")
    lens = [300, 129, 17]
    tok = _tokens(9, lens, d.vocab)
    cut = [0, 100, 0]
    n_new = [300, 29, 17]
    hid, cache = _run_chunks(hra, d, w, tok, lens, cut, n_new, 320)
    _check(d, w, tok, cut, n_new, hid, cache, 320)
