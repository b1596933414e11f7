"""GPU parity of the persistent decoder pass (one cooperative kernel over every layer for at most 64
rows) against the oracle, next to the layer-by-layer kernels on the same inputs.

Cases: one full-width layer at 1, 33 and 64 rows over long cached prefixes (attention key splits
and their merge, both TMEM lane quarters, every projection tile), four full-width layers at 8 rows
(the weight stream across layers), and the tiny model (head_dim 64, GQA group 2) through prefill
and decode.  The cache prefix is seeded N(0, 1) data written straight into both caches."""
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


def _host(w):
    return {"embed": w["embed"].cpu(), "final_norm": w["final_norm"].cpu(),
            "layers": [{k: v.cpu() for k, v in l.items()} for l in w["layers"]]}


def _decode_both_paths(hra, d, bb, hw, B, n_slots, pos, seed, what, tier="layer"):
    """Random cache prefix + one decode pass of B rows at positions `pos`, through the persistent
    pass and through the layer-by-layer kernels, each against the oracle (both summation orders)."""
    g = torch.Generator().manual_seed(seed)
    prefix = torch.randn(d.n_layers, B, 2, d.n_kv_heads, n_slots, d.head_dim, generator=g).to(torch.bfloat16)
    emb = (torch.randn(B, d.hidden, generator=g) * 0.5).to(torch.bfloat16)
    kv_o = W.to_u16(prefix).copy()
    kv_a = kv_o.copy()
    hid_o = oracle.decode(d, hw, W.to_u16(emb), pos, kv_o, n_slots)
    with oracle.sum_order(True):
        hid_a = oracle.decode(d, hw, W.to_u16(emb), pos, kv_a, n_slots)
    results = {}
    for persistent in (True, False):
        prev = hra.hra_set_decode_pass(persistent)
        try:
            cache = prefix.to(DEV)
            hid = bb.decode(emb.to(DEV), pos, cache)
            torch.cuda.synchronize()
        finally:
            hra.hra_set_decode_pass(prev)
        tag = f"{what} [{'persistent' if persistent else 'layered'}]"
        assert_parity(to_np(hid), ref_np(hid_o), ref_np(hid_a), what=f"{tag} hidden", tier=tier)
        c = cache.float().cpu().numpy()
        for l in range(d.n_layers):
            for b in range(B):
                p = pos[b]
                # the new K/V slot of every row, and the untouched prefix around it
                assert_parity(c[l, b, :, :, p].astype(np.float64), ref_np(kv_o[l, b, :, :, p]),
                              ref_np(kv_a[l, b, :, :, p]), what=f"{tag} kv layer {l} row {b}",
                              tier="layer" if l == 0 else tier)
        pre = prefix.float().numpy()
        for b in range(B):
            np.testing.assert_array_equal(np.delete(c[:, b], pos[b], axis=-2), np.delete(pre[:, b], pos[b], axis=-2),
                                          err_msg=f"{tag}: a cache slot other than the row's position changed")
        results[persistent] = to_np(hid)
    return results


@pytest.fixture(scope="module")
def single(hra):
    wl = W.single_layer(13, "cpu")
    d = wl["dims"]
    wl["bb"] = hra.Backbone(d, _dev(wl["weights"]))
    wl["hw"] = oracle.host_weights_from(d, wl["weights"])
    return wl


@pytest.mark.parametrize("B", [1, 33, 64])
def test_full_width_layer_long_prefix(hra, single, B):
    d = single["dims"]
    n_slots = 2048
    pos = [(b * 613 + 37) % 1990 + 3 for b in range(B)]
    pos[0] = 1999           # the longest row: several key splits
    _decode_both_paths(hra, d, single["bb"], single["hw"], B, n_slots, pos, seed=40 + B, what=f"B={B}")


def test_four_full_width_layers(hra):
    d = W.full_dims(4)
    g = W._gen(44, DEV)
    w = W.make_backbone(d, 44, DEV, gen=g)
    w.pop("_gen", None)
    bb = hra.Backbone(d, _dev(w))
    hw = oracle.host_weights_from(d, _host(w))
    pos = [700, 1, 1500, 64, 129, 1023, 5, 300]
    _decode_both_paths(hra, d, bb, hw, 8, 1536, pos, seed=45, what="4 layers", tier="deep")


def test_tiny_prefill_and_decode_through_the_pass(hra):
    """Tiny model (head_dim 64, GQA 2): a ragged prefill of 28 rows and two decode passes, persistent
    and layered, each against the oracle."""
    wl = W.tiny_reference("cpu")
    d = wl["dims"]
    bb = hra.Backbone(d, _dev(wl["weights"]))
    hw = oracle.host_weights_from(d, wl["weights"])
    lens = [13, 5, 9, 1]
    pr = W.make_prompts(21, len(lens), 13, 13, d.vocab, fixed_len=13)
    tok = torch.full((len(lens), 13), 0, dtype=torch.int32)
    for b, n in enumerate(lens):
        tok[b, :n] = pr.tokens[b, :n]
    (kv_o, last_o) = oracle.prefill(d, hw, tok.numpy(), lens, 32)
    with oracle.sum_order(True):
        (kv_a, last_a) = oracle.prefill(d, hw, tok.numpy(), lens, 32)
    g = torch.Generator().manual_seed(22)
    embs = [(torch.randn(len(lens), d.hidden, generator=g) * 0.5).to(torch.bfloat16) for _ in range(2)]
    hids_o, hids_a = [], []
    for s, emb in enumerate(embs):
        p = [n + s for n in lens]
        hids_o.append(oracle.decode(d, hw, W.to_u16(emb), p, kv_o, 32))
        with oracle.sum_order(True):
            hids_a.append(oracle.decode(d, hw, W.to_u16(emb), p, kv_a, 32))
    for persistent in (True, False):
        prev = hra.hra_set_decode_pass(persistent)
        try:
            cache = hra.new_kv_cache(d, len(lens), 32, DEV, fill=float("nan"))
            last = bb.prefill(tok.to(DEV), lens, cache)
            tag = "persistent" if persistent else "layered"
            assert_parity(to_np(last), ref_np(last_o), ref_np(last_a), what=f"tiny prefill [{tag}]")
            for s, emb in enumerate(embs):
                hid = bb.decode(emb.to(DEV), [n + s for n in lens], cache)
                assert_parity(to_np(hid), ref_np(hids_o[s]), ref_np(hids_a[s]), what=f"tiny decode {s} [{tag}]")
            c = cache.float().cpu().numpy()
            for b, n in enumerate(lens):
                assert_parity(c[:, b, :, :, :n + 2].astype(np.float64), ref_np(kv_o[:, b, :, :, :n + 2]),
                              ref_np(kv_a[:, b, :, :, :n + 2]), what=f"tiny kv seq {b} [{tag}]")
                assert np.all(np.isnan(c[:, b, :, :, n + 2:])), "slots past the last position were written"
        finally:
            hra.hra_set_decode_pass(prev)
