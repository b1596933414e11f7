"""GPU parity of the single-query attention of hra_decode against the oracle, over the shapes its
kernel is specialised for (head_dim 64 / 128; 1, 2, 4 or 8 q heads per kv head) and over key
counts that land on every tile and split boundary.

The cache is filled with seeded N(0, 1) keys and values below each row's position and NaN above
it, so a read past the used keys would poison the output.  One decode layer then runs at those
positions; the oracle runs the same layer on the same cache.  Rows are independent sequences, so
one call mixes a single key (position 0), partial and full 64-key tiles, and 2048 keys spread over
many splits (some of them empty)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from parity import assert_parity, ref_np, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"
N_SLOTS = 2048
POSITIONS = [0, 1, 15, 63, 64, 65, 127, 128, 129, 200, 1000, 1500, 2047]


@pytest.fixture(scope="module")
def hra():
    import qwen3_prefill_delayed_gb300 as h
    h.lib()
    return h


def _dev(w):
    return {"embed": w["embed"].to(DEV), "final_norm": w["final_norm"].to(DEV),
            "layers": [{k: v.to(DEV) for k, v in l.items()} for l in w["layers"]]}


def _run(hra, d, positions, seed):
    w = W.make_backbone(d, seed, "cpu")
    hw = oracle.host_weights_from(d, w)
    bb = hra.Backbone(d, _dev(w))
    B = len(positions)
    g = torch.Generator().manual_seed(seed + 7)
    cache = torch.randn(1, B, 2, d.n_kv_heads, N_SLOTS, d.head_dim, generator=g).to(torch.bfloat16)
    for b, p in enumerate(positions):
        cache[:, b, :, :, p:] = float("nan")   # slot p is written by the pass; slots past it are never read
    emb = (torch.randn(B, d.hidden, generator=g) * 0.5).to(torch.bfloat16)
    cache_dev = cache.to(DEV)
    hid = bb.decode(emb.to(DEV), positions, cache_dev)
    assert hra.hra_device_error(bb.last_ws) == 0
    kv_o = W.to_u16(cache).copy()
    kv_a = kv_o.copy()
    hid_o = oracle.decode(d, hw, W.to_u16(emb), positions, kv_o, N_SLOTS)
    with oracle.sum_order(True):
        hid_a = oracle.decode(d, hw, W.to_u16(emb), positions, kv_a, N_SLOTS)
    assert_parity(to_np(hid), ref_np(hid_o), ref_np(hid_a), what="decode hidden")
    got = cache_dev.float().cpu().numpy()
    for b, p in enumerate(positions):
        assert_parity(got[0, b, :, :, p].astype(np.float64), ref_np(kv_o[0, b, :, :, p]),
                      ref_np(kv_a[0, b, :, :, p]), what=f"kv written at slot {p}")
        assert np.all(np.isnan(got[0, b, :, :, p + 1:])), f"row {b}: slots past position {p} were written"


@pytest.mark.parametrize("hd,nq,nkv", [(64, 2, 2), (64, 4, 2), (128, 8, 2), (64, 8, 1), (128, 32, 8)])
def test_decode_attention_boundaries(hra, hd, nq, nkv):
    d = W.Dims(n_layers=1, hidden=256, n_q_heads=nq, n_kv_heads=nkv, head_dim=hd, ffn=512, vocab=64)
    _run(hra, d, POSITIONS, seed=100 + hd + nq + nkv)


def test_decode_attention_one_split_long_rows(hra):
    """40 rows x 8 kv heads fill a wave of CTAs, so each row takes one split and its CTA walks up to
    32 key tiles through the stage ring."""
    d = W.Dims(n_layers=1, hidden=256, n_q_heads=32, n_kv_heads=8, head_dim=128, ffn=512, vocab=64)
    positions = [(37 * b * b + 11 * b) % N_SLOTS for b in range(39)] + [N_SLOTS - 1]
    _run(hra, d, positions, seed=321)
