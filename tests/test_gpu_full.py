"""GPU parity at the full-width workload sizes, in the launch configuration the benchmark times.

- 36-layer backbone, 32 ragged prompts (lengths 16..256), 2048-slot cache: the oracle recomputes
  the two shortest sequences end to end (every layer's K/V and the last hidden); every sequence's
  unused cache slots must stay untouched.
- long prompts (8 x 1024..2048, 4096-slot cache): the oracle recomputes the first two layers of the
  shortest sequence at every position (multi-tile causal attention); all 36 layers' slots past each
  length stay untouched, and the default last-layer path agrees with the full last layer."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from parity import assert_close, assert_parity, ref_np, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def hra():
    import qwen3_prefill_delayed_gb300 as h
    h.lib()
    return h


def _sub_weights(w, n_layers):
    return {"embed": w["embed"], "final_norm": w["final_norm"], "layers": w["layers"][:n_layers]}


def _untouched(cache, lens):
    for b, n in enumerate(lens):
        assert bool(torch.isnan(cache[:, b, :, :, n:]).all()), f"seq {b}: slots past its length were written"


def test_ragged_batch_36_layers(hra):
    wl = W.ragged_batch(DEV)
    d, p, w = wl["dims"], wl["prompts"], wl["weights"]
    bb = hra.Backbone(d, w)
    cache = hra.new_kv_cache(d, len(p.lengths), wl["n_slots"], DEV, fill=float("nan"))
    hid = bb.prefill(p.tokens.to(DEV), p.lengths, cache)
    assert hra.hra_device_error(bb.last_ws) == 0
    _untouched(cache, p.lengths)
    idx = sorted(range(len(p.lengths)), key=lambda b: p.lengths[b])[:2]
    lens = [p.lengths[b] for b in idx]
    hw = oracle.host_weights_from(d, w)
    tok = p.tokens[idx].numpy()
    kv_o, hid_o = oracle.prefill(d, hw, tok, lens, max(lens))
    with oracle.sum_order(True):
        kv_a, hid_a = oracle.prefill(d, hw, tok, lens, max(lens))
    for j, b in enumerate(idx):
        assert_parity(to_np(hid[b]), ref_np(hid_o[j]), ref_np(hid_a[j]), what=f"last hidden seq {b}")
        got = cache[:, b, :, :, :lens[j]].float().cpu().numpy().astype(np.float64)
        for l in range(d.n_layers):
            assert_parity(got[l], ref_np(kv_o[l, j, :, :, :lens[j]]), ref_np(kv_a[l, j, :, :, :lens[j]]),
                          what=f"kv seq {b} layer {l}")
    # full last layer gives the same last hidden
    hid_full = bb.prefill(p.tokens.to(DEV), p.lengths, cache, full_last_layer=True)
    # two GPU code paths for the last layer (all rows vs the last rows only): one layer of
    # summation-order spread, at most 2 bf16 ulps of the largest magnitudes
    assert_close(to_np(hid_full), to_np(hid), what="full last layer vs last rows", max_abs=0.0625, min_cos=0.99999)


def test_long_prompts_two_layers_and_cache(hra):
    wl = W.long_prompts(DEV)
    d, p, w = wl["dims"], wl["prompts"], wl["weights"]
    bb = hra.Backbone(d, w)
    cache = hra.new_kv_cache(d, len(p.lengths), wl["n_slots"], DEV, fill=float("nan"))
    hid = bb.prefill(p.tokens.to(DEV), p.lengths, cache)
    assert hra.hra_device_error(bb.last_ws) == 0
    assert torch.isfinite(hid.float()).all()
    _untouched(cache, p.lengths)
    b = min(range(len(p.lengths)), key=lambda i: p.lengths[i])
    n = p.lengths[b]
    d2 = W.Dims(**{**d.__dict__, "n_layers": 2})
    hw = oracle.host_weights_from(d2, _sub_weights(w, 2))
    tok = p.tokens[b:b + 1, :n].numpy()
    kv_o, _ = oracle.prefill(d2, hw, tok, [n], n)
    with oracle.sum_order(True):
        kv_a, _ = oracle.prefill(d2, hw, tok, [n], n)
    got = cache[:2, b, :, :, :n].float().cpu().numpy().astype(np.float64)
    for l in range(2):
        assert_parity(got[l], ref_np(kv_o[l, 0]), ref_np(kv_a[l, 0]), what=f"layer {l} kv of seq {b} (len {n})")
    hid_full = bb.prefill(p.tokens.to(DEV), p.lengths, cache, full_last_layer=True)
    # two GPU code paths for the last layer (all rows vs the last rows only): one layer of
    # summation-order spread, at most 2 bf16 ulps of the largest magnitudes
    assert_close(to_np(hid_full), to_np(hid), what="full last layer vs last rows", max_abs=0.0625, min_cos=0.99999)
