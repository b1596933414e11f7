"""GPU parity at the full-width workload sizes, in the launch configuration the benchmark times.

- 36-layer backbone, 32 ragged prompts (lengths 16..256), 2048-slot cache: the oracle recomputes
  the two shortest sequences, the shortest one longer than 64 tokens (more than one attention
  key tile, so the heaviest-first schedule at depth) and the last one (its rows end the batch, in
  the last, partly empty 256-row tile of the projection GEMMs) end to end (every layer's K/V and
  the last hidden); every sequence's unused cache slots must stay untouched.
- the same backbone's autoregressive audio loop: the shortest prompt prefilled, then three K = 8
  frames (codebook step + 36-layer decode pass) captured in one CUDA graph, against the oracle's
  prefill + codebook step + decode chain: codes, stop flags and the delay state bit for bit (a
  disagreement is excused only at a near-tie of the oracle's logits), hidden and K/V at the
  deep-stack bar.
- long prompts (8 x 1024..2048, 4096-slot cache): the oracle recomputes the first two layers of the
  shortest sequence at every position (multi-tile causal attention); all 36 layers' slots past each
  length stay untouched, and the default last-layer path agrees with the full last layer."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from parity import ARGMAX_MARGIN, assert_close, assert_parity, ref_np, to_np

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


@pytest.fixture(scope="module")
def ragged(hra):
    wl = W.ragged_batch(DEV)
    d, w = wl["dims"], wl["weights"]
    wl["bb"] = hra.Backbone(d, w)
    wl["hw"] = oracle.host_weights_from(d, w)
    return wl


def test_ragged_batch_36_layers(hra, ragged):
    wl = ragged
    d, p, bb, hw = wl["dims"], wl["prompts"], wl["bb"], wl["hw"]
    cache = hra.new_kv_cache(d, len(p.lengths), wl["n_slots"], DEV, fill=float("nan"))
    hid = bb.prefill(p.tokens.to(DEV), p.lengths, cache)
    assert hra.hra_device_error(bb.last_ws) == 0
    _untouched(cache, p.lengths)
    order = sorted(range(len(p.lengths)), key=lambda b: p.lengths[b])
    longer = next(b for b in order if p.lengths[b] > 64)
    for idx in (order[:2], [longer], [len(p.lengths) - 1]):
        lens = [p.lengths[b] for b in idx]
        tok = p.tokens[idx].numpy()
        kv_o, hid_o = oracle.prefill(d, hw, tok, lens, max(lens))
        with oracle.sum_order(True):
            kv_a, hid_a = oracle.prefill(d, hw, tok, lens, max(lens))
        for j, b in enumerate(idx):
            assert_parity(to_np(hid[b]), ref_np(hid_o[j]), ref_np(hid_a[j]),
                          what=f"last hidden seq {b} (len {lens[j]})", tier="deep")
            got = cache[:, b, :, :, :lens[j]].float().cpu().numpy().astype(np.float64)
            for l in range(d.n_layers):
                assert_parity(got[l], ref_np(kv_o[l, j, :, :, :lens[j]]), ref_np(kv_a[l, j, :, :, :lens[j]]),
                              what=f"kv seq {b} (len {lens[j]}) layer {l}", tier="deep" if l >= 1 else "layer")
    # full last layer gives the same last hidden
    hid_full = bb.prefill(p.tokens.to(DEV), p.lengths, cache, full_last_layer=True)
    # two GPU code paths for the last layer (all rows vs the last rows only): one layer of
    # summation-order spread, at most 2 bf16 ulps of the largest magnitudes
    assert_close(to_np(hid_full), to_np(hid), what="full last layer vs last rows", max_abs=0.0625, min_cos=0.99999)


def _forced_logits(K, Vc, codes):
    """Logits whose argmax is `codes` [1, K] (used to advance the oracle's state machine with codes
    the GPU chose at a near-tie)."""
    lg = np.full((1, K, Vc), -1e30, np.float32)
    for k in range(K):
        lg[0, k, codes[0, k]] = 0.0
    return lg


def test_full_depth_ar_loop(hra, ragged):
    wl = ragged
    d, p, bb, hw = wl["dims"], wl["prompts"], wl["bb"], wl["hw"]
    K, Vc, F = d.n_codebooks, d.codebook_size, 3
    b0 = min(range(len(p.lengths)), key=lambda b: p.lengths[b])
    n = p.lengths[b0]
    n_slots = n + F + 5
    head = hra.AudioHead(d, wl["audio"]["head_w"], wl["audio"]["code_emb"])
    head_u, tab_u = W.to_u16(wl["audio"]["head_w"].cpu()), W.to_u16(wl["audio"]["code_emb"].cpu())
    tok = p.tokens[b0:b0 + 1, :n].contiguous()
    cache = hra.new_kv_cache(d, 1, n_slots, DEV, fill=float("nan"))
    hid = bb.prefill(tok.to(DEV), [n], cache)
    bias = torch.zeros(F, 1, K, dtype=torch.float32)
    bias[1, 0, 0] = 10.0      # EOC forced on codebook 0 at frame 1: codebook 1 follows at frame 2
    loop = hra.ARLoop(bb, head, cache, hid, [n], n + F)
    loop.capture(F, eoc_bias_seq=bias.to(DEV).contiguous())
    loop.replay()
    torch.cuda.synchronize()
    assert hra.hra_device_error(loop.bws) == 0 and hra.hra_device_error(loop.cws) == 0
    codes_g = loop.codes_seq.cpu().numpy()
    done_g = loop.done_seq.cpu().numpy()

    kv_o, h_o = oracle.prefill(d, hw, tok.numpy(), [n], n_slots)
    with oracle.sum_order(True):
        kv_a, h_a = oracle.prefill(d, hw, tok.numpy(), [n], n_slots)
    st = np.array([[0, -1, 0, 0]], np.int32)
    excused = 0
    for t in range(F):
        c_o, nxt_o, d_o, lg_o = oracle.codebook_step(d, h_o, head_u, tab_u, st.copy(), bias[t].numpy())
        if not np.array_equal(c_o, codes_g[t]):
            # excused only where the oracle's top-1 / top-2 margin is a near-tie
            for k in np.nonzero(c_o[0] != codes_g[t, 0])[0]:
                z = lg_o[0, k] + np.where(np.arange(Vc) == d.eoc_id, bias[t, 0, k].item(), 0.0)
                top = np.sort(z)[-2:]
                assert top[1] - top[0] <= ARGMAX_MARGIN, f"frame {t} codebook {k}: argmax differs"
            excused += 1
            c_o = codes_g[t].copy()
            nxt_o = oracle.code_embed_sum(tab_u, c_o)
            _, d_o = oracle.delay_step(K, Vc, d.bos_id, d.eoc_id, _forced_logits(K, Vc, c_o), None, st)
        else:
            oracle.delay_step(K, Vc, d.bos_id, d.eoc_id, lg_o, bias[t].numpy(), st)
        assert np.array_equal(d_o, done_g[t]), f"frame {t}: done"
        h_o = oracle.decode(d, hw, nxt_o, [n + t], kv_o, n_slots)
        with oracle.sum_order(True):
            h_a = oracle.decode(d, hw, nxt_o, [n + t], kv_a, n_slots)
    assert excused <= 1, f"{excused} frames needed the near-tie excuse"
    assert codes_g[1, 0, 0] == d.eoc_id and codes_g[2, 0, 1] == d.eoc_id, "EOC on codebook 0 did not propagate"
    assert loop.state.cpu().numpy().tolist() == st.tolist(), "delay state after the loop"
    assert loop.pos.item() == n + F
    assert_parity(to_np(loop.hidden), ref_np(h_o), ref_np(h_a), what="hidden after the last frame", tier="deep")
    got = cache.float().cpu().numpy()
    for l in range(d.n_layers):
        assert_parity(got[l, 0, :, :, :n + F].astype(np.float64), ref_np(kv_o[l, 0, :, :, :n + F]),
                      ref_np(kv_a[l, 0, :, :, :n + F]), what=f"kv layer {l} after the loop",
                      tier="deep" if l >= 1 else "layer")
    assert bool(torch.isnan(cache[:, 0, :, :, n + F:]).all()), "slots past the loop were written"


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
        assert_parity(got[l], ref_np(kv_o[l, 0]), ref_np(kv_a[l, 0]), what=f"layer {l} kv of seq {b} (len {n})",
                      tier="deep" if l >= 1 else "layer")
    hid_full = bb.prefill(p.tokens.to(DEV), p.lengths, cache, full_last_layer=True)
    # two GPU code paths for the last layer (all rows vs the last rows only): one layer of
    # summation-order spread, at most 2 bf16 ulps of the largest magnitudes
    assert_close(to_np(hid_full), to_np(hid), what="full last layer vs last rows", max_abs=0.0625, min_cos=0.99999)
