"""GPU tests of the AR audio loop on device-resident state (hra_ar_frame / hra_decode_dev), captured
once into a CUDA graph and replayed.

- tiny model: a 6-frame graph (EOC bias on codebook 0 at frame 2) against the oracle's loop of
  codebook step + decode pass: codes and stop flags bit-exact, final hidden and cache within the
  parity bar, delay state and positions advanced on the device;
- full-width 2-layer backbone with the K=8 audio head, 8 ragged rows: the graph's frames are bit for
  bit the frames of an eager host-driven loop of hra_codebook_step + hra_decode;
- a device position outside the cache raises HRA_DEVERR_POS_RANGE instead of touching memory past
  the cache; bad arguments are refused before anything is enqueued."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from parity import ARGMAX_MARGIN, assert_parity, ref_np, to_np

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


def test_tiny_graph_loop_matches_oracle(hra):
    wl = W.tiny_reference("cpu")
    d, p, n_slots, F = wl["dims"], wl["prompts"], wl["n_slots"], wl["frames"]
    bb = hra.Backbone(d, _dev(wl["weights"]))
    head = hra.AudioHead(d, wl["audio"]["head_w"].to(DEV), wl["audio"]["code_emb"].to(DEV))
    cache = hra.new_kv_cache(d, 1, n_slots, DEV, fill=float("nan"))
    hid = bb.prefill(p.tokens.to(DEV), p.lengths, cache)
    n = p.lengths[0]
    loop = hra.ARLoop(bb, head, cache, hid, [n], n_slots - 1)
    loop.capture(F, eoc_bias_seq=wl["eoc_bias"].to(DEV).contiguous())
    assert loop.pos.item() == n and loop.state[0, 0].item() == 0      # capturing ran nothing
    loop.replay()
    torch.cuda.synchronize()
    assert hra.hra_device_error(loop.bws) == 0 and hra.hra_device_error(loop.cws) == 0

    hw = oracle.host_weights_from(d, wl["weights"])
    head_u, tab_u = W.to_u16(wl["audio"]["head_w"]), W.to_u16(wl["audio"]["code_emb"])

    codes_g = loop.codes_seq.cpu().numpy()
    K, Vc = d.n_codebooks, d.codebook_size

    def oracle_loop():
        """The oracle's loop; where its codes differ from the GPU's it checks that the oracle's own
        top-1 / top-2 margin is a near-tie (the stated bar: 0.1) and continues from the GPU's codes."""
        kv, h = oracle.prefill(d, hw, p.tokens.numpy(), p.lengths, n_slots)
        st = np.array([[0, -1, 0, 0]], np.int32)
        codes, dones, excused = [], [], 0
        for t in range(F):
            bias = wl["eoc_bias"][t].numpy()
            st0 = st.copy()
            c, nxt, dn, lg = oracle.codebook_step(d, h, head_u, tab_u, st, bias)
            if not np.array_equal(c, codes_g[t]):
                for k in np.nonzero(c[0] != codes_g[t, 0])[0]:
                    z = lg[0, k] + np.where(np.arange(Vc) == d.eoc_id, bias[0, k], 0.0)
                    top = np.sort(z)[-2:]
                    assert top[1] - top[0] <= ARGMAX_MARGIN, f"frame {t} codebook {k}: argmax differs"
                excused += 1
                c = codes_g[t].copy()
                nxt = oracle.code_embed_sum(tab_u, c)
                st = st0
                forced = np.full((1, K, Vc), -1e30, np.float32)
                for k in range(K):
                    forced[0, k, c[0, k]] = 0.0
                _, dn = oracle.delay_step(K, Vc, d.bos_id, d.eoc_id, forced, None, st)
            codes.append(c)
            dones.append(dn)
            h = oracle.decode(d, hw, nxt, [n + t], kv, n_slots)
        return kv, h, st, np.stack(codes), np.stack(dones), excused

    kv_o, h_o, st_o, codes_o, done_o, excused = oracle_loop()
    with oracle.sum_order(True):
        kv_a, h_a, _, _, _, _ = oracle_loop()
    assert excused <= 1, f"{excused} frames needed the near-tie excuse"
    assert codes_g.tolist() == codes_o.tolist()
    assert loop.done_seq.cpu().numpy().tolist() == done_o.tolist()
    assert loop.done_seq[:, 0].cpu().tolist() == [0, 0, 0, 0, 0, 1]
    assert loop.state.cpu().numpy().tolist() == st_o.tolist()
    assert loop.pos.item() == n + F
    assert_parity(to_np(loop.hidden), ref_np(h_o), ref_np(h_a), what="hidden after the last frame")
    got = cache.float().cpu().numpy()
    assert_parity(got[:, 0, :, :, :n + F].astype(np.float64), ref_np(kv_o[:, 0, :, :, :n + F]),
                  ref_np(kv_a[:, 0, :, :, :n + F]), what="kv after the loop")
    assert np.all(np.isnan(got[:, 0, :, :, n + F:]))


def test_graph_frames_equal_eager_frames(hra):
    d = W.full_dims(2)
    w = W.make_backbone(d, 21, DEV)
    au = W.make_audio(d, w["_gen"], DEV)
    p = W.make_prompts(21, 8, 16, 200, d.vocab)
    B, F, n_slots = 8, 12, 512
    bb = hra.Backbone(d, w)
    head = hra.AudioHead(d, au["head_w"], au["code_emb"])
    chain = W.make_decode_chain(d, 21, B, F, device=DEV)
    bias = chain.eoc_bias.contiguous()
    tok = p.tokens.to(DEV)

    # eager: host positions, one hra_codebook_step and one hra_decode per frame
    cache_e = hra.new_kv_cache(d, B, n_slots, DEV, fill=float("nan"))
    hid = bb.prefill(tok, p.lengths, cache_e)
    state = torch.zeros(B, 4, dtype=torch.int32, device=DEV)
    state[:, 1] = -1
    codes_e, done_e = [], []
    for f in range(F):
        c, nxt, dn = head.step(hid, state, eoc_bias=bias[f])
        codes_e.append(c.clone())
        done_e.append(dn.clone())
        hid = bb.decode(nxt, [n + f for n in p.lengths], cache_e)
    torch.cuda.synchronize()

    # graph: device positions, F frames captured once, one replay
    cache_g = hra.new_kv_cache(d, B, n_slots, DEV, fill=float("nan"))
    hid_g = bb.prefill(tok, p.lengths, cache_g)
    loop = hra.ARLoop(bb, head, cache_g, hid_g, p.lengths, max(p.lengths) + F)
    loop.capture(F, eoc_bias_seq=bias)
    loop.replay()
    torch.cuda.synchronize()
    assert hra.hra_device_error(loop.bws) == 0 and hra.hra_device_error(loop.cws) == 0
    assert torch.equal(loop.codes_seq, torch.stack(codes_e))
    assert torch.equal(loop.done_seq, torch.stack(done_e))
    assert torch.equal(loop.state, state)
    assert torch.equal(loop.hidden, hid)
    assert torch.equal(torch.nan_to_num(cache_g.float(), nan=7.0), torch.nan_to_num(cache_e.float(), nan=7.0))
    assert loop.pos.cpu().tolist() == [n + F for n in p.lengths]


def test_device_position_outside_cache(hra):
    d = W.tiny_dims()
    w = W.make_backbone(d, 0, "cpu")
    bb = hra.Backbone(d, _dev(w))
    cache = hra.new_kv_cache(d, 2, 32, DEV, fill=0.0)
    emb = (torch.randn(2, d.hidden, generator=torch.Generator().manual_seed(4)) * 0.5).to(torch.bfloat16).to(DEV)
    pos = torch.tensor([3, 32], dtype=torch.int32, device=DEV)    # row 1 is one past the last slot
    out = bb.decode_dev(emb, pos, 31, cache)
    err = hra.hra_device_error(bb.last_ws)
    assert err & hra.DEVERR_POS_RANGE
    assert torch.isfinite(out.float()).all()
    assert pos.cpu().tolist() == [4, 33]
    # a bound outside the cache is refused before anything runs
    with pytest.raises(hra.HraError, match="outside the cache"):
        bb.decode_dev(emb, pos, 32, cache)
    assert pos.cpu().tolist() == [4, 33]
