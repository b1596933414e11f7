"""GPU parity of the chained delayed-codebook step at batch 1, 32 and 64 (full-width head
[8 x 1026, 2560], 8 tables [1026, 2560], 200 chained steps, EOC injected on a quarter of the rows).

Every step: the state machine is checked bit for bit by running the oracle's delay step on the
GPU's own logits, and the next embedding bit for bit from the GPU's codes.  Sampled steps: the
oracle recomputes the logits (max |err| <= 5e-2) and its codes must agree wherever its top-1/top-2
margin exceeds 0.1.  A CUDA-graph capture of the 200 steps replays bit-identical to eager calls."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from parity import ARGMAX_MARGIN, LOGIT_TOL

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def hra():
    import qwen3_prefill_delayed_gb300 as h
    h.lib()
    return h


@pytest.fixture(scope="module")
def audio(hra):
    wl = W.codebook_chain(1, steps=1, device="cpu")
    d = wl["dims"]
    head = hra.AudioHead(d, wl["audio"]["head_w"].to(DEV), wl["audio"]["code_emb"].to(DEV))
    return d, head, W.to_u16(wl["audio"]["head_w"]), W.to_u16(wl["audio"]["code_emb"])


def _run_chain(head, d, chain, steps, logits_all=None):
    B = chain.hidden.shape[1]
    state = chain.state0.to(DEV).clone()
    hid = chain.hidden.to(DEV)
    bias = chain.eoc_bias.to(DEV)
    K, H = d.n_codebooks, d.hidden
    codes = torch.empty(steps, B, K, dtype=torch.int32, device=DEV)
    nxt = torch.empty(steps, B, H, dtype=torch.bfloat16, device=DEV)
    done = torch.empty(steps, B, dtype=torch.int32, device=DEV)
    states = torch.empty(steps + 1, B, 4, dtype=torch.int32, device=DEV)
    states[0] = state
    for s in range(steps):
        head.step(hid[s], state, eoc_bias=bias[s], codes=codes[s], next_emb=nxt[s], done=done[s],
                  logits=None if logits_all is None else logits_all[s])
        states[s + 1] = state
    return codes, nxt, done, states


@pytest.mark.parametrize("B", [1, 32, 64])
def test_chain(hra, audio, B):
    d, head, head_u, tab_u = audio
    steps = 200
    chain = W.make_decode_chain(d, 3, B, steps)
    K, Vc = d.n_codebooks, d.codebook_size
    logits = torch.empty(steps, B, K, Vc, dtype=torch.float32, device=DEV)
    codes, nxt, done, states = _run_chain(head, d, chain, steps, logits)
    assert hra.hra_device_error(head.last_ws) == 0
    codes, nxt, done, states = codes.cpu().numpy(), nxt.cpu(), done.cpu().numpy(), states.cpu().numpy()
    lg = logits.cpu().numpy()
    bias = chain.eoc_bias.numpy()
    for s in range(steps):
        st = states[s].copy()
        c_chk, d_chk = oracle.delay_step(K, Vc, d.bos_id, d.eoc_id, lg[s], bias[s], st)
        assert np.array_equal(codes[s], c_chk), f"step {s}: codes differ from the state machine on GPU logits"
        assert np.array_equal(st, states[s + 1]) and np.array_equal(done[s], d_chk), f"step {s}: state"
        np.testing.assert_array_equal(W.to_u16(nxt[s]), oracle.code_embed_sum(tab_u, codes[s]))
    for s in (0, 1, 57, 123, steps - 1):
        st = states[s].copy()
        c_o, _, _, lg_o = oracle.codebook_step(d, W.to_u16(chain.hidden[s]), head_u, tab_u, st, bias[s])
        assert np.max(np.abs(lg[s] - lg_o)) <= LOGIT_TOL, f"step {s}: logits"
        for b in range(B):
            for k in range(K):
                if c_o[b, k] != codes[s, b, k]:
                    top = np.sort(lg_o[b, k] + np.where(np.arange(Vc) == d.eoc_id, bias[s, b, k], 0))[-2:]
                    assert top[1] - top[0] <= ARGMAX_MARGIN, f"step {s} row {b} cb {k}: argmax differs"
    # every injected row stops K - 1 frames after its injection (when that fits in the chain)
    for b, when in enumerate(chain.inject_step):
        if 0 <= when and when + K - 1 < steps:
            assert done[when + K - 1, b] == 1, f"row {b} injected at {when} did not stop"


def test_graph_replay_matches_eager(hra, audio):
    d, head, _, _ = audio
    B, steps = 32, 200
    chain = W.make_decode_chain(d, 3, B, steps)
    ref = _run_chain(head, d, chain, steps)
    torch.cuda.synchronize()
    hid = chain.hidden.to(DEV)
    bias = chain.eoc_bias.to(DEV)
    state = chain.state0.to(DEV).clone()
    codes = torch.empty(steps, B, d.n_codebooks, dtype=torch.int32, device=DEV)
    nxt = torch.empty(steps, B, d.hidden, dtype=torch.bfloat16, device=DEV)
    done = torch.empty(steps, B, dtype=torch.int32, device=DEV)
    ws = torch.empty(head.workspace_size(B), dtype=torch.uint8, device=DEV)
    s0 = torch.cuda.Stream()
    with torch.cuda.stream(s0):
        head.step(hid[0], state.clone(), eoc_bias=bias[0], workspace=ws)   # warm-up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for s in range(steps):
            head.step(hid[s], state, eoc_bias=bias[s], codes=codes[s], next_emb=nxt[s], done=done[s], workspace=ws)
    state.copy_(chain.state0.to(DEV))
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(codes, ref[0]) and torch.equal(nxt, ref[1]) and torch.equal(done, ref[2])
    assert torch.equal(state, ref[3][-1])
