"""The no-allocation delayed-codebook step (for callers that cannot call cudaMalloc, such as a
streaming-audio callback with a hard per-frame deadline) must give what the workspace-taking
hra_codebook_step gives, call after call, through the C ABI; and it must refuse a batch whose
scratch need exceeds its fixed array.  Kept in a file of its own that pytest collects last."""
import numpy as np
import pytest
import torch

import workloads as W
from parity import LOGIT_TOL

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_noalloc_matches_workspace_step_twice():
    import qwen3_prefill_delayed_gb300 as hra
    hra.lib()
    d = W.full_dims(0)
    g = torch.Generator(device=DEV).manual_seed(11)
    audio = W.make_audio(d, g, DEV)
    head = hra.AudioHead(d, audio["head_w"], audio["code_emb"])
    B, K, Vc, H = 32, d.n_codebooks, d.codebook_size, d.hidden
    chain = W.make_decode_chain(d, 5, B, 2, device=DEV, inject_frac=0.5)
    chain.eoc_bias[1] += 10.0 * (torch.arange(K, device=DEV) == 2)   # an EOC on codebook 2 in call 2
    st_ref = chain.state0.clone()
    st_na = chain.state0.clone()
    # the output buffers are created up front, so the no-allocation calls themselves allocate nothing
    out = {k: (torch.empty(B, K, dtype=torch.int32, device=DEV), torch.empty(B, H, dtype=torch.bfloat16, device=DEV),
               torch.empty(B, dtype=torch.int32, device=DEV), torch.empty(B, K, Vc, dtype=torch.float32, device=DEV))
           for k in ("ref", "na")}
    for call in range(2):
        c_r, n_r, d_r, l_r = out["ref"]
        c_n, n_n, d_n, l_n = out["na"]
        head.step(chain.hidden[call], st_ref, eoc_bias=chain.eoc_bias[call], codes=c_r, next_emb=n_r, done=d_r,
                  logits=l_r)
        head.step_noalloc(chain.hidden[call], st_na, eoc_bias=chain.eoc_bias[call], codes=c_n, next_emb=n_n,
                          done=d_n, logits=l_n)
        torch.cuda.synchronize()
        assert float((l_r - l_n).abs().max()) <= LOGIT_TOL, f"call {call}: logits"
        assert torch.equal(c_r, c_n), f"call {call}: codes"
        assert torch.equal(st_ref, st_na) and torch.equal(d_r, d_n), f"call {call}: state / done"
        assert torch.equal(n_r, n_n), f"call {call}: next embedding"
    assert int(st_na[:, 0].min()) == int(chain.state0[:, 0].min()) + 2


def test_noalloc_refuses_batch_beyond_scratch():
    import qwen3_prefill_delayed_gb300 as hra
    d = W.full_dims(0)
    g = torch.Generator(device=DEV).manual_seed(12)
    audio = W.make_audio(d, g, DEV)
    head = hra.AudioHead(d, audio["head_w"], audio["code_emb"])
    B = 256
    hid = torch.zeros(B, d.hidden, dtype=torch.bfloat16, device=DEV)
    state = torch.zeros(B, 4, dtype=torch.int32, device=DEV)
    with pytest.raises(hra.HraError, match="workspace"):
        head.step_noalloc(hid, state)
