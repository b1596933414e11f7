"""Seeded synthetic inputs for the Higgs-Audio-style prefill + delayed-codebook path.

This module is the only code shared by the CUDA path's tests/bench and the CPU
oracle.  It holds no arithmetic of the method: it draws random numbers from a
seeded ``torch.Generator``, rounds each draw once to its bf16 storage type, and
arranges shapes.  Every tensor is returned as a torch tensor on the requested
device; ``to_u16`` gives the raw bf16 bit pattern as a numpy ``uint16`` array
for the oracle.

Shapes follow the Qwen3-style backbone reused by Higgs Audio (pegainfer PR #864
"add checkpoint loading and validation foundation", Why this shape) and the
delayed-codebook step (FlashRT PR #141 "Stabilize Higgs Audio termination and
prefill", Summary).  K = 8 codebooks for the full-width model comes from the
codec row shape ``[N, 8]`` on the vLLM-Omni Higgs Audio v3 page (Test Plan).

Draw order (one generator per workload, in this order):
  backbone: embed, then per layer attn_norm, w_qkv, q_norm, k_norm, w_o,
            mlp_norm, w_gate_up, w_down, then final_norm;
  audio:    head_w, code_emb;
  prompts:  a separate CPU generator (seed + 1000) draws lengths, then ids.
Matrices and embeddings are N(0, 0.02); RMSNorm gains are 1 + N(0, 0.02)
(a literal N(0, 0.02) gain would shrink every activation ~50x per norm).
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np
import torch

BF16 = torch.bfloat16


@dataclasses.dataclass(frozen=True)
class Dims:
    n_layers: int
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    rope_theta: float = 1.0e6
    rms_eps: float = 1.0e-6
    n_codebooks: int = 8
    codebook_size: int = 1026   # 1024 codes + BOS + EOC
    bos_id: int = 1024
    eoc_id: int = 1025

    @property
    def qkv_rows(self) -> int:
        return (self.n_q_heads + 2 * self.n_kv_heads) * self.head_dim


def tiny_dims() -> Dims:
    """2-layer tiny reference: hidden 256, 4 q / 2 kv heads, head_dim 64, FFN 768, vocab 1024, K=4."""
    return Dims(n_layers=2, hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64,
                ffn=768, vocab=1024, n_codebooks=4)


def full_dims(n_layers: int = 36) -> Dims:
    """Full-width layer shape: hidden 2560, 32 q / 8 kv heads, head_dim 128, FFN 9728, vocab 151936, K=8."""
    return Dims(n_layers=n_layers, hidden=2560, n_q_heads=32, n_kv_heads=8, head_dim=128,
                ffn=9728, vocab=151936, n_codebooks=8)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(g, shape, std, device, mean=0.0):
    t = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t.to(BF16)


def make_backbone(d: Dims, seed: int, device="cpu", gen: Optional[torch.Generator] = None) -> dict:
    """Random-init backbone weights, row-major [out, in] bf16 (HF convention).

    w_qkv stacks q rows, then k rows, then v rows; w_gate_up stacks gate rows then up rows.
    """
    g = gen if gen is not None else _gen(seed, device)
    H, hd = d.hidden, d.head_dim
    w = {"embed": _normal(g, (d.vocab, H), 0.02, device), "layers": []}
    for _ in range(d.n_layers):
        w["layers"].append({
            "attn_norm": _normal(g, (H,), 0.02, device, mean=1.0),
            "w_qkv": _normal(g, (d.qkv_rows, H), 0.02, device),
            "q_norm": _normal(g, (hd,), 0.02, device, mean=1.0),
            "k_norm": _normal(g, (hd,), 0.02, device, mean=1.0),
            "w_o": _normal(g, (H, d.n_q_heads * hd), 0.02, device),
            "mlp_norm": _normal(g, (H,), 0.02, device, mean=1.0),
            "w_gate_up": _normal(g, (2 * d.ffn, H), 0.02, device),
            "w_down": _normal(g, (H, d.ffn), 0.02, device),
        })
    w["final_norm"] = _normal(g, (H,), 0.02, device, mean=1.0)
    w["_gen"] = g
    return w


def make_audio(d: Dims, g: torch.Generator, device="cpu") -> dict:
    """Audio head [K*Vc, H] and the K codebook embedding tables [K, Vc, H], bf16 N(0, 0.02)."""
    K, Vc, H = d.n_codebooks, d.codebook_size, d.hidden
    return {"head_w": _normal(g, (K * Vc, H), 0.02, device),
            "code_emb": _normal(g, (K, Vc, H), 0.02, device)}


@dataclasses.dataclass
class Prompts:
    lengths: List[int]          # host copy, one per sequence
    tokens: torch.Tensor        # int32 [B, P_max], pads trailing
    max_len: int

    @property
    def total(self) -> int:
        return int(sum(self.lengths))


def make_prompts(seed: int, batch: int, lo: int, hi: int, vocab: int,
                 fixed_len: Optional[int] = None, pad_value: int = 0) -> Prompts:
    """Ragged prompts: lengths uniform in [lo, hi] (or fixed), ids uniform in [0, vocab), pads trailing."""
    g = _gen(seed + 1000, "cpu")
    if fixed_len is not None:
        lens = [int(fixed_len)] * batch
    else:
        lens = torch.randint(lo, hi + 1, (batch,), generator=g).tolist()
    pmax = max(lens)
    ids = torch.randint(0, vocab, (batch, pmax), generator=g, dtype=torch.int64).to(torch.int32)
    for b, n in enumerate(lens):
        ids[b, n:] = pad_value
    return Prompts(lengths=[int(x) for x in lens], tokens=ids.contiguous(), max_len=pmax)


@dataclasses.dataclass
class DecodeWorkload:
    """Inputs of a chain of delayed-codebook steps.

    hidden: [S, B, H] bf16 per-step hidden bank; state0: int32 [B, 4] = (frame, eoc_frame, done, 0);
    eoc_bias: fp32 [S, B, K] (added to each codebook's EOC logit at that step).
    """
    hidden: torch.Tensor
    state0: torch.Tensor
    eoc_bias: torch.Tensor
    inject_step: List[int]      # -1 where a row gets no injection


def make_decode_chain(d: Dims, seed: int, batch: int, steps: int, device="cpu",
                      max_offset: int = 40, inject_frac: float = 0.25,
                      bias: float = 10.0) -> DecodeWorkload:
    """Seeded chained-step inputs: hidden N(0,1); start frames U{0..max_offset}; EOC bias on codebook 0
    at one uniform step for ceil(inject_frac * B) rows."""
    g = _gen(seed + 2000, "cpu")
    hidden = torch.randn(steps, batch, d.hidden, generator=g, dtype=torch.float32).to(BF16)
    frames = torch.randint(0, max_offset + 1, (batch,), generator=g)
    n_inj = int(math.ceil(inject_frac * batch))
    rows = torch.randperm(batch, generator=g)[:n_inj].tolist()
    when = torch.randint(0, steps, (batch,), generator=g).tolist()
    eoc_bias = torch.zeros(steps, batch, d.n_codebooks, dtype=torch.float32)
    inject = [-1] * batch
    for b in rows:
        eoc_bias[when[b], b, 0] = bias
        inject[b] = int(when[b])
    state0 = torch.zeros(batch, 4, dtype=torch.int32)
    state0[:, 0] = frames.to(torch.int32)
    state0[:, 1] = -1
    return DecodeWorkload(hidden=hidden.to(device), state0=state0.to(device),
                          eoc_bias=eoc_bias.to(device), inject_step=inject)


def to_u16(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 array of its bit patterns (host copy, contiguous)."""
    assert t.dtype == BF16
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def from_u16(a: np.ndarray) -> torch.Tensor:
    """numpy uint16 bit patterns -> bf16 CPU tensor."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(BF16)


# ---- named workloads ------------------------------------------------------------------------

def tiny_reference(device="cpu") -> dict:
    """2-layer tiny model, one P=13 prompt, K=4 audio head and tables, 32-slot cache; 6 frames with
    a +10 EOC bias on codebook 0 at frame 2."""
    d = tiny_dims()
    w = make_backbone(d, 0, device)
    a = make_audio(d, w["_gen"], device)
    p = make_prompts(0, 1, 13, 13, d.vocab, fixed_len=13)
    frames = 6
    bias = torch.zeros(frames, 1, d.n_codebooks, dtype=torch.float32)
    bias[2, 0, 0] = 10.0
    return {"dims": d, "weights": w, "audio": a, "prompts": p, "n_slots": 32,
            "frames": frames, "eoc_bias": bias.to(device)}


def single_layer(P: int, device="cpu") -> dict:
    """One full-width layer, batch 1, P random ids from the 151936 vocab, cache [8, 2048, 128]."""
    d = full_dims(1)
    w = make_backbone(d, 1, device)
    p = make_prompts(1, 1, P, P, d.vocab, fixed_len=P)
    return {"dims": d, "weights": w, "prompts": p, "n_slots": 2048}


def ragged_batch(device="cuda", n_layers: int = 36, batch: int = 32) -> dict:
    """36-layer backbone of the full-width shape; 32 prompts with lengths U{16..256}; 2048 slots."""
    d = full_dims(n_layers)
    w = make_backbone(d, 2, device)
    a = make_audio(d, w["_gen"], device)
    p = make_prompts(2, batch, 16, 256, d.vocab)
    return {"dims": d, "weights": w, "audio": a, "prompts": p, "n_slots": 2048}


def codebook_chain(batch: int, steps: int = 200, device="cpu") -> dict:
    """Decode-step workload: head [8*1026, 2560] and 8 tables [1026, 2560] N(0,0.02); hidden N(0,1)."""
    d = full_dims(0)
    g = _gen(3, device)
    a = make_audio(d, g, device)
    chain = make_decode_chain(d, 3, batch, steps, device)
    return {"dims": d, "audio": a, "chain": chain}


def long_prompts(device="cuda", n_layers: int = 36, batch: int = 8) -> dict:
    """8 prompts with lengths U{1024..2048} on the full-width backbone, 4096-slot cache, K=8 audio."""
    d = full_dims(n_layers)
    w = make_backbone(d, 4, device)
    a = make_audio(d, w["_gen"], device)
    p = make_prompts(4, batch, 1024, 2048, d.vocab)
    return {"dims": d, "weights": w, "audio": a, "prompts": p, "n_slots": 4096, "frames": 64}
