"""GPU parity of the tensor-core projection GEMM (through the C ABI's hra_linear) against the
oracle's fp32 linear, for every epilogue, ragged M / N tails, several M tiles and forced or
automatic K splits.  Shapes of at least 512 rows run in both GEMM forms: on 2-CTA clusters
(256-row tiles, the default) and on single CTAs."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from parity import bf16_ulp, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hra():
    import qwen3_prefill_delayed_gb300 as h
    h.lib()
    return h


def _rand(shape, std, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * std).to(torch.bfloat16)


CASES = [
    # M, N, K, epilogue, split
    (13, 512, 256, "store", 0),
    (200, 384, 640, "store", 0),
    (1000, 1040, 512, "store", 0),
    (1, 6144, 2560, "store", 3),
    (8, 2560, 2560, "residual", 5),
    (100, 2560, 2560, "residual", 3),
    (33, 1040, 640, "store", 0),
    (48, 768, 256, "swiglu", 2),
    (64, 2560, 4096, "residual", 0),
    (517, 2560, 9728, "residual", 0),
    (300, 768, 256, "swiglu", 0),
    (8, 9728, 2560, "swiglu", 0),
    (130, 1000, 512, "swiglu", 0),
    (4255, 2560, 2560, "residual", 0),     # 340 tiles: the last round runs as 4 K pieces per tile
    (4255, 2560, 1024, "swiglu", 0),       # 680 tiles: last round in 2 K pieces
    (4255, 2560, 640, "store", 0),
    (4196, 2560, 2560, "residual", 0),     # pairs: the last 256-row tile's second CTA has no valid row
    (2600, 2560, 4096, "residual", 0),     # pairs: 110 tiles, the last round in 2 K pieces
    (600, 6144, 2560, "store", 0),         # pairs: 3 x 24 tiles, one round
    (1000, 1000, 512, "swiglu", 0),        # ragged N: the last gate/up tile runs past F
    (3, 4104, 256, "f32", 0),
    (1, 8208, 2560, "f32", 0),             # row ranges of 54 weight rows per CTA, whole K
    (8, 6144, 2560, "store", 0),           # row ranges of 41 rows
    (16, 6144, 2560, "residual", 0),
    (64, 8208, 2560, "f32", 0),
    (64, 8208, 2560, "f32", 7),
    # small M, one K split: SwiGLU applied in the GEMM epilogue (gate and up halves of the tile)
    (1, 9728, 2560, "swiglu", 0),
    (32, 9728, 2560, "swiglu", 1),
    (64, 1000, 512, "swiglu", 0),          # ragged last tile: 1000 = 15 x 64 + 40
    (17, 200, 256, "swiglu", 1),
    (32, 768, 256, "swiglu", 3),           # partials + reduction
]


PAIR_MIN_M = 512   # the library's threshold for the 2-CTA form
CASES_BOTH = [c + (True,) for c in CASES] + [c + (False,) for c in CASES if c[0] >= PAIR_MIN_M]


@pytest.fixture()
def gemm_form(hra, request):
    prev = hra.hra_set_gemm_pairs(request.param)
    yield request.param
    hra.hra_set_gemm_pairs(prev)


@pytest.mark.parametrize("M,N,K,epi,split,gemm_form", CASES_BOTH, indirect=["gemm_form"])
def test_linear(hra, M, N, K, epi, split, gemm_form):
    code = {"store": hra.EPI_STORE, "residual": hra.EPI_RESIDUAL, "swiglu": hra.EPI_SWIGLU, "f32": hra.EPI_F32}[epi]
    rows = 2 * N if epi == "swiglu" else N
    x = _rand((M, K), 1.0, M * 7 + K)
    w = _rand((rows, K), 0.02, N * 3 + K)
    acc = oracle.linear(W.to_u16(x), W.to_u16(w)).astype(np.float64)
    xa, wa = np.abs(x.double().numpy()), np.abs(w.double().numpy())
    bound = 2 * K * 2.0 ** -24 * (xa @ wa.T)           # fp32 summation-order bound, both sides
    out = None
    if epi == "residual":
        r0 = _rand((M, N), 1.0, 99)
        out = r0.cuda().clone()
    got = to_np(hra.hra_linear(x.cuda(), w.cuda(), code, out=out, split_k=split))
    torch.cuda.synchronize()
    if epi == "f32":
        assert np.all(np.abs(got - acc) <= bound + 1e-6)
        return
    if epi == "store":
        ref = acc
        tol = bf16_ulp(ref) + bound
    elif epi == "residual":
        ref = r0.double().numpy() + acc
        tol = bf16_ulp(ref) + bound
    else:
        g = np.float32(acc[:, :N]); u = np.float32(acc[:, N:])
        gb = oracle.bf16_value(oracle.bf16_bits(g)).astype(np.float32)
        ub = oracle.bf16_value(oracle.bf16_bits(u)).astype(np.float32)
        ref = (gb / (np.float32(1) + np.exp(-gb)) * ub).astype(np.float64)
        dg = np.abs(ub.astype(np.float64)) * 1.1 * (bound[:, :N] + bf16_ulp(g))
        du = np.abs(gb.astype(np.float64)) * (bound[:, N:] + bf16_ulp(u))
        tol = 2 * bf16_ulp(ref) + dg + du
    refb = oracle.bf16_value(oracle.bf16_bits(np.float32(ref))).astype(np.float64)
    bad = np.abs(got - refb) > tol + 1e-7
    assert not bad.any(), f"{bad.sum()} of {bad.size} outside tolerance; worst {np.max(np.abs(got - refb))}"
