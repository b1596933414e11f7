"""GPU parity of the NVFP4 quantizer (hra_nvfp4_quantize) against the pinned oracle
(oracle_quantize_nvfp4; the chain's FP4 band, the fp8_chain page's precision bands): codes and
block scales bit
for bit on the same bf16 input and the same global scale, over magnitudes that put block scales in
the E4M3 normal and subnormal ranges, an all-zero block and saturating elements."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def hra():
    import qwen3_prefill_delayed_gb300 as h
    h.lib()
    return h


@pytest.mark.parametrize("rows,K,gmode", [(40, 256, "tensor"), (7, 64, "tensor"), (33, 512, "one"), (5, 4096, "small")])
def test_nvfp4_quantize_bit_exact(hra, rows, K, gmode):
    g_rng = np.random.default_rng(rows + K)
    x = g_rng.standard_normal((rows, K)) * np.exp(g_rng.uniform(-6, 4, (rows, 1)))
    x[0, 16:32] = 0.0                        # an all-zero block
    x[1, 40] = 1e4                           # a block whose other elements round to 0
    xb = oracle.bf16_bits(x.astype(np.float32))
    g = {"tensor": oracle.nvfp4_global(xb), "one": 1.0, "small": 1e-3}[gmode]
    codes_o, scales_o = oracle.quantize_nvfp4(xb, g)
    xt = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).to(DEV)
    gt = torch.tensor([g], dtype=torch.float32, device=DEV)
    codes, scales = hra.nvfp4_quantize(xt, gt)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(scales.cpu().numpy(), scales_o)
    np.testing.assert_array_equal(codes.cpu().numpy(), codes_o)
