"""CPU-only checks of the C ABI: the library loads without a GPU, exports every entry point that
include/hra.h declares, sizes workspaces, and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def hra():
    import qwen3_prefill_delayed_gb300 as h
    if not os.path.exists(h.LIB_PATH):
        if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
            pytest.skip("no nvcc to build the library")
        from qwen3_prefill_delayed_gb300 import _build
        _build.build()
    h.lib()
    return h


def _declared():
    with open(os.path.join(ROOT, "include", "hra.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"\b(hra_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(hra):
    names = _declared()
    assert len(names) >= 12
    L = ctypes.CDLL(hra.LIB_PATH)
    for n in names:
        assert hasattr(L, n), f"{n} declared in include/hra.h but not exported"
    assert set(names) == set(hra.EXPORTED)


def test_status_strings(hra):
    for rc in (0, -1, -2, -3, -4, -5):
        assert hra.lib().hra_status_string(rc).decode() != "unknown status"
    assert hra.lib().hra_status_string(7).decode() == "unknown status"


def _dims(hra, **kw):
    import workloads as W
    d = W.tiny_dims()
    base = dict(d.__dict__)
    base.update(kw)
    return hra.HraDims(*[base[f] for f, _ in hra.HraDims._fields_])


def test_workspace_sizes(hra):
    L = hra.lib()
    d = _dims(hra)
    a = L.hra_prefill_workspace_size(ctypes.byref(d), 4, 28, 13)
    b = L.hra_prefill_workspace_size(ctypes.byref(d), 4, 52, 13)
    assert 0 < a < b
    assert L.hra_decode_workspace_size(ctypes.byref(d), 4, 32) > 0
    assert L.hra_codebook_workspace_size(ctypes.byref(d), 4) >= 4 * 4 * 1026 * 4
    assert L.hra_prefill_workspace_size(ctypes.byref(_dims(hra, head_dim=96)), 4, 28, 13) == 0
    assert L.hra_linear_workspace_size(13, 512, 256, 0, 0) >= 256
    assert L.hra_linear_workspace_size(0, 512, 256, 0, 0) == 0


def test_bad_arguments_rejected_without_cuda(hra):
    L = hra.lib()
    d = _dims(hra)
    fake = ctypes.c_void_p(0x10000)          # aligned, never dereferenced: validation fails first
    lens = (ctypes.c_int32 * 1)(5)
    kv = hra.HraKvCache(fake.value, 1, 8)
    layers = (hra.HraLayerWeights * 2)()
    for i in range(2):
        for f, _ in hra.HraLayerWeights._fields_:
            setattr(layers[i], f, 0x10000)
    w = hra.HraWeights(0x10000, layers, 0x10000)
    # null dims / weights
    assert L.hra_prefill(None, ctypes.byref(w), fake, lens, 1, 5, ctypes.byref(kv), fake, fake, 1 << 30, 0, None) == -1
    # unsupported head_dim
    d96 = _dims(hra, head_dim=96)
    assert L.hra_prefill(ctypes.byref(d96), ctypes.byref(w), fake, lens, 1, 5, ctypes.byref(kv), fake, fake,
                         1 << 30, 0, None) == -2
    # sequence longer than the cache
    lens9 = (ctypes.c_int32 * 1)(9)
    assert L.hra_prefill(ctypes.byref(d), ctypes.byref(w), fake, lens9, 1, 9, ctypes.byref(kv), fake, fake,
                         1 << 30, 0, None) == -4
    # workspace too small
    assert L.hra_prefill(ctypes.byref(d), ctypes.byref(w), fake, lens, 1, 5, ctypes.byref(kv), fake, fake,
                         16, 0, None) == -3
    # misaligned output
    assert L.hra_prefill(ctypes.byref(d), ctypes.byref(w), fake, lens, 1, 5, ctypes.byref(kv),
                         ctypes.c_void_p(0x10002), fake, 1 << 30, 0, None) == -1
    # decode position outside the cache
    pos = (ctypes.c_int32 * 1)(8)
    assert L.hra_decode(ctypes.byref(d), ctypes.byref(w), fake, pos, 1, ctypes.byref(kv), fake, fake, 1 << 30,
                        None) == -4
    # codebook step: unsupported number of codebooks, bad batch
    d0 = _dims(hra, n_codebooks=0)
    assert L.hra_codebook_step(ctypes.byref(d0), fake, fake, fake, fake, None, 1, fake, fake, fake, None, fake,
                               1 << 30, None) == -2
    assert L.hra_codebook_step(ctypes.byref(d), fake, fake, fake, fake, None, 0, fake, fake, fake, None, fake,
                               1 << 30, None) == -1
    # linear: K not a multiple of 64, N not a multiple of 8
    assert L.hra_linear(fake, fake, fake, 4, 64, 100, 0, 0, fake, 1 << 20, None) == -1
    assert L.hra_linear(fake, fake, fake, 4, 60, 128, 0, 0, fake, 1 << 20, None) == -1
    assert L.hra_launch_counter() == 0


def test_binding_refuses_cpu_tensors(hra):
    import torch
    with pytest.raises(hra.HraError, match="CUDA tensor"):
        hra.hra_linear(torch.zeros(4, 64, dtype=torch.bfloat16), torch.zeros(8, 64, dtype=torch.bfloat16))


def test_newer_entry_points_reject_bad_arguments_without_cuda(hra):
    """Chunked prefill, device-position decode, the AR frame, the sampled step and the FP8 calls
    return the status codes include/hra.h documents, before touching CUDA."""
    L = hra.lib()
    d = _dims(hra)
    A = 0x10000                                # aligned, never dereferenced: validation fails first
    fake = ctypes.c_void_p(A)
    kv = hra.HraKvCache(A, 1, 8)
    layers = (hra.HraLayerWeights * 2)()
    for i in range(2):
        for f, _ in hra.HraLayerWeights._fields_:
            setattr(layers[i], f, A)
    w = hra.HraWeights(A, layers, A)
    big = 1 << 30
    lens5 = (ctypes.c_int32 * 1)(5)

    # chunked prefill: start_pos NULL; start + len past the cache; negative start
    assert L.hra_prefill_chunk(ctypes.byref(d), ctypes.byref(w), fake, lens5, None, 1, 5, ctypes.byref(kv), fake,
                               fake, big, 0, None) == -1
    for start in (4, -1):
        st = (ctypes.c_int32 * 1)(start)
        assert L.hra_prefill_chunk(ctypes.byref(d), ctypes.byref(w), fake, lens5, st, 1, 5, ctypes.byref(kv), fake,
                                   fake, big, 0, None) == -4
    st3 = (ctypes.c_int32 * 1)(3)                                        # 3 + 5 = 8: fits, then too small a workspace
    assert L.hra_prefill_chunk(ctypes.byref(d), ctypes.byref(w), fake, lens5, st3, 1, 5, ctypes.byref(kv), fake,
                               fake, 16, 0, None) == -3

    # device-position decode: no positions; misaligned positions; bound outside [0, n_slots)
    assert L.hra_decode_dev(ctypes.byref(d), ctypes.byref(w), fake, None, 7, 1, 1, ctypes.byref(kv), fake, fake,
                            big, None) == -1
    assert L.hra_decode_dev(ctypes.byref(d), ctypes.byref(w), fake, ctypes.c_void_p(A + 2), 7, 1, 1,
                            ctypes.byref(kv), fake, fake, big, None) == -1
    for bound in (8, -1):
        assert L.hra_decode_dev(ctypes.byref(d), ctypes.byref(w), fake, fake, bound, 1, 1, ctypes.byref(kv), fake,
                                fake, big, None) == -4

    # sampled codebook step: parameter ranges, seeds, codebook size
    def sampled(s, seeds=fake, dims=d):
        return L.hra_codebook_step_sampled(ctypes.byref(dims), fake, fake, fake, fake, None,
                                           ctypes.byref(s) if s is not None else None, seeds, 1, fake, fake, fake,
                                           None, fake, big, None)
    assert sampled(None) == -1
    for t, k, p in ((0.0, 50, 0.95), (float("inf"), 50, 0.95), (float("nan"), 50, 0.95), (1.0, -1, 0.95),
                    (1.0, 50, 0.0), (1.0, 50, 1.5)):
        assert sampled(hra.HraSampling(t, k, p)) == -1, (t, k, p)
    ok = hra.HraSampling(1.0, 50, 0.95)
    assert sampled(ok, seeds=None) == -1
    assert sampled(ok, dims=_dims(hra, codebook_size=3000, bos_id=2998, eoc_id=2999)) == -2

    # AR frame: positions NULL; bound outside the cache; bad sampling parameters
    def frame(pos, bound, s=None):
        return L.hra_ar_frame(ctypes.byref(d), ctypes.byref(w), fake, fake, fake, None,
                              ctypes.byref(s) if s is not None else None, fake if s is not None else None, fake,
                              pos, bound, 1, ctypes.byref(kv), fake, fake, fake, fake, big, fake, big, None)
    assert frame(None, 7) == -1
    assert frame(fake, 8) == -4
    assert frame(fake, 7, hra.HraSampling(-1.0, 0, 1.0)) == -1

    # FP8: quantizers (n a multiple of 8, alignment), the FP8 linear (K a multiple of 128), the FP8
    # prefill (widths a multiple of 128, layer pointers) and calibration (outputs)
    assert L.hra_fp8_quantize_weight(fake, 12, fake, fake, None) == -1
    assert L.hra_fp8_quantize_weight(fake, 64, ctypes.c_void_p(A + 1), fake, None) == -1
    assert L.hra_fp8_quantize(fake, 0, fake, fake, None) == -1
    assert L.hra_linear_fp8(fake, fake, fake, 4, 128, 192, fake, fake, 0, fake, big, None) == -1
    assert L.hra_linear_fp8(fake, fake, fake, 4, 100, 256, fake, fake, 0, fake, big, None) == -1
    assert L.hra_linear_fp8(fake, fake, fake, 4, 128, 256, fake, fake, 0, fake, 16, None) == -3
    f8 = (hra.HraFp8Layer * 2)()
    for i in range(2):
        for f, _ in hra.HraFp8Layer._fields_:
            setattr(f8[i], f, A)
    assert L.hra_prefill_fp8(ctypes.byref(d), ctypes.byref(w), None, fake, lens5, 1, 5, ctypes.byref(kv), fake,
                             fake, big, 0, None) == -1
    assert L.hra_prefill_fp8(ctypes.byref(_dims(hra, ffn=832)), ctypes.byref(w), f8, fake, lens5, 1, 5,
                             ctypes.byref(kv), fake, fake, big, 0, None) == -2
    f8[1].a_scale = A + 2
    assert L.hra_prefill_fp8(ctypes.byref(d), ctypes.byref(w), f8, fake, lens5, 1, 5, ctypes.byref(kv), fake,
                             fake, big, 0, None) == -1
    assert L.hra_fp8_calibrate(ctypes.byref(d), ctypes.byref(w), fake, lens5, 1, 5, ctypes.byref(kv), None, fake,
                               fake, big, None) == -1
    # NVFP4 quantizer: K a multiple of 16, aligned operands
    assert L.hra_nvfp4_quantize(fake, 4, 24, fake, fake, fake, None) == -1
    assert L.hra_nvfp4_quantize(fake, 4, 64, ctypes.c_void_p(A + 2), fake, fake, None) == -1
    assert L.hra_nvfp4_quantize(fake, 0, 64, fake, fake, fake, None) == -1
    assert L.hra_launch_counter() == 0


def test_form_switches_return_the_previous_setting(hra):
    """hra_set_gemm_pairs and hra_set_decode_pass are host-side flags: each returns the setting it
    replaced, and the defaults are the 2-CTA GEMMs on and the persistent decoder pass off."""
    assert hra.hra_set_gemm_pairs(False) is True
    assert hra.hra_set_gemm_pairs(True) is False
    assert hra.hra_set_gemm_pairs(True) is True
    assert hra.hra_set_decode_pass(True) is False
    assert hra.hra_set_decode_pass(False) is True


def test_linear_workspace_covers_both_gemm_forms(hra):
    """The workspace size of a projection of at least 512 rows is valid in both GEMM forms (the last
    round's K pieces are sized for the form that runs)."""
    L = hra.lib()
    sizes = {}
    for pairs in (True, False):
        prev = hra.hra_set_gemm_pairs(pairs)
        try:
            sizes[pairs] = L.hra_linear_workspace_size(4255, 2560, 4096, 1, 0)
        finally:
            hra.hra_set_gemm_pairs(prev)
    assert all(s >= 256 for s in sizes.values())
