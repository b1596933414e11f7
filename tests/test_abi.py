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
