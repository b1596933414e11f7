"""GB300-native Higgs-Audio-style hot path: batched BF16 prefill of a Qwen3-style backbone and the
per-frame delayed-codebook step.

This module is a thin ctypes binding of the in-tree CUDA library ``libhra.so`` (C ABI in
``include/hra.h``).  It only marshals torch tensors into pointers and sizes: every step of the
path runs in the library's kernels.  There is no CPU fallback -- calling anything here without the
built library, or with tensors not on a CUDA device, raises.

Entry points (same names as the C ABI): ``hra_prefill`` (and ``hra_prefill_chunk`` through
``Backbone.prefill(..., start_pos=...)``), ``hra_decode``, ``hra_codebook_step``,
``hra_linear``, ``hra_device_error``; convenience wrappers ``Backbone`` and ``AudioHead`` keep the
weight tables and workspaces.
"""
from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Sequence

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libhra.so")

HRA_OK = 0
STATUS = {0: "ok", -1: "invalid argument", -2: "unsupported dims", -3: "workspace too small",
          -4: "length or position outside the cache", -5: "CUDA error"}
DEVERR_TOKEN_RANGE, DEVERR_WAIT_TIMEOUT, DEVERR_CODE_RANGE, DEVERR_POS_RANGE = 1, 2, 4, 8
EPI_STORE, EPI_RESIDUAL, EPI_SWIGLU, EPI_F32 = 0, 1, 2, 3
PREFILL_FULL_LAST_LAYER = 1

EXPORTED = ["hra_prefill_workspace_size", "hra_prefill", "hra_prefill_chunk_workspace_size", "hra_prefill_chunk",
            "hra_decode_workspace_size", "hra_decode", "hra_decode_dev", "hra_ar_frame",
            "hra_codebook_workspace_size", "hra_codebook_step", "hra_codebook_step_sampled",
            "hra_codebook_step_noalloc",
            "hra_linear_workspace_size",
            "hra_linear", "hra_fp8_quantize_weight", "hra_fp8_quantize", "hra_nvfp4_quantize", "hra_linear_fp8_workspace_size",
            "hra_linear_fp8", "hra_fp8_calibrate_workspace_size", "hra_fp8_calibrate",
            "hra_prefill_fp8_workspace_size", "hra_prefill_fp8",
            "hra_nvfp4_quantize_weight", "hra_linear_nvfp4_workspace_size", "hra_linear_nvfp4",
            "hra_nvfp4_band_scales",
            "hra_prefill_nvfp4_workspace_size", "hra_prefill_nvfp4",
            "hra_launch_counter", "hra_probe_select", "hra_probe_collect", "hra_set_decode_pass",
            "hra_set_gemm_pairs", "hra_device_error", "hra_status_string"]
PROBE = {"none": 0, "qkv": 1, "o_proj": 2, "gate_up": 3, "down": 4, "attention": 5, "audio_head": 6,
         "decode_attention": 7, "decode_linear": 8}


class HraError(RuntimeError):
    pass


class HraDims(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("hidden", ctypes.c_int32),
                ("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("ffn", ctypes.c_int32), ("vocab", ctypes.c_int32),
                ("rope_theta", ctypes.c_float), ("rms_eps", ctypes.c_float),
                ("n_codebooks", ctypes.c_int32), ("codebook_size", ctypes.c_int32),
                ("bos_id", ctypes.c_int32), ("eoc_id", ctypes.c_int32)]


class HraLayerWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("attn_norm", "w_qkv", "q_norm", "k_norm", "w_o", "mlp_norm", "w_gate_up", "w_down")]


class HraWeights(ctypes.Structure):
    _fields_ = [("embed", ctypes.c_void_p), ("layers", ctypes.POINTER(HraLayerWeights)),
                ("final_norm", ctypes.c_void_p)]


class HraKvCache(ctypes.Structure):
    _fields_ = [("base", ctypes.c_void_p), ("batch", ctypes.c_int32), ("n_slots", ctypes.c_int32)]


class HraFp8Layer(ctypes.Structure):
    _fields_ = [("w_qkv", ctypes.c_void_p), ("w_o", ctypes.c_void_p), ("w_gate_up", ctypes.c_void_p),
                ("w_down", ctypes.c_void_p), ("w_scale", ctypes.c_void_p), ("a_scale", ctypes.c_void_p)]


class HraNvfp4Layer(ctypes.Structure):
    _fields_ = [("w_qkv", ctypes.c_void_p), ("codes", ctypes.c_void_p * 4), ("scales", ctypes.c_void_p * 4),
                ("w_scale", ctypes.c_void_p), ("a_scale", ctypes.c_void_p)]


class HraSampling(ctypes.Structure):
    """hra_sampling: temperature (> 0), top_k (0 = off), top_p (1 = off)."""
    _fields_ = [("temperature", ctypes.c_float), ("top_k", ctypes.c_int32), ("top_p", ctypes.c_float)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise HraError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                           "(there is no CPU fallback)")
        L = ctypes.CDLL(LIB_PATH)
        sz, i32, vp, u32 = ctypes.c_size_t, ctypes.c_int32, ctypes.c_void_p, ctypes.c_uint32
        dp = ctypes.POINTER(HraDims)
        L.hra_prefill_workspace_size.argtypes = [dp, i32, i32, i32]
        L.hra_prefill_workspace_size.restype = sz
        L.hra_prefill.argtypes = [dp, ctypes.POINTER(HraWeights), vp, ctypes.POINTER(i32), i32, i32,
                                  ctypes.POINTER(HraKvCache), vp, vp, sz, u32, vp]
        L.hra_prefill.restype = ctypes.c_int
        L.hra_prefill_chunk_workspace_size.argtypes = [dp, i32, i32, i32, i32]
        L.hra_prefill_chunk_workspace_size.restype = sz
        L.hra_prefill_chunk.argtypes = [dp, ctypes.POINTER(HraWeights), vp, ctypes.POINTER(i32),
                                        ctypes.POINTER(i32), i32, i32, ctypes.POINTER(HraKvCache), vp, vp, sz,
                                        u32, vp]
        L.hra_prefill_chunk.restype = ctypes.c_int
        L.hra_decode_workspace_size.argtypes = [dp, i32, i32]
        L.hra_decode_workspace_size.restype = sz
        L.hra_decode.argtypes = [dp, ctypes.POINTER(HraWeights), vp, ctypes.POINTER(i32), i32,
                                 ctypes.POINTER(HraKvCache), vp, vp, sz, vp]
        L.hra_decode.restype = ctypes.c_int
        L.hra_decode_dev.argtypes = [dp, ctypes.POINTER(HraWeights), vp, vp, i32, i32, i32,
                                     ctypes.POINTER(HraKvCache), vp, vp, sz, vp]
        L.hra_decode_dev.restype = ctypes.c_int
        L.hra_ar_frame.argtypes = [dp, ctypes.POINTER(HraWeights), vp, vp, vp, vp, ctypes.POINTER(HraSampling), vp,
                                   vp, vp, i32, i32, ctypes.POINTER(HraKvCache), vp, vp, vp, vp, sz, vp, sz, vp]
        L.hra_ar_frame.restype = ctypes.c_int
        L.hra_codebook_workspace_size.argtypes = [dp, i32]
        L.hra_codebook_workspace_size.restype = sz
        L.hra_codebook_step.argtypes = [dp, vp, vp, vp, vp, vp, i32, vp, vp, vp, vp, vp, sz, vp]
        L.hra_codebook_step.restype = ctypes.c_int
        L.hra_codebook_step_sampled.argtypes = [dp, vp, vp, vp, vp, vp, ctypes.POINTER(HraSampling), vp, i32, vp,
                                                vp, vp, vp, vp, sz, vp]
        L.hra_codebook_step_sampled.restype = ctypes.c_int
        L.hra_codebook_step_noalloc.argtypes = [dp, vp, vp, vp, vp, vp, i32, vp, vp, vp, vp, vp]
        L.hra_codebook_step_noalloc.restype = ctypes.c_int
        i64 = ctypes.c_int64
        L.hra_fp8_quantize_weight.argtypes = [vp, i64, vp, vp, vp]
        L.hra_fp8_quantize.argtypes = [vp, i64, vp, vp, vp]
        L.hra_nvfp4_quantize.argtypes = [vp, i32, i32, vp, vp, vp, vp]
        L.hra_nvfp4_quantize.restype = ctypes.c_int
        L.hra_linear_fp8_workspace_size.argtypes = [i32, i32, i32, i32]
        L.hra_linear_fp8_workspace_size.restype = sz
        L.hra_linear_fp8.argtypes = [vp, vp, vp, i32, i32, i32, vp, vp, i32, vp, sz, vp]
        L.hra_fp8_calibrate_workspace_size.argtypes = [dp, i32, i32, i32]
        L.hra_fp8_calibrate_workspace_size.restype = sz
        L.hra_fp8_calibrate.argtypes = [dp, ctypes.POINTER(HraWeights), vp, ctypes.POINTER(i32), i32, i32,
                                        ctypes.POINTER(HraKvCache), vp, vp, vp, sz, vp]
        L.hra_prefill_fp8_workspace_size.argtypes = [dp, i32, i32, i32]
        L.hra_prefill_fp8_workspace_size.restype = sz
        L.hra_prefill_fp8.argtypes = [dp, ctypes.POINTER(HraWeights), ctypes.POINTER(HraFp8Layer), vp,
                                      ctypes.POINTER(i32), i32, i32, ctypes.POINTER(HraKvCache), vp, vp, sz, u32, vp]
        L.hra_nvfp4_quantize_weight.argtypes = [vp, i32, i32, vp, vp, vp, vp]
        L.hra_nvfp4_band_scales.argtypes = [vp, vp, i32, vp]
        L.hra_linear_nvfp4_workspace_size.argtypes = []
        L.hra_linear_nvfp4_workspace_size.restype = sz
        L.hra_linear_nvfp4.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, vp, vp, i32, vp, sz, vp]
        L.hra_prefill_nvfp4_workspace_size.argtypes = [dp, i32, i32, i32]
        L.hra_prefill_nvfp4_workspace_size.restype = sz
        L.hra_prefill_nvfp4.argtypes = [dp, ctypes.POINTER(HraWeights), ctypes.POINTER(HraNvfp4Layer), vp,
                                        ctypes.POINTER(i32), i32, i32, ctypes.POINTER(HraKvCache), vp, vp, sz, u32, vp]
        for f in ("hra_fp8_quantize_weight", "hra_fp8_quantize", "hra_linear_fp8", "hra_fp8_calibrate",
                  "hra_prefill_fp8", "hra_nvfp4_quantize_weight", "hra_linear_nvfp4", "hra_prefill_nvfp4",
                  "hra_nvfp4_band_scales"):
            getattr(L, f).restype = ctypes.c_int
        L.hra_linear_workspace_size.argtypes = [i32, i32, i32, i32, i32]
        L.hra_linear_workspace_size.restype = sz
        L.hra_linear.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, vp, sz, vp]
        L.hra_linear.restype = ctypes.c_int
        L.hra_launch_counter.argtypes = []
        L.hra_launch_counter.restype = ctypes.c_uint64
        L.hra_probe_select.argtypes = [ctypes.c_int]
        L.hra_probe_select.restype = ctypes.c_int
        L.hra_set_decode_pass.argtypes = [i32]
        L.hra_set_decode_pass.restype = i32
        L.hra_set_gemm_pairs.argtypes = [i32]
        L.hra_set_gemm_pairs.restype = i32
        L.hra_probe_collect.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int64),
                                        ctypes.POINTER(ctypes.c_double)]
        L.hra_probe_collect.restype = ctypes.c_int
        L.hra_device_error.argtypes = [vp, vp]
        L.hra_device_error.restype = i32
        L.hra_status_string.argtypes = [ctypes.c_int]
        L.hra_status_string.restype = ctypes.c_char_p
        _lib = L
    return _lib


def _check(rc: int, what: str) -> None:
    if rc != HRA_OK:
        msg = lib().hra_status_string(rc).decode()
        raise HraError(f"{what} failed: {msg} ({rc})")


def _ptr(t: Optional[torch.Tensor], dtype=None, name="tensor"):
    if t is None:
        return None
    if not t.is_cuda:
        raise HraError(f"{name} must be a CUDA tensor (there is no CPU path)")
    if not t.is_contiguous():
        raise HraError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise HraError(f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def make_dims(d) -> HraDims:
    """HraDims from any object with the Dims field names (e.g. workloads.Dims)."""
    return HraDims(d.n_layers, d.hidden, d.n_q_heads, d.n_kv_heads, d.head_dim, d.ffn, d.vocab,
                   d.rope_theta, d.rms_eps, d.n_codebooks, d.codebook_size, d.bos_id, d.eoc_id)


def new_kv_cache(d, batch: int, n_slots: int, device="cuda", fill=None) -> torch.Tensor:
    """Cache tensor [n_layers, batch, 2, n_kv_heads, n_slots, head_dim] bf16."""
    shape = (d.n_layers, batch, 2, d.n_kv_heads, n_slots, d.head_dim)
    if fill is None:
        return torch.empty(shape, dtype=torch.bfloat16, device=device)
    return torch.full(shape, fill, dtype=torch.bfloat16, device=device)


class _Workspace:
    def __init__(self):
        self.buf: Optional[torch.Tensor] = None

    def get(self, nbytes: int, device) -> torch.Tensor:
        if self.buf is None or self.buf.numel() < nbytes or self.buf.device != torch.device(device):
            self.buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        return self.buf


_LAYER_KEYS = ("attn_norm", "w_qkv", "q_norm", "k_norm", "w_o", "mlp_norm", "w_gate_up", "w_down")


class Backbone:
    """A Qwen3-style backbone on the GPU: weights dict as produced by ``workloads.make_backbone``
    (embed [V,H], layers[...] with the ``hra_layer_weights`` names, final_norm [H], bf16 CUDA)."""

    def __init__(self, d, weights: dict):
        self.d = d
        self.dims = make_dims(d)
        self.w = weights
        n = d.n_layers
        self._layers = (HraLayerWeights * n)()
        for i in range(n):
            for k in _LAYER_KEYS:
                setattr(self._layers[i], k, _ptr(weights["layers"][i][k], torch.bfloat16, k).value)
        self.table = HraWeights(_ptr(weights["embed"], torch.bfloat16, "embed").value, self._layers,
                                _ptr(weights["final_norm"], torch.bfloat16, "final_norm").value)
        self.ws = _Workspace()
        self.device = weights["embed"].device

    def kv(self, cache: torch.Tensor) -> HraKvCache:
        d = self.d
        if cache.dtype != torch.bfloat16 or cache.dim() != 6 or cache.shape[0] != d.n_layers \
                or cache.shape[2] != 2 or cache.shape[3] != d.n_kv_heads or cache.shape[5] != d.head_dim:
            raise HraError("KV cache must be bf16 [n_layers, batch, 2, n_kv_heads, n_slots, head_dim]")
        return HraKvCache(_ptr(cache, torch.bfloat16, "kv cache").value, cache.shape[1], cache.shape[4])

    def prefill_workspace_size(self, batch, total, max_len) -> int:
        return lib().hra_prefill_workspace_size(ctypes.byref(self.dims), batch, total, max_len)

    def prefill_chunk_workspace_size(self, batch, total, max_len, max_end) -> int:
        return lib().hra_prefill_chunk_workspace_size(ctypes.byref(self.dims), batch, total, max_len, max_end)

    def prefill(self, tokens: torch.Tensor, seq_lens: Sequence[int], cache: torch.Tensor,
                out: Optional[torch.Tensor] = None, full_last_layer: bool = False,
                workspace: Optional[torch.Tensor] = None, stream=None,
                start_pos: Optional[Sequence[int]] = None) -> torch.Tensor:
        """hra_prefill: tokens int32 [B, P_max] (CUDA), seq_lens host ints -> last hidden [B, H].

        With start_pos (host ints), hra_prefill_chunk: row b's tokens sit at positions
        start_pos[b] .. start_pos[b] + seq_lens[b] - 1 after the ones already in the cache."""
        B, P = tokens.shape
        lens = (ctypes.c_int32 * B)(*[int(x) for x in seq_lens])
        if out is None:
            out = torch.empty(B, self.d.hidden, dtype=torch.bfloat16, device=tokens.device)
        flags = PREFILL_FULL_LAST_LAYER if full_last_layer else 0
        kv = self.kv(cache)
        if start_pos is None:
            need = self.prefill_workspace_size(B, int(sum(seq_lens)), P)
        else:
            starts = (ctypes.c_int32 * B)(*[int(x) for x in start_pos])
            max_end = max(int(a) + int(n) for a, n in zip(start_pos, seq_lens))
            need = self.prefill_chunk_workspace_size(B, int(sum(seq_lens)), P, max(max_end, P))
        ws = workspace if workspace is not None else self.ws.get(need, tokens.device)
        if start_pos is None:
            rc = lib().hra_prefill(ctypes.byref(self.dims), ctypes.byref(self.table),
                                   _ptr(tokens, torch.int32, "tokens"), lens, B, P, ctypes.byref(kv),
                                   _ptr(out, torch.bfloat16, "last_hidden"), _ptr(ws, None, "workspace"),
                                   ws.numel(), flags, _stream(stream))
            _check(rc, "hra_prefill")
        else:
            rc = lib().hra_prefill_chunk(ctypes.byref(self.dims), ctypes.byref(self.table),
                                         _ptr(tokens, torch.int32, "tokens"), lens, starts, B, P,
                                         ctypes.byref(kv), _ptr(out, torch.bfloat16, "last_hidden"),
                                         _ptr(ws, None, "workspace"), ws.numel(), flags, _stream(stream))
            _check(rc, "hra_prefill_chunk")
        self.last_ws = ws
        return out

    def decode_dev(self, in_emb: torch.Tensor, pos: torch.Tensor, pos_bound: int, cache: torch.Tensor,
                   advance: bool = True, out: Optional[torch.Tensor] = None,
                   workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        """hra_decode_dev: positions in the CUDA int32 tensor `pos` (advanced in place when
        `advance`); pos_bound is a host upper bound of every position."""
        B = in_emb.shape[0]
        if out is None:
            out = torch.empty(B, self.d.hidden, dtype=torch.bfloat16, device=in_emb.device)
        need = self.decode_workspace_size(B, cache.shape[4])
        ws = workspace if workspace is not None else self.ws.get(need, in_emb.device)
        kv = self.kv(cache)
        rc = lib().hra_decode_dev(ctypes.byref(self.dims), ctypes.byref(self.table),
                                  _ptr(in_emb, torch.bfloat16, "in_emb"), _ptr(pos, torch.int32, "pos"),
                                  int(pos_bound), 1 if advance else 0, B, ctypes.byref(kv),
                                  _ptr(out, torch.bfloat16, "hidden"), _ptr(ws, None, "workspace"), ws.numel(),
                                  _stream(stream))
        _check(rc, "hra_decode_dev")
        self.last_ws = ws
        return out

    def decode_workspace_size(self, batch, n_slots) -> int:
        return lib().hra_decode_workspace_size(ctypes.byref(self.dims), batch, n_slots)

    def decode(self, in_emb: torch.Tensor, pos: Sequence[int], cache: torch.Tensor,
               out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
               stream=None) -> torch.Tensor:
        """hra_decode: in_emb bf16 [B, H] (CUDA), pos host ints -> hidden [B, H]."""
        B = in_emb.shape[0]
        p = (ctypes.c_int32 * B)(*[int(x) for x in pos])
        if out is None:
            out = torch.empty(B, self.d.hidden, dtype=torch.bfloat16, device=in_emb.device)
        need = self.decode_workspace_size(B, cache.shape[4])
        ws = workspace if workspace is not None else self.ws.get(need, in_emb.device)
        kv = self.kv(cache)
        rc = lib().hra_decode(ctypes.byref(self.dims), ctypes.byref(self.table),
                              _ptr(in_emb, torch.bfloat16, "in_emb"), p, B, ctypes.byref(kv),
                              _ptr(out, torch.bfloat16, "hidden"), _ptr(ws, None, "workspace"),
                              ws.numel(), _stream(stream))
        _check(rc, "hra_decode")
        self.last_ws = ws
        return out


class ARLoop:
    """The AR audio loop on device-resident state: each frame is one hra_ar_frame call (codebook
    step on the current hidden, then the decode pass at the device positions, which advance by
    one).  No frame depends on host data, so `capture(n)` records n frames into one CUDA graph and
    `replay()` runs them with a single launch from the host.

    pos0: host ints, the position of each row's first decoded frame (its prompt length); pos_bound
    (host) must cover every position the loop will reach."""

    def __init__(self, bb: "Backbone", head: "AudioHead", cache: torch.Tensor, hidden: torch.Tensor,
                 pos0: Sequence[int], pos_bound: int, eoc_bias: Optional[torch.Tensor] = None,
                 sampling=None, seeds: Optional[torch.Tensor] = None):
        self.bb, self.head, self.cache = bb, head, cache
        self.sampling = None if sampling is None else HraSampling(*sampling)   # (temperature, top_k, top_p)
        self.seeds = seeds                                                      # CUDA int64 [B] (uint64 bits)
        d = bb.d
        B = hidden.shape[0]
        dev = hidden.device
        self.B = B
        self.hidden = hidden                      # in/out: the current backbone hidden
        self.state = torch.zeros(B, 4, dtype=torch.int32, device=dev)
        self.state[:, 1] = -1
        self.pos = torch.tensor([int(x) for x in pos0], dtype=torch.int32, device=dev)
        self.pos_bound = int(pos_bound)
        self.eoc_bias = eoc_bias
        self.codes = torch.empty(B, d.n_codebooks, dtype=torch.int32, device=dev)
        self.next_emb = torch.empty(B, d.hidden, dtype=torch.bfloat16, device=dev)
        self.done = torch.empty(B, dtype=torch.int32, device=dev)
        self.bws = torch.empty(bb.decode_workspace_size(B, cache.shape[4]), dtype=torch.uint8, device=dev)
        self.cws = torch.empty(head.workspace_size(B), dtype=torch.uint8, device=dev)
        self.kv = bb.kv(cache)
        self.graph = None

    def frame(self, codes: Optional[torch.Tensor] = None, done: Optional[torch.Tensor] = None,
              eoc_bias: Optional[torch.Tensor] = None, stream=None):
        """Enqueue one frame; codes/done default to the loop's own buffers, eoc_bias (fp32 [B, K])
        to the loop's.  Returns (codes, done)."""
        codes = self.codes if codes is None else codes
        done = self.done if done is None else done
        bias = self.eoc_bias if eoc_bias is None else eoc_bias
        rc = lib().hra_ar_frame(ctypes.byref(self.bb.dims), ctypes.byref(self.bb.table),
                                _ptr(self.head.head_w, torch.bfloat16, "head_w"),
                                _ptr(self.head.code_emb, torch.bfloat16, "code_emb"),
                                _ptr(self.state, torch.int32, "state"),
                                _ptr(bias, torch.float32, "eoc_bias"),
                                ctypes.byref(self.sampling) if self.sampling is not None else None,
                                _ptr(self.seeds, torch.int64, "seeds"),
                                _ptr(self.hidden, torch.bfloat16, "hidden"), _ptr(self.pos, torch.int32, "pos"),
                                self.pos_bound, self.B, ctypes.byref(self.kv),
                                _ptr(codes, torch.int32, "codes"), _ptr(self.next_emb, torch.bfloat16, "next_emb"),
                                _ptr(done, torch.int32, "done"), _ptr(self.bws, None, "backbone workspace"),
                                self.bws.numel(), _ptr(self.cws, None, "codebook workspace"), self.cws.numel(),
                                _stream(stream))
        _check(rc, "hra_ar_frame")
        return codes, done

    def capture(self, n_frames: int, eoc_bias_seq: Optional[torch.Tensor] = None) -> None:
        """Record n_frames frames into one CUDA graph; frame f writes codes_seq[f] and done_seq[f]
        (and adds eoc_bias_seq[f], fp32 [n_frames, B, K], when given).  Capturing runs nothing: the
        state, positions and hidden are untouched until replay()."""
        dev = self.hidden.device
        self.codes_seq = torch.empty(n_frames, self.B, self.bb.d.n_codebooks, dtype=torch.int32, device=dev)
        self.done_seq = torch.empty(n_frames, self.B, dtype=torch.int32, device=dev)
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            for f in range(n_frames):
                bias = None if eoc_bias_seq is None else eoc_bias_seq[f]
                self.frame(self.codes_seq[f], self.done_seq[f], eoc_bias=bias, stream=side)
        torch.cuda.current_stream(dev).wait_stream(side)
        self.graph = g

    def replay(self) -> None:
        self.graph.replay()


class AudioHead:
    """Audio head [K*Vc, H] and codebook tables [K, Vc, H] (bf16, CUDA) for hra_codebook_step."""

    def __init__(self, d, head_w: torch.Tensor, code_emb: torch.Tensor):
        self.d = d
        self.dims = make_dims(d)
        self.head_w = head_w
        self.code_emb = code_emb
        self.ws = _Workspace()

    def workspace_size(self, batch: int) -> int:
        return lib().hra_codebook_workspace_size(ctypes.byref(self.dims), batch)

    def step(self, hidden: torch.Tensor, state: torch.Tensor, eoc_bias: Optional[torch.Tensor] = None,
             codes: Optional[torch.Tensor] = None, next_emb: Optional[torch.Tensor] = None,
             done: Optional[torch.Tensor] = None, logits: Optional[torch.Tensor] = None,
             workspace: Optional[torch.Tensor] = None, stream=None, sampling=None,
             seeds: Optional[torch.Tensor] = None):
        """hra_codebook_step: state int32 [B, 4] (frame, eoc_frame, done, 0), advanced in place.
        Returns (codes int32 [B, K], next_emb bf16 [B, H], done int32 [B]).

        With sampling = (temperature, top_k, top_p) and seeds (CUDA uint64 [B], one per row; torch
        int64 holding the same bits), hra_codebook_step_sampled."""
        B = hidden.shape[0]
        K, Vc, H = self.d.n_codebooks, self.d.codebook_size, self.d.hidden
        dev = hidden.device
        if codes is None:
            codes = torch.empty(B, K, dtype=torch.int32, device=dev)
        if next_emb is None:
            next_emb = torch.empty(B, H, dtype=torch.bfloat16, device=dev)
        if done is None:
            done = torch.empty(B, dtype=torch.int32, device=dev)
        if state.dtype != torch.int32 or tuple(state.shape) != (B, 4):
            raise HraError("state must be int32 [B, 4]")
        ws = workspace if workspace is not None else self.ws.get(self.workspace_size(B), dev)
        if sampling is not None:
            sp = HraSampling(*sampling)
            rc = lib().hra_codebook_step_sampled(ctypes.byref(self.dims), _ptr(hidden, torch.bfloat16, "hidden"),
                                                 _ptr(self.head_w, torch.bfloat16, "head_w"),
                                                 _ptr(self.code_emb, torch.bfloat16, "code_emb"),
                                                 _ptr(state, torch.int32, "state"),
                                                 _ptr(eoc_bias, torch.float32, "eoc_bias"), ctypes.byref(sp),
                                                 _ptr(seeds, torch.int64, "seeds"), B,
                                                 _ptr(codes, torch.int32, "codes"),
                                                 _ptr(next_emb, torch.bfloat16, "next_emb"),
                                                 _ptr(done, torch.int32, "done"),
                                                 _ptr(logits, torch.float32, "logits"),
                                                 _ptr(ws, None, "workspace"), ws.numel(), _stream(stream))
            _check(rc, "hra_codebook_step_sampled")
            self.last_ws = ws
            return codes, next_emb, done
        rc = lib().hra_codebook_step(ctypes.byref(self.dims), _ptr(hidden, torch.bfloat16, "hidden"),
                                     _ptr(self.head_w, torch.bfloat16, "head_w"),
                                     _ptr(self.code_emb, torch.bfloat16, "code_emb"),
                                     _ptr(state, torch.int32, "state"),
                                     _ptr(eoc_bias, torch.float32, "eoc_bias"), B,
                                     _ptr(codes, torch.int32, "codes"),
                                     _ptr(next_emb, torch.bfloat16, "next_emb"),
                                     _ptr(done, torch.int32, "done"),
                                     _ptr(logits, torch.float32, "logits"),
                                     _ptr(ws, None, "workspace"), ws.numel(), _stream(stream))
        _check(rc, "hra_codebook_step")
        self.last_ws = ws
        return codes, next_emb, done

    def step_noalloc(self, hidden: torch.Tensor, state: torch.Tensor, eoc_bias: Optional[torch.Tensor] = None,
                     codes: Optional[torch.Tensor] = None, next_emb: Optional[torch.Tensor] = None,
                     done: Optional[torch.Tensor] = None, logits: Optional[torch.Tensor] = None, stream=None):
        """hra_codebook_step_noalloc: the same step for callers that cannot allocate device memory
        (the library's fixed per-device scratch replaces the workspace).  The output tensors may be
        passed in so that the call itself allocates nothing."""
        B = hidden.shape[0]
        K, H = self.d.n_codebooks, self.d.hidden
        dev = hidden.device
        if codes is None:
            codes = torch.empty(B, K, dtype=torch.int32, device=dev)
        if next_emb is None:
            next_emb = torch.empty(B, H, dtype=torch.bfloat16, device=dev)
        if done is None:
            done = torch.empty(B, dtype=torch.int32, device=dev)
        if state.dtype != torch.int32 or tuple(state.shape) != (B, 4):
            raise HraError("state must be int32 [B, 4]")
        rc = lib().hra_codebook_step_noalloc(ctypes.byref(self.dims), _ptr(hidden, torch.bfloat16, "hidden"),
                                             _ptr(self.head_w, torch.bfloat16, "head_w"),
                                             _ptr(self.code_emb, torch.bfloat16, "code_emb"),
                                             _ptr(state, torch.int32, "state"),
                                             _ptr(eoc_bias, torch.float32, "eoc_bias"), B,
                                             _ptr(codes, torch.int32, "codes"),
                                             _ptr(next_emb, torch.bfloat16, "next_emb"),
                                             _ptr(done, torch.int32, "done"),
                                             _ptr(logits, torch.float32, "logits"), _stream(stream))
        _check(rc, "hra_codebook_step_noalloc")
        return codes, next_emb, done


def hra_linear(a: torch.Tensor, w: torch.Tensor, epilogue: int = EPI_STORE,
               out: Optional[torch.Tensor] = None, split_k: int = 0, stream=None) -> torch.Tensor:
    """out = epilogue(a [M, K] @ w^T) through the tensor-core GEMM of the library."""
    M, K = a.shape
    N = w.shape[0] // 2 if epilogue == EPI_SWIGLU else w.shape[0]
    if out is None:
        dt = torch.float32 if epilogue == EPI_F32 else torch.bfloat16
        out = torch.empty(M, N, dtype=dt, device=a.device)
    need = lib().hra_linear_workspace_size(M, N, K, epilogue, split_k)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device=a.device)
    rc = lib().hra_linear(_ptr(a, torch.bfloat16, "a"), _ptr(w, torch.bfloat16, "w"), _ptr(out, None, "out"),
                          M, N, K, epilogue, split_k, _ptr(ws, None, "workspace"), ws.numel(),
                          _stream(stream))
    _check(rc, "hra_linear")
    err = lib().hra_device_error(_ptr(ws, None, "workspace"), _stream(stream))
    if err != 0:
        raise HraError(f"hra_linear device error bits {err}")
    return out


def fp8_quantize_weight(w: torch.Tensor, stream=None):
    """hra_fp8_quantize_weight: bf16 CUDA tensor -> (E4M3 codes uint8 same shape, scale float32 [1])."""
    w8 = torch.empty(w.shape, dtype=torch.uint8, device=w.device)
    sc = torch.empty(1, dtype=torch.float32, device=w.device)
    _check(lib().hra_fp8_quantize_weight(_ptr(w, torch.bfloat16, "w"), w.numel(), _ptr(w8, torch.uint8, "w8"),
                                         _ptr(sc, torch.float32, "scale"), _stream(stream)), "hra_fp8_quantize_weight")
    return w8, sc


def fp8_quantize(x: torch.Tensor, scale: torch.Tensor, stream=None) -> torch.Tensor:
    """hra_fp8_quantize: e4m3(x / scale) as uint8 codes (scale: CUDA float32 scalar tensor)."""
    x8 = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    _check(lib().hra_fp8_quantize(_ptr(x, torch.bfloat16, "x"), x.numel(), _ptr(scale, torch.float32, "scale"),
                                  _ptr(x8, torch.uint8, "x8"), _stream(stream)), "hra_fp8_quantize")
    return x8


def nvfp4_quantize(x: torch.Tensor, g: torch.Tensor, stream=None):
    """hra_nvfp4_quantize: bf16 CUDA [rows, K] and the global scale (CUDA float32 scalar) ->
    (E2M1 codes uint8 [rows, K], E4M3 block scales uint8 [rows, K / 16])."""
    rows, K = x.shape
    codes = torch.empty(rows, K, dtype=torch.uint8, device=x.device)
    scales = torch.empty(rows, K // 16, dtype=torch.uint8, device=x.device)
    _check(lib().hra_nvfp4_quantize(_ptr(x, torch.bfloat16, "x"), rows, K, _ptr(g, torch.float32, "g"),
                                    _ptr(codes, torch.uint8, "codes"), _ptr(scales, torch.uint8, "scales"),
                                    _stream(stream)), "hra_nvfp4_quantize")
    return codes, scales


def hra_linear_fp8(a8: torch.Tensor, w8: torch.Tensor, a_scale: torch.Tensor, w_scale: torch.Tensor,
                   epilogue: int = EPI_STORE, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """hra_linear_fp8: a8 [M, K] and w8 [N or 2N, K] E4M3 codes (uint8), per-tensor scales."""
    M, K = a8.shape
    rows = w8.shape[0]
    N = rows // 2 if epilogue == EPI_SWIGLU else rows
    if out is None:
        dt = torch.float32 if epilogue == EPI_F32 else torch.bfloat16
        out = torch.empty(M, N, dtype=dt, device=a8.device)
    ws = torch.empty(lib().hra_linear_fp8_workspace_size(M, N, K, epilogue), dtype=torch.uint8, device=a8.device)
    _check(lib().hra_linear_fp8(_ptr(a8, torch.uint8, "a8"), _ptr(w8, torch.uint8, "w8"), _ptr(out, None, "out"),
                                M, N, K, _ptr(a_scale, torch.float32, "a_scale"),
                                _ptr(w_scale, torch.float32, "w_scale"), epilogue, _ptr(ws, None, "workspace"),
                                ws.numel(), _stream(stream)), "hra_linear_fp8")
    return out


class Fp8Backbone:
    """The static-FP8 variant of a Backbone: E4M3 copies of every projection (hra_fp8_quantize_weight)
    and static activation scales from hra_fp8_calibrate."""

    NAMES = ("w_qkv", "w_o", "w_gate_up", "w_down")

    def __init__(self, bb: "Backbone"):
        self.bb = bb
        d = bb.d
        dev = bb.device
        self.w8, self.w_scale = [], torch.empty(d.n_layers, 4, dtype=torch.float32, device=dev)
        for l, lay in enumerate(bb.w["layers"]):
            q = []
            for i, name in enumerate(self.NAMES):
                w8, sc = fp8_quantize_weight(lay[name])
                q.append(w8)
                self.w_scale[l, i] = sc[0]
            self.w8.append(q)
        self.amax = torch.zeros(d.n_layers, 4, dtype=torch.float32, device=dev)
        self.a_scale = torch.ones(d.n_layers, 4, dtype=torch.float32, device=dev)
        self._table()

    def _table(self):
        t = (HraFp8Layer * len(self.w8))()
        for l, q in enumerate(self.w8):
            t[l].w_qkv, t[l].w_o, t[l].w_gate_up, t[l].w_down = [x.data_ptr() for x in q]
            t[l].w_scale = self.w_scale[l].data_ptr()
            t[l].a_scale = self.a_scale[l].data_ptr()
        self.table = t

    def calibrate(self, tokens: torch.Tensor, seq_lens: Sequence[int], cache: torch.Tensor, stream=None):
        """hra_fp8_calibrate on a calibration batch: fills amax and a_scale [n_layers, 4]."""
        B, P = tokens.shape
        lens = (ctypes.c_int32 * B)(*[int(x) for x in seq_lens])
        need = lib().hra_fp8_calibrate_workspace_size(ctypes.byref(self.bb.dims), B, int(sum(seq_lens)), P)
        ws = torch.empty(need, dtype=torch.uint8, device=tokens.device)
        kv = self.bb.kv(cache)
        _check(lib().hra_fp8_calibrate(ctypes.byref(self.bb.dims), ctypes.byref(self.bb.table),
                                       _ptr(tokens, torch.int32, "tokens"), lens, B, P, ctypes.byref(kv),
                                       _ptr(self.amax, torch.float32, "amax"),
                                       _ptr(self.a_scale, torch.float32, "a_scale"), _ptr(ws, None, "workspace"),
                                       ws.numel(), _stream(stream)), "hra_fp8_calibrate")
        return self.amax, self.a_scale

    def prefill_workspace_size(self, batch, total, max_len) -> int:
        return lib().hra_prefill_fp8_workspace_size(ctypes.byref(self.bb.dims), batch, total, max_len)

    def prefill(self, tokens: torch.Tensor, seq_lens: Sequence[int], cache: torch.Tensor,
                out: Optional[torch.Tensor] = None, full_last_layer: bool = False,
                workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        """hra_prefill_fp8 -> last hidden [B, H] bf16."""
        B, P = tokens.shape
        lens = (ctypes.c_int32 * B)(*[int(x) for x in seq_lens])
        if out is None:
            out = torch.empty(B, self.bb.d.hidden, dtype=torch.bfloat16, device=tokens.device)
        need = self.prefill_workspace_size(B, int(sum(seq_lens)), P)
        ws = workspace if workspace is not None else self.bb.ws.get(need, tokens.device)
        kv = self.bb.kv(cache)
        _check(lib().hra_prefill_fp8(ctypes.byref(self.bb.dims), ctypes.byref(self.bb.table), self.table,
                                     _ptr(tokens, torch.int32, "tokens"), lens, B, P, ctypes.byref(kv),
                                     _ptr(out, torch.bfloat16, "last_hidden"), _ptr(ws, None, "workspace"),
                                     ws.numel(), PREFILL_FULL_LAST_LAYER if full_last_layer else 0,
                                     _stream(stream)), "hra_prefill_fp8")
        self.last_ws = ws
        return out


def nvfp4_quantize_weight(w: torch.Tensor, stream=None):
    """hra_nvfp4_quantize_weight: bf16 CUDA [rows, K] -> (E2M1 codes uint8 [rows, K], E4M3 block
    scales uint8 [rows, K / 16], global scale float32 [1] = max|w| / (6 * 448))."""
    rows, K = w.shape
    codes = torch.empty(rows, K, dtype=torch.uint8, device=w.device)
    scales = torch.empty(rows, K // 16, dtype=torch.uint8, device=w.device)
    g = torch.empty(1, dtype=torch.float32, device=w.device)
    _check(lib().hra_nvfp4_quantize_weight(_ptr(w, torch.bfloat16, "w"), rows, K, _ptr(codes, torch.uint8, "codes"),
                                           _ptr(scales, torch.uint8, "scales"), _ptr(g, torch.float32, "g"),
                                           _stream(stream)), "hra_nvfp4_quantize_weight")
    return codes, scales, g


def hra_linear_nvfp4(a_codes: torch.Tensor, a_scales: torch.Tensor, w_codes: torch.Tensor, w_scales: torch.Tensor,
                     g_a: torch.Tensor, g_w: torch.Tensor, epilogue: int = EPI_STORE,
                     out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """hra_linear_nvfp4: NVFP4 operands (codes uint8 one per byte, block scales uint8 E4M3, global
    scales CUDA float32 scalars) -> out [M, N] (bf16, or fp32 for EPI_F32)."""
    M, K = a_codes.shape
    N = w_codes.shape[0] // 2 if epilogue == EPI_SWIGLU else w_codes.shape[0]
    if out is None:
        out = torch.empty(M, N, dtype=torch.float32 if epilogue == EPI_F32 else torch.bfloat16,
                          device=a_codes.device)
    ws = torch.empty(lib().hra_linear_nvfp4_workspace_size(), dtype=torch.uint8, device=a_codes.device)
    _check(lib().hra_linear_nvfp4(_ptr(a_codes, torch.uint8, "a_codes"), _ptr(a_scales, torch.uint8, "a_scales"),
                                  _ptr(w_codes, torch.uint8, "w_codes"), _ptr(w_scales, torch.uint8, "w_scales"),
                                  _ptr(out, None, "out"), M, N, K, _ptr(g_a, torch.float32, "g_a"),
                                  _ptr(g_w, torch.float32, "g_w"), epilogue, _ptr(ws, None, "workspace"), ws.numel(),
                                  _stream(stream)), "hra_linear_nvfp4")
    return out


class Nvfp4Backbone:
    """The NVFP4-band variant of a Backbone: the merged QKV in E4M3 (hra_fp8_quantize_weight), the
    output, gate/up and down weights in NVFP4 (hra_nvfp4_quantize_weight); the static input scales
    come from hra_fp8_calibrate's amax (QKV: amax / 448; the NVFP4 inputs: amax / (6 * 448))."""

    NV = ("w_o", "w_gate_up", "w_down")

    def __init__(self, bb: "Backbone"):
        self.bb = bb
        d = bb.d
        dev = bb.device
        self.w_scale = torch.empty(d.n_layers, 4, dtype=torch.float32, device=dev)
        self.keep = []
        for l, lay in enumerate(bb.w["layers"]):
            w8, sc = fp8_quantize_weight(lay["w_qkv"])
            self.w_scale[l, 0] = sc[0]
            entry = {"w_qkv": w8, "codes": [None], "scales": [None]}
            for i, name in enumerate(self.NV):
                c, s, g = nvfp4_quantize_weight(lay[name])
                entry["codes"].append(c)
                entry["scales"].append(s)
                self.w_scale[l, 1 + i] = g[0]
            self.keep.append(entry)
        self.fp8 = Fp8Backbone.__new__(Fp8Backbone)   # only for its calibration pass
        self.fp8.bb = bb
        self.fp8.amax = torch.zeros(d.n_layers, 4, dtype=torch.float32, device=dev)
        self.fp8.a_scale = torch.ones(d.n_layers, 4, dtype=torch.float32, device=dev)
        self.a_scale = torch.ones(d.n_layers, 4, dtype=torch.float32, device=dev)
        self._table()

    def _table(self):
        t = (HraNvfp4Layer * len(self.keep))()
        for l, e in enumerate(self.keep):
            t[l].w_qkv = e["w_qkv"].data_ptr()
            for p in range(1, 4):
                t[l].codes[p] = e["codes"][p].data_ptr()
                t[l].scales[p] = e["scales"][p].data_ptr()
            t[l].w_scale = self.w_scale[l].data_ptr()
            t[l].a_scale = self.a_scale[l].data_ptr()
        self.table = t

    def calibrate(self, tokens: torch.Tensor, seq_lens: Sequence[int], cache: torch.Tensor, stream=None):
        """hra_fp8_calibrate's amax, then a_scale [n_layers, 4] as described above."""
        amax, _ = self.fp8.calibrate(tokens, seq_lens, cache, stream=stream)
        _check(lib().hra_nvfp4_band_scales(_ptr(amax, torch.float32, "amax"), _ptr(self.a_scale, torch.float32, "a_scale"),
                                           self.bb.d.n_layers, _stream(stream)), "hra_nvfp4_band_scales")
        return amax, self.a_scale

    def prefill_workspace_size(self, batch, total, max_len) -> int:
        return lib().hra_prefill_nvfp4_workspace_size(ctypes.byref(self.bb.dims), batch, total, max_len)

    def prefill(self, tokens: torch.Tensor, seq_lens: Sequence[int], cache: torch.Tensor,
                out: Optional[torch.Tensor] = None, full_last_layer: bool = False,
                workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        """hra_prefill_nvfp4 -> last hidden [B, H] bf16."""
        B, P = tokens.shape
        lens = (ctypes.c_int32 * B)(*[int(x) for x in seq_lens])
        if out is None:
            out = torch.empty(B, self.bb.d.hidden, dtype=torch.bfloat16, device=tokens.device)
        need = self.prefill_workspace_size(B, int(sum(seq_lens)), P)
        ws = workspace if workspace is not None else self.bb.ws.get(need, tokens.device)
        kv = self.bb.kv(cache)
        _check(lib().hra_prefill_nvfp4(ctypes.byref(self.bb.dims), ctypes.byref(self.bb.table), self.table,
                                       _ptr(tokens, torch.int32, "tokens"), lens, B, P, ctypes.byref(kv),
                                       _ptr(out, torch.bfloat16, "last_hidden"), _ptr(ws, None, "workspace"),
                                       ws.numel(), PREFILL_FULL_LAST_LAYER if full_last_layer else 0,
                                       _stream(stream)), "hra_prefill_nvfp4")
        self.last_ws = ws
        return out


def hra_device_error(workspace: torch.Tensor, stream=None) -> int:
    """Synchronise and return the sticky device error bits of the last call on this workspace."""
    return int(lib().hra_device_error(_ptr(workspace, None, "workspace"), _stream(stream)))


def hra_launch_counter() -> int:
    """Kernels launched by the library so far in this process."""
    return int(lib().hra_launch_counter())


def hra_set_decode_pass(enable: bool) -> bool:
    """Run passes over at most 64 BF16 rows as one persistent kernel (True) or as one kernel per
    step of each layer (False, the default); returns the previous setting."""
    return bool(lib().hra_set_decode_pass(1 if enable else 0))


def hra_set_gemm_pairs(enable: bool) -> bool:
    """Run projection GEMMs of at least 512 BF16 rows on 2-CTA clusters (True, the default) or on
    single CTAs (False); returns the previous setting."""
    return bool(lib().hra_set_gemm_pairs(1 if enable else 0))


def hra_probe_select(kernel_class: str) -> None:
    """Bracket every launch of one kernel class with CUDA events (see PROBE for the names)."""
    _check(lib().hra_probe_select(PROBE[kernel_class]), "hra_probe_select")


def hra_probe_collect():
    """(summed milliseconds, launches, summed algorithmic work) of the probed launches; clears them.

    The work is FLOPs for the prefill and audio-head classes and bytes for the two decode classes."""
    ms, n, fl = ctypes.c_double(), ctypes.c_int64(), ctypes.c_double()
    _check(lib().hra_probe_collect(ctypes.byref(ms), ctypes.byref(n), ctypes.byref(fl)), "hra_probe_collect")
    return ms.value, n.value, fl.value
