"""CPU oracle of the Higgs-Audio-style prefill + delayed-codebook path.

TEST INFRASTRUCTURE ONLY.  Imported by the tests, by the smoke check and by the benchmark's
CPU-baseline / reference arm; never by the product path.  The arithmetic lives in the plain C file
``hra_oracle.c`` beside this module (fp32 on bf16-rounded values, loops in textbook order); this
wrapper only marshals numpy arrays.  bf16 tensors cross this boundary as numpy ``uint16`` arrays
holding the bf16 bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hra_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

_u16p = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP, no FP contraction so x86 and Arm agree)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC",
                               "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class OracleDims(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("hidden", ctypes.c_int32),
                ("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("ffn", ctypes.c_int32), ("vocab", ctypes.c_int32),
                ("rope_theta", ctypes.c_float), ("rms_eps", ctypes.c_float),
                ("n_codebooks", ctypes.c_int32), ("codebook_size", ctypes.c_int32),
                ("bos_id", ctypes.c_int32), ("eoc_id", ctypes.c_int32)]


class OracleLayer(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("attn_norm", "w_qkv", "q_norm", "k_norm", "w_o", "mlp_norm", "w_gate_up", "w_down")]


class OracleFp8Layer(ctypes.Structure):
    _fields_ = [("w_qkv", ctypes.c_void_p), ("w_o", ctypes.c_void_p), ("w_gate_up", ctypes.c_void_p),
                ("w_down", ctypes.c_void_p), ("w_scale", ctypes.c_float * 4), ("a_scale", ctypes.c_float * 4)]


class OracleNvfp4Layer(ctypes.Structure):
    _fields_ = [("w_qkv", ctypes.c_void_p), ("codes", ctypes.c_void_p * 4), ("scales", ctypes.c_void_p * 4),
                ("w_scale", ctypes.c_float * 4), ("a_scale", ctypes.c_float * 4)]


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        L.oracle_round_bf16.argtypes = [_f32p, _u16p, ctypes.c_int64]
        L.oracle_rmsnorm.argtypes = [_u16p, _u16p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, _u16p]
        L.oracle_linear.argtypes = [_u16p, _u16p, ctypes.c_int, ctypes.c_int, ctypes.c_int, _f32p]
        L.oracle_rope_table.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_double, _f32p, _f32p]
        L.oracle_qk_norm_rope.argtypes = [_u16p, _u16p, _i32p, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_float, ctypes.c_double, _u16p]
        L.oracle_attend.argtypes = [_u16p, _u16p, _u16p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_int, ctypes.c_int, _u16p, ctypes.c_void_p,
                                    ctypes.c_int]
        L.oracle_prefill.argtypes = [ctypes.POINTER(OracleDims), _u16p, ctypes.POINTER(OracleLayer),
                                     _u16p, _i32p, _i32p, ctypes.c_int, ctypes.c_int, _u16p,
                                     ctypes.c_int, ctypes.c_int, _u16p]
        L.oracle_prefill_chunk.argtypes = [ctypes.POINTER(OracleDims), _u16p, ctypes.POINTER(OracleLayer),
                                           _u16p, _i32p, _i32p, _i32p, ctypes.c_int, ctypes.c_int, _u16p,
                                           ctypes.c_int, ctypes.c_int, _u16p]
        L.oracle_decode.argtypes = [ctypes.POINTER(OracleDims), ctypes.POINTER(OracleLayer), _u16p,
                                    _u16p, _i32p, ctypes.c_int, _u16p, ctypes.c_int, ctypes.c_int,
                                    _u16p]
        L.oracle_delay_step.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, _f32p,
                                        ctypes.c_void_p, ctypes.c_int, _i32p, _i32p, _i32p]
        L.oracle_code_embed_sum.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, _u16p, _i32p,
                                            ctypes.c_int, _u16p]
        L.oracle_codebook_step.argtypes = [ctypes.POINTER(OracleDims), _u16p, _u16p, _u16p, _i32p,
                                           ctypes.c_void_p, ctypes.c_int, _i32p, _u16p, _i32p,
                                           ctypes.c_void_p]
        _u32p = np.ctypeslib.ndpointer(np.uint32, flags="C_CONTIGUOUS")
        _u64p = np.ctypeslib.ndpointer(np.uint64, flags="C_CONTIGUOUS")
        L.oracle_philox4x32_10.argtypes = [_u32p, _u32p, _u32p]
        L.oracle_exponential.argtypes = [ctypes.c_uint64, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        L.oracle_exponential.restype = ctypes.c_float
        L.oracle_sample_step.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, _f32p,
                                         ctypes.c_void_p, ctypes.c_float, ctypes.c_int, ctypes.c_float, _u64p,
                                         ctypes.c_int, _i32p, _i32p, _i32p, ctypes.c_void_p, ctypes.c_void_p]
        L.oracle_sample_step.restype = ctypes.c_int
        L.oracle_codebook_step_sampled.argtypes = [ctypes.POINTER(OracleDims), _u16p, _u16p, _u16p, _i32p,
                                                   ctypes.c_void_p, ctypes.c_float, ctypes.c_int, ctypes.c_float,
                                                   _u64p, ctypes.c_int, _i32p, _u16p, _i32p, ctypes.c_void_p]
        L.oracle_codebook_step_sampled.restype = ctypes.c_int
        _u8p = np.ctypeslib.ndpointer(np.uint8, flags="C_CONTIGUOUS")
        L.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.oracle_e4m3_decode.restype = ctypes.c_float
        L.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        L.oracle_e4m3_encode.restype = ctypes.c_uint8
        L.oracle_quantize_e4m3.argtypes = [_u16p, ctypes.c_int64, ctypes.c_float, _u8p]
        L.oracle_quantize_weight_e4m3.argtypes = [_u16p, ctypes.c_int64, ctypes.POINTER(ctypes.c_float), _u8p]
        L.oracle_linear_fp8.argtypes = [_u8p, _u8p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float, _f32p]
        L.oracle_e2m1_decode.argtypes = [ctypes.c_uint8]
        L.oracle_e2m1_decode.restype = ctypes.c_float
        L.oracle_e2m1_encode.argtypes = [ctypes.c_float]
        L.oracle_e2m1_encode.restype = ctypes.c_uint8
        L.oracle_nvfp4_global.argtypes = [_u16p, ctypes.c_int64]
        L.oracle_nvfp4_global.restype = ctypes.c_float
        L.oracle_quantize_nvfp4.argtypes = [_u16p, ctypes.c_int, ctypes.c_int, ctypes.c_float, _u8p, _u8p]
        L.oracle_linear_nvfp4.argtypes = [_u8p, _u8p, _u8p, _u8p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_float, ctypes.c_float, _f32p]
        L.oracle_prefill_fp8.argtypes = [ctypes.POINTER(OracleDims), _u16p, ctypes.POINTER(OracleLayer),
                                         ctypes.POINTER(OracleFp8Layer), _u16p, _i32p, _i32p, ctypes.c_int,
                                         ctypes.c_int, _u16p, ctypes.c_int, ctypes.c_int, _u16p]
        L.oracle_calibrate.argtypes = [ctypes.POINTER(OracleDims), _u16p, ctypes.POINTER(OracleLayer), _u16p, _i32p,
                                       _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, _f32p]
        L.oracle_prefill_nvfp4.argtypes = [ctypes.POINTER(OracleDims), _u16p, ctypes.POINTER(OracleLayer),
                                           ctypes.POINTER(OracleNvfp4Layer), _u16p, _i32p, _i32p, ctypes.c_int,
                                           ctypes.c_int, _u16p, ctypes.c_int, ctypes.c_int, _u16p]
        for f in ("oracle_prefill_fp8", "oracle_calibrate", "oracle_prefill_nvfp4"):
            getattr(L, f).restype = ctypes.c_int
        for f in ("oracle_prefill", "oracle_prefill_chunk", "oracle_decode", "oracle_codebook_step",
                  "oracle_max_threads"):
            getattr(L, f).restype = ctypes.c_int
        L.oracle_set_threads.argtypes = [ctypes.c_int]
        L.oracle_set_sum_order.argtypes = [ctypes.c_int]
        _lib = L
    return _lib


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def max_threads() -> int:
    return lib().oracle_max_threads()


def set_threads(n: int) -> None:
    lib().oracle_set_threads(int(n))


class sum_order:
    """Context manager: evaluate every linear dot product in descending k order inside the block."""

    def __init__(self, descending: bool = True):
        self.descending = descending

    def __enter__(self):
        lib().oracle_set_sum_order(1 if self.descending else 0)
        return self

    def __exit__(self, *exc):
        lib().oracle_set_sum_order(0)
        return False


# ------------------------------------------------------------------ element-wise helpers

def bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even."""
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().oracle_round_bf16(x.reshape(-1), out.reshape(-1), x.size)
    return out


def bf16_value(u: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> fp32 values (exact)."""
    return (np.asarray(u, np.uint16).astype(np.uint32) << 16).view(np.float32)


def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    x, g = _c(x, np.uint16), _c(g, np.uint16)
    n = x.shape[-1]
    out = np.empty_like(x)
    lib().oracle_rmsnorm(x, g, x.size // n, n, eps, out)
    return out


def linear(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """x [T, K] bf16 bits, w [N, K] bf16 bits -> fp32 [T, N] (unrounded)."""
    x, w = _c(x, np.uint16), _c(w, np.uint16)
    T, K = x.shape
    N = w.shape[0]
    assert w.shape[1] == K
    out = np.empty((T, N), np.float32)
    lib().oracle_linear(x, w, T, N, K, out)
    return out


def rope_table(n_pos: int, hd: int, theta: float):
    c = np.empty((n_pos, hd // 2), np.float32)
    s = np.empty((n_pos, hd // 2), np.float32)
    lib().oracle_rope_table(n_pos, hd, theta, c, s)
    return c, s


def qk_norm_rope(x: np.ndarray, g: np.ndarray, pos, eps: float, theta: float) -> np.ndarray:
    x, g = _c(x, np.uint16), _c(g, np.uint16)
    pos = _c(pos, np.int32)
    rows, hd = x.shape
    out = np.empty_like(x)
    lib().oracle_qk_norm_rope(x, g, pos, rows, hd, eps, theta, out)
    return out


def attend(q, kc, vc, q_pos0: int, want_probs: bool = False):
    """q [n, nq, hd], kc/vc [nkv, n_slots, hd] bf16 bits -> out [n, nq*hd] (+ probs [n, nq, keys])."""
    q, kc, vc = _c(q, np.uint16), _c(kc, np.uint16), _c(vc, np.uint16)
    n, nq, hd = q.shape
    nkv, n_slots, _ = kc.shape
    out = np.empty((n, nq * hd), np.uint16)
    nk = q_pos0 + n
    probs = np.zeros((n, nq, nk), np.float32) if want_probs else None
    lib().oracle_attend(q, kc, vc, n_slots, q_pos0, n, nq, nkv, hd, out,
                        probs.ctypes.data if want_probs else None, nk)
    return (out, probs) if want_probs else out


# ------------------------------------------------------------------ model level

def make_dims(d) -> OracleDims:
    return OracleDims(d.n_layers, d.hidden, d.n_q_heads, d.n_kv_heads, d.head_dim, d.ffn, d.vocab,
                      d.rope_theta, d.rms_eps, d.n_codebooks, d.codebook_size, d.bos_id, d.eoc_id)


_LAYER_KEYS = ("attn_norm", "w_qkv", "q_norm", "k_norm", "w_o", "mlp_norm", "w_gate_up", "w_down")


class HostWeights:
    """Backbone weights as contiguous numpy uint16 arrays plus the ctypes layer table."""

    def __init__(self, d, embed, layers, final_norm):
        self.d = d
        self.embed = _c(embed, np.uint16)
        self.layers = [{k: _c(l[k], np.uint16) for k in _LAYER_KEYS} for l in layers]
        self.final_norm = _c(final_norm, np.uint16)
        n = len(self.layers)
        self.table = (OracleLayer * max(n, 1))()
        for i, l in enumerate(self.layers):
            for k in _LAYER_KEYS:
                setattr(self.table[i], k, l[k].ctypes.data)


def kv_shape(d, kv_batch: int, n_slots: int):
    return (d.n_layers, kv_batch, 2, d.n_kv_heads, n_slots, d.head_dim)


def prefill(d, w: HostWeights, tokens: np.ndarray, lens, n_slots: int,
            kv: Optional[np.ndarray] = None):
    """Returns (kv [L, B, 2, nkv, n_slots, hd] uint16, last_hidden [B, H] uint16)."""
    tokens = _c(tokens, np.int32)
    lens = _c(lens, np.int32)
    B, P = tokens.shape
    if kv is None:
        kv = np.zeros(kv_shape(d, B, n_slots), np.uint16)
    last = np.empty((B, d.hidden), np.uint16)
    dims = make_dims(d)
    rc = lib().oracle_prefill(ctypes.byref(dims), w.embed, w.table, w.final_norm, tokens, lens, B, P,
                              kv, kv.shape[1], n_slots, last)
    if rc != 0:
        raise ValueError("oracle_prefill rejected its arguments")
    return kv, last


def prefill_chunk(d, w: HostWeights, tokens: np.ndarray, lens, starts, kv: np.ndarray, n_slots: int):
    """One chunk per sequence at positions starts[b] .. starts[b] + lens[b] - 1 after the cached ones.

    kv [L, B, 2, nkv, n_slots, hd] uint16 is read below each start and written in place; returns
    last_hidden [B, H] uint16."""
    tokens = _c(tokens, np.int32)
    lens = _c(lens, np.int32)
    starts = _c(starts, np.int32)
    B, P = tokens.shape
    last = np.empty((B, d.hidden), np.uint16)
    dims = make_dims(d)
    rc = lib().oracle_prefill_chunk(ctypes.byref(dims), w.embed, w.table, w.final_norm, tokens, lens, starts,
                                    B, P, kv, kv.shape[1], n_slots, last)
    if rc != 0:
        raise ValueError("oracle_prefill_chunk rejected its arguments")
    return last


def decode(d, w: HostWeights, in_emb: np.ndarray, pos, kv: np.ndarray, n_slots: int) -> np.ndarray:
    in_emb = _c(in_emb, np.uint16)
    pos = _c(pos, np.int32)
    B = in_emb.shape[0]
    out = np.empty((B, d.hidden), np.uint16)
    dims = make_dims(d)
    rc = lib().oracle_decode(ctypes.byref(dims), w.table, w.final_norm, in_emb, pos, B, kv,
                             kv.shape[1], n_slots, out)
    if rc != 0:
        raise ValueError("oracle_decode rejected its arguments")
    return out


def philox4x32_10(ctr, key) -> np.ndarray:
    """Philox4x32-10 of counter (4 x uint32) under key (2 x uint32) -> 4 x uint32."""
    c = np.ascontiguousarray(ctr, np.uint32)
    k = np.ascontiguousarray(key, np.uint32)
    out = np.empty(4, np.uint32)
    lib().oracle_philox4x32_10(c, k, out)
    return out


def exponential(seed: int, t: int, k: int, v: int) -> float:
    """The sampler's exponential noise of entry v, codebook k, frame t for a row seeded `seed`."""
    return float(lib().oracle_exponential(ctypes.c_uint64(seed), t, k, v))


def sample_step(K: int, Vc: int, bos: int, eoc: int, logits: np.ndarray, eoc_bias, temperature: float,
                top_k: int, top_p: float, seeds, state: np.ndarray):
    """Sampled state machine (state [B,4] int32 updated in place).
    Returns (codes [B,K], done [B], margin [B,K], ambiguous [B,K])."""
    logits = _c(logits, np.float32)
    B = logits.shape[0]
    assert state.dtype == np.int32 and state.flags.c_contiguous
    seeds = np.ascontiguousarray(seeds, np.uint64)
    codes = np.empty((B, K), np.int32)
    done = np.empty((B,), np.int32)
    margin = np.empty((B, K), np.float32)
    amb = np.empty((B, K), np.int32)
    bias = None if eoc_bias is None else _c(eoc_bias, np.float32)
    rc = lib().oracle_sample_step(K, Vc, bos, eoc, logits, None if bias is None else bias.ctypes.data,
                                  float(temperature), int(top_k), float(top_p), seeds, B, state, codes, done,
                                  margin.ctypes.data, amb.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_sample_step rejected its arguments")
    return codes, done, margin, amb


def codebook_step_sampled(d, hidden: np.ndarray, head_w: np.ndarray, code_emb: np.ndarray, state: np.ndarray,
                          eoc_bias, temperature: float, top_k: int, top_p: float, seeds):
    """Returns (codes [B,K], next [B,H] uint16, done [B], logits [B,K,Vc] fp32)."""
    hidden = _c(hidden, np.uint16)
    B = hidden.shape[0]
    K, Vc = d.n_codebooks, d.codebook_size
    codes = np.empty((B, K), np.int32)
    nxt = np.empty((B, d.hidden), np.uint16)
    done = np.empty((B,), np.int32)
    logits = np.empty((B, K, Vc), np.float32)
    bias = None if eoc_bias is None else _c(eoc_bias, np.float32)
    rc = lib().oracle_codebook_step_sampled(ctypes.byref(make_dims(d)), hidden, _c(head_w, np.uint16),
                                            _c(code_emb, np.uint16), state,
                                            None if bias is None else bias.ctypes.data, float(temperature),
                                            int(top_k), float(top_p), np.ascontiguousarray(seeds, np.uint64), B,
                                            codes, nxt, done, logits.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_codebook_step_sampled rejected its arguments")
    return codes, nxt, done, logits


def e4m3_decode(codes) -> np.ndarray:
    c = np.asarray(codes, np.uint8).ravel()
    return np.array([lib().oracle_e4m3_decode(int(x)) for x in c], np.float32).reshape(np.shape(codes))


def e4m3_encode(x) -> np.ndarray:
    a = np.asarray(x, np.float32).ravel()
    return np.array([lib().oracle_e4m3_encode(float(v)) for v in a], np.uint8).reshape(np.shape(x))


def quantize_e4m3(x_u16: np.ndarray, scale: float) -> np.ndarray:
    x = _c(x_u16, np.uint16)
    out = np.empty(x.shape, np.uint8)
    lib().oracle_quantize_e4m3(x, x.size, float(scale), out)
    return out


def quantize_weight_e4m3(w_u16: np.ndarray):
    """(scale, E4M3 codes) with scale = max|w| / 448."""
    w = _c(w_u16, np.uint16)
    out = np.empty(w.shape, np.uint8)
    sc = ctypes.c_float()
    lib().oracle_quantize_weight_e4m3(w, w.size, ctypes.byref(sc), out)
    return sc.value, out


def linear_fp8(x8: np.ndarray, w8: np.ndarray, scale: float) -> np.ndarray:
    x8 = np.ascontiguousarray(x8, np.uint8)
    w8 = np.ascontiguousarray(w8, np.uint8)
    T, K = x8.shape
    N = w8.shape[0]
    y = np.empty((T, N), np.float32)
    lib().oracle_linear_fp8(x8, w8, T, N, K, float(scale), y)
    return y


def e2m1_decode(codes) -> np.ndarray:
    c = np.asarray(codes, np.uint8).ravel()
    return np.array([lib().oracle_e2m1_decode(int(x)) for x in c], np.float32).reshape(np.shape(codes))


def e2m1_encode(x) -> np.ndarray:
    a = np.asarray(x, np.float32).ravel()
    return np.array([lib().oracle_e2m1_encode(float(v)) for v in a], np.uint8).reshape(np.shape(x))


def nvfp4_global(x_u16: np.ndarray) -> float:
    """Global scale max|x| / (6 * 448) of an NVFP4 tensor (1 for an all-zero tensor)."""
    x = _c(x_u16, np.uint16)
    return float(lib().oracle_nvfp4_global(x, x.size))


def quantize_nvfp4(x_u16: np.ndarray, g: float):
    """(codes [rows, K] one E2M1 code per byte, block scales [rows, K/16] E4M3) of bf16 bits x."""
    x = _c(x_u16, np.uint16)
    rows, K = x.shape
    codes = np.empty((rows, K), np.uint8)
    scales = np.empty((rows, K // 16), np.uint8)
    lib().oracle_quantize_nvfp4(x, rows, K, float(g), codes, scales)
    return codes, scales


def linear_nvfp4(a, sa, w, sw, g_a: float, g_w: float) -> np.ndarray:
    """fp32 y [T, N] of NVFP4 operands a [T, K] / w [N, K] with block scales sa / sw."""
    a, sa, w, sw = (np.ascontiguousarray(v, np.uint8) for v in (a, sa, w, sw))
    T, K = a.shape
    N = w.shape[0]
    y = np.empty((T, N), np.float32)
    lib().oracle_linear_nvfp4(a, sa, w, sw, T, N, K, float(g_a), float(g_w), y)
    return y


class Fp8Weights:
    """E4M3 copies of every layer's projections with per-tensor weight scales, plus the static
    activation scales (a_scale [L, 4]: qkv, o, gate_up, down inputs)."""

    def __init__(self, hw: "HostWeights", a_scale: np.ndarray):
        self.w8, self.w_scale = [], []
        for lay in hw.layers:
            ws, ws8 = [], []
            for name in ("w_qkv", "w_o", "w_gate_up", "w_down"):
                sc, q = quantize_weight_e4m3(lay[name])
                ws.append(sc)
                ws8.append(q)
            self.w8.append(ws8)
            self.w_scale.append(ws)
        self.a_scale = np.asarray(a_scale, np.float32)
        self.table = (OracleFp8Layer * len(self.w8))()
        for l, ws8 in enumerate(self.w8):
            self.table[l].w_qkv, self.table[l].w_o, self.table[l].w_gate_up, self.table[l].w_down = \
                [x.ctypes.data for x in ws8]
            for i in range(4):
                self.table[l].w_scale[i] = self.w_scale[l][i]
                self.table[l].a_scale[i] = float(self.a_scale[l, i])


def prefill_fp8(d, w: "HostWeights", f8: Fp8Weights, tokens: np.ndarray, lens, n_slots: int):
    """Returns (kv, last_hidden) of the FP8 variant."""
    tokens = _c(tokens, np.int32)
    lens = _c(lens, np.int32)
    B, P = tokens.shape
    kv = np.zeros(kv_shape(d, B, n_slots), np.uint16)
    last = np.empty((B, d.hidden), np.uint16)
    rc = lib().oracle_prefill_fp8(ctypes.byref(make_dims(d)), w.embed, w.table, f8.table, w.final_norm, tokens,
                                  lens, B, P, kv, B, n_slots, last)
    if rc != 0:
        raise ValueError("oracle_prefill_fp8 rejected its arguments")
    return kv, last


class Nvfp4Weights:
    """The NVFP4 band of every layer (the fp8_chain page, its precision bands): the merged QKV as
    E4M3 with a per-tensor scale (static input scale a_scale[l, 0]); the output, gate/up and down
    weights as E2M1 codes + E4M3 block scales under a per-tensor global scale g_w = max|w| / 2688,
    their inputs quantized per call under the static global scale a_scale[l, p] (e.g. the
    calibration's max |input| / 2688)."""

    def __init__(self, hw: "HostWeights", a_scale: np.ndarray):
        self.keep, self.w_scale = [], []
        for lay in hw.layers:
            sc, q = quantize_weight_e4m3(lay["w_qkv"])
            entry = {"w_qkv": q, "codes": [None], "scales": [None]}
            ws = [sc]
            for name in ("w_o", "w_gate_up", "w_down"):
                w = lay[name]
                g = nvfp4_global(w)
                c, s = quantize_nvfp4(w, g)
                entry["codes"].append(c)
                entry["scales"].append(s)
                ws.append(g)
            self.keep.append(entry)
            self.w_scale.append(ws)
        self.a_scale = np.asarray(a_scale, np.float32)
        self.table = (OracleNvfp4Layer * len(self.keep))()
        for l, e in enumerate(self.keep):
            self.table[l].w_qkv = e["w_qkv"].ctypes.data
            for p in range(4):
                self.table[l].codes[p] = None if e["codes"][p] is None else e["codes"][p].ctypes.data
                self.table[l].scales[p] = None if e["scales"][p] is None else e["scales"][p].ctypes.data
                self.table[l].w_scale[p] = float(self.w_scale[l][p])
                self.table[l].a_scale[p] = float(self.a_scale[l, p])


def nvfp4_a_scales(amax: np.ndarray) -> np.ndarray:
    """Static input scales of the NVFP4 band from the calibration amax [L, 4]: the QKV input's E4M3
    scale amax / 448 (1 where amax is 0); the other inputs' NVFP4 global scale amax / (6 * 448)."""
    a = np.asarray(amax, np.float32)
    out = np.empty_like(a)
    out[:, 0] = np.where(a[:, 0] > 0, a[:, 0] / np.float32(448.0), np.float32(1.0))
    out[:, 1:] = np.where(a[:, 1:] > 0, a[:, 1:] / np.float32(6.0 * 448.0), np.float32(1.0))
    return out


def prefill_nvfp4(d, w: "HostWeights", nv: Nvfp4Weights, tokens: np.ndarray, lens, n_slots: int):
    """Returns (kv, last_hidden) of the NVFP4-band variant."""
    tokens = _c(tokens, np.int32)
    lens = _c(lens, np.int32)
    B, P = tokens.shape
    kv = np.zeros(kv_shape(d, B, n_slots), np.uint16)
    last = np.empty((B, d.hidden), np.uint16)
    rc = lib().oracle_prefill_nvfp4(ctypes.byref(make_dims(d)), w.embed, w.table, nv.table, w.final_norm, tokens,
                                    lens, B, P, kv, B, n_slots, last)
    if rc != 0:
        raise ValueError("oracle_prefill_nvfp4 rejected its arguments")
    return kv, last


def calibrate(d, w: "HostWeights", tokens: np.ndarray, lens, n_slots: int) -> np.ndarray:
    """amax [L, 4] of the qkv, o, gate_up and down inputs over a bf16 prefill of the batch."""
    tokens = _c(tokens, np.int32)
    lens = _c(lens, np.int32)
    B, P = tokens.shape
    amax = np.empty((d.n_layers, 4), np.float32)
    rc = lib().oracle_calibrate(ctypes.byref(make_dims(d)), w.embed, w.table, w.final_norm, tokens, lens, B, P,
                                n_slots, amax)
    if rc != 0:
        raise ValueError("oracle_calibrate rejected its arguments")
    return amax


def delay_step(K: int, Vc: int, bos: int, eoc: int, logits: np.ndarray, eoc_bias, state: np.ndarray):
    """State machine only (state [B,4] int32 updated in place).  Returns (codes [B,K], done [B])."""
    logits = _c(logits, np.float32)
    B = logits.shape[0]
    assert state.dtype == np.int32 and state.flags.c_contiguous
    codes = np.empty((B, K), np.int32)
    done = np.empty((B,), np.int32)
    bias = None if eoc_bias is None else _c(eoc_bias, np.float32)
    lib().oracle_delay_step(K, Vc, bos, eoc, logits, None if bias is None else bias.ctypes.data, B,
                            state, codes, done)
    return codes, done


def code_embed_sum(code_emb: np.ndarray, codes: np.ndarray) -> np.ndarray:
    code_emb = _c(code_emb, np.uint16)
    codes = _c(codes, np.int32)
    K, Vc, H = code_emb.shape
    B = codes.shape[0]
    out = np.empty((B, H), np.uint16)
    lib().oracle_code_embed_sum(K, Vc, H, code_emb, codes, B, out)
    return out


def codebook_step(d, hidden, head_w, code_emb, state: np.ndarray, eoc_bias=None):
    """Returns (codes [B,K], next [B,H] uint16, done [B], logits [B,K,Vc] fp32); state updated."""
    hidden, head_w, code_emb = _c(hidden, np.uint16), _c(head_w, np.uint16), _c(code_emb, np.uint16)
    B = hidden.shape[0]
    K, Vc = d.n_codebooks, d.codebook_size
    codes = np.empty((B, K), np.int32)
    nxt = np.empty((B, d.hidden), np.uint16)
    done = np.empty((B,), np.int32)
    logits = np.empty((B, K, Vc), np.float32)
    bias = None if eoc_bias is None else _c(eoc_bias, np.float32)
    dims = make_dims(d)
    rc = lib().oracle_codebook_step(ctypes.byref(dims), hidden, head_w, code_emb, state,
                                    None if bias is None else bias.ctypes.data, B, codes, nxt, done,
                                    logits.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_codebook_step rejected its arguments")
    return codes, nxt, done, logits


def host_weights_from(d, w: dict) -> HostWeights:
    """Host copy of a backbone weight dict produced by the workloads module (torch bf16 tensors)."""
    from workloads import to_u16
    return HostWeights(d, to_u16(w["embed"]), [{k: to_u16(l[k]) for k in _LAYER_KEYS} for l in
                                               w["layers"]], to_u16(w["final_norm"]))
